// Status codes and the per-thread error message of the C ABI.
#include <string>

#include "plan.h"

namespace uvu {
namespace {
thread_local std::string g_last;
}

uvu_status fail(uvu_status s, const std::string& msg) {
    g_last = msg;
    return s;
}

const char* g_last_message_cstr() { return g_last.c_str(); }

uvu_status ok() {
    g_last.clear();
    return UVU_OK;
}

uvu_status cuda_fail(cudaError_t e, const char* what) {
    g_last = std::string(what) + ": " + cudaGetErrorName(e) + " (" + cudaGetErrorString(e) + ")";
    return e == cudaErrorMemoryAllocation ? UVU_ERR_OUT_OF_MEMORY : UVU_ERR_CUDA;
}

}  // namespace uvu

extern "C" const char* uvu_status_string(uvu_status s) {
    switch (s) {
        case UVU_OK: return "UVU_OK";
        case UVU_ERR_INVALID_ARGUMENT: return "UVU_ERR_INVALID_ARGUMENT";
        case UVU_ERR_UNSUPPORTED: return "UVU_ERR_UNSUPPORTED";
        case UVU_ERR_COMPILE: return "UVU_ERR_COMPILE";
        case UVU_ERR_CUDA: return "UVU_ERR_CUDA";
        case UVU_ERR_OUT_OF_MEMORY: return "UVU_ERR_OUT_OF_MEMORY";
    }
    return "UVU_ERR_UNKNOWN";
}

extern "C" const char* uvu_last_error_message(void) { return uvu::g_last_message_cstr(); }
