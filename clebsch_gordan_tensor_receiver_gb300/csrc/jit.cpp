// NVRTC compilation of a plan's emitted source for sm_103a, and per-device module loading.
//
// The cubin is produced on the host at plan creation (no GPU needed) and loaded with
// cudaLibraryLoadData on each device at its first launch there.  Compiled code is only loaded,
// never inspected.  Identical sources share one compilation through a process-wide cache.
#include <nvrtc.h>

#include <cstdint>
#include <cstdio>
#include <cstdlib>
#include <fstream>
#include <functional>
#include <map>
#include <mutex>
#include <string>
#include <vector>

#include "plan.h"

namespace uvu {
namespace {

struct CacheEntry {
    std::vector<char> cubin;
    std::string log;
};
std::mutex g_cache_mu;
std::map<std::string, CacheEntry> g_cache;  // keyed by the full source text

// 64-bit FNV-1a of the text (names cache and dump files; the cache also stores the full source
// and compares it, so a collision cannot return the wrong module).
std::string text_hash(const std::string& t) {
    uint64_t h = 1469598103934665603ull;
    for (unsigned char c : t) h = (h ^ c) * 1099511628211ull;
    char buf[17];
    std::snprintf(buf, sizeof buf, "%016llx", (unsigned long long)h);
    return buf;
}

const char* env_dir(const char* name) {
    const char* d = std::getenv(name);
    return (d && *d) ? d : nullptr;
}

// Disk cache (UVU_CACHE_DIR): one file per source, holding the source, the cubin and the NVRTC
// log (the log carries the register/spill report the planner reads).  Written to a temporary
// name and renamed, so concurrent processes never read a partial file.
bool cache_read(const std::string& path, const std::string& src, CacheEntry* out) {
    std::ifstream f(path, std::ios::binary);
    if (!f) return false;
    uint64_t n[3];
    char magic[8];
    if (!f.read(magic, 8) || std::string(magic, 8) != "UVUCUBN1" || !f.read(reinterpret_cast<char*>(n), sizeof n)) return false;
    if (n[0] != src.size() || n[1] > (1ull << 30) || n[2] > (1ull << 30)) return false;
    std::string s(n[0], '\0');
    out->cubin.resize(n[1]);
    out->log.assign(n[2], '\0');
    if (!f.read(&s[0], std::streamsize(n[0])) || s != src) return false;
    if (!f.read(out->cubin.data(), std::streamsize(n[1])) || !f.read(&out->log[0], std::streamsize(n[2]))) return false;
    return true;
}

void cache_write(const std::string& path, const std::string& src, const CacheEntry& e) {
    const std::string tmp = path + ".tmp" + std::to_string(uint64_t(reinterpret_cast<uintptr_t>(&e)));
    {
        std::ofstream f(tmp, std::ios::binary);
        if (!f) return;
        const uint64_t n[3] = {src.size(), e.cubin.size(), e.log.size()};
        f.write("UVUCUBN1", 8);
        f.write(reinterpret_cast<const char*>(n), sizeof n);
        f.write(src.data(), std::streamsize(src.size()));
        f.write(e.cubin.data(), std::streamsize(e.cubin.size()));
        f.write(e.log.data(), std::streamsize(e.log.size()));
        if (!f) {
            std::remove(tmp.c_str());
            return;
        }
    }
    std::rename(tmp.c_str(), path.c_str());
}

uvu_status nvrtc_compile_uncached(const std::string& src, CacheEntry* out, std::string* err);

// --no-cache: NVRTC's cross-process compile cache returns the cubin without running ptxas on a
// hit, so the log would lack the register/spill report the planner's register-budget choice
// reads (a later process then kept a spilling four-block budget: edge kernel 1.35 ms instead of
// 0.87 ms on MACE-medium).  Modules are cached by this library instead (UVU_CACHE_DIR), log included.
const char* const kNvrtcOpts[] = {"--gpu-architecture=sm_103a", "--std=c++17", "-lineinfo",
                                  "--ptxas-options=-v", "--fmad=true", "--no-cache"};

// UVU_FAIL_COMPILE=1 makes every compilation fail (host-side fault injection for the error
// path); UVU_DUMP_SOURCE=<dir> writes each emitted source there for review.
uvu_status nvrtc_compile(const std::string& src, CacheEntry* out, std::string* err) {
    if (const char* f = std::getenv("UVU_FAIL_COMPILE"); f && std::atoi(f) != 0) {
        *err = "NVRTC compile failed: failure injected by UVU_FAIL_COMPILE";
        return UVU_ERR_COMPILE;
    }
    int ver_major = 0, ver_minor = 0;
    nvrtcVersion(&ver_major, &ver_minor);
    std::string salt = "|nvrtc " + std::to_string(ver_major) + "." + std::to_string(ver_minor);
    for (const char* o : kNvrtcOpts) salt += std::string("|") + o;
    const std::string key = text_hash(src + salt);
    if (const char* d = env_dir("UVU_DUMP_SOURCE")) {
        std::ofstream f(std::string(d) + "/uvu_" + key + ".cu");
        f << src;
    }
    const char* cdir = env_dir("UVU_CACHE_DIR");
    const std::string cpath = cdir ? std::string(cdir) + "/uvu_" + key + ".bin" : std::string();
    if (cdir && cache_read(cpath, src, out)) return UVU_OK;
    uvu_status s = nvrtc_compile_uncached(src, out, err);
    if (s == UVU_OK && cdir) cache_write(cpath, src, *out);
    return s;
}

uvu_status nvrtc_compile_uncached(const std::string& src, CacheEntry* out, std::string* err) {
    nvrtcProgram prog;
    nvrtcResult r = nvrtcCreateProgram(&prog, src.c_str(), "uvu_plan.cu", 0, nullptr, nullptr);
    if (r != NVRTC_SUCCESS) {
        *err = std::string("nvrtcCreateProgram: ") + nvrtcGetErrorString(r);
        return UVU_ERR_COMPILE;
    }
    r = nvrtcCompileProgram(prog, int(sizeof(kNvrtcOpts) / sizeof(kNvrtcOpts[0])), kNvrtcOpts);
    size_t log_size = 0;
    nvrtcGetProgramLogSize(prog, &log_size);
    std::string log(log_size, '\0');
    if (log_size) nvrtcGetProgramLog(prog, &log[0]);
    if (r != NVRTC_SUCCESS) {
        *err = std::string("NVRTC compile failed: ") + nvrtcGetErrorString(r) + "\n" + log;
        nvrtcDestroyProgram(&prog);
        return UVU_ERR_COMPILE;
    }
    size_t n = 0;
    nvrtcGetCUBINSize(prog, &n);
    out->cubin.resize(n);
    nvrtcGetCUBIN(prog, out->cubin.data());
    out->log = log;
    nvrtcDestroyProgram(&prog);
    return UVU_OK;
}

}  // namespace

// Spill store bytes ptxas reported for one entry function (0 if not found).
size_t spill_bytes(const std::string& log, const char* kernel) {
    const std::string key = std::string("Function properties for ") + kernel + "\n";
    const size_t at = log.find(key);
    if (at == std::string::npos) return 0;
    const size_t eol = log.find('\n', at + key.size());
    const std::string line = log.substr(at + key.size(), eol == std::string::npos ? std::string::npos : eol - at - key.size());
    const size_t sp = line.find(" bytes spill stores");
    if (sp == std::string::npos) return 0;
    size_t b = line.rfind(' ', sp - 1);
    return size_t(std::strtoull(line.c_str() + (b == std::string::npos ? 0 : b + 1), nullptr, 10));
}

uvu_status compile_plan(Plan* plan, std::string* err) {
    {
        std::lock_guard<std::mutex> g(g_cache_mu);
        auto it = g_cache.find(plan->source);
        if (it != g_cache.end()) {
            plan->cubin = it->second.cubin;
            plan->log = it->second.log;
            return UVU_OK;
        }
    }
    CacheEntry e;
    uvu_status s = nvrtc_compile(plan->source, &e, err);
    if (s != UVU_OK) return s;
    plan->cubin = e.cubin;
    plan->log = e.log;
    std::lock_guard<std::mutex> g(g_cache_mu);
    g_cache.emplace(plan->source, std::move(e));
    return UVU_OK;
}

uvu_status module_for_current_device(Plan* plan, DeviceModule** out, std::string* err) {
    int dev = 0;
    cudaError_t ce = cudaGetDevice(&dev);
    if (ce != cudaSuccess) {
        *err = std::string("cudaGetDevice: ") + cudaGetErrorString(ce);
        return UVU_ERR_CUDA;
    }
    std::lock_guard<std::mutex> g(plan->mu);
    auto it = plan->modules.find(dev);
    if (it != plan->modules.end()) {
        *out = &it->second;
        return UVU_OK;
    }
    DeviceModule m;
    ce = cudaLibraryLoadData(&m.lib, plan->cubin.data(), nullptr, nullptr, 0, nullptr, nullptr, 0);
    if (ce != cudaSuccess) {
        *err = std::string("cudaLibraryLoadData: ") + cudaGetErrorString(ce);
        return UVU_ERR_CUDA;
    }
    struct {
        const char* name;
        cudaKernel_t* k;
    } ks[] = {{"uvu_fwd", &m.fwd}, {"uvu_bwd_edge", &m.bwd_edge}, {"uvu_bwd_dx", &m.bwd_dx},
              {"uvu_bwd_dx_reduce", &m.bwd_dx_reduce}, {"uvu_fwd_sender", &m.fwd_sender}};
    for (auto& k : ks) {
        ce = cudaLibraryGetKernel(k.k, m.lib, k.name);
        if (ce != cudaSuccess) {
            *err = std::string("cudaLibraryGetKernel(") + k.name + "): " + cudaGetErrorString(ce);
            cudaLibraryUnload(m.lib);
            return UVU_ERR_CUDA;
        }
    }
    struct {
        cudaKernel_t k;
        const KernelGeom* g;
        int* occ;
        const char* name;
    } kk[] = {{m.fwd, &plan->g_fwd, &m.occ_fwd, "uvu_fwd"},
              {m.bwd_edge, &plan->g_edge, &m.occ_edge, "uvu_bwd_edge"},
              {m.bwd_dx, &plan->g_dx, &m.occ_dx, "uvu_bwd_dx"}};
    for (auto& k : kk) {
        const void* f = reinterpret_cast<const void*>(k.k);
        if (k.g->smem > 48 * 1024) {
            ce = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, int(k.g->smem));
            if (ce != cudaSuccess) {
                *err = std::string("cudaFuncSetAttribute(") + k.name + "): " + cudaGetErrorString(ce);
                cudaLibraryUnload(m.lib);
                return UVU_ERR_CUDA;
            }
        }
        if (k.g->persistent) {
            // The persistent grid is sized for the resident blocks the occupancy calculation
            // reports, which assumes the largest shared-memory carveout.  Without this
            // preference the driver sometimes kept a smaller L1/shared split, fewer blocks fit,
            // and the grid ran as 1.5 waves (the edge kernel measured 1.35 ms instead of 0.87 ms
            // in some processes).
            ce = cudaFuncSetAttribute(f, cudaFuncAttributePreferredSharedMemoryCarveout,
                                      int(cudaSharedmemCarveoutMaxShared));
            if (ce != cudaSuccess) {
                *err = std::string("cudaFuncSetAttribute(carveout, ") + k.name + "): " + cudaGetErrorString(ce);
                cudaLibraryUnload(m.lib);
                return UVU_ERR_CUDA;
            }
        }
        int occ = 0;
        ce = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, f, k.g->threads, k.g->smem);
        if (ce != cudaSuccess || occ < 1) {
            *err = std::string("kernel ") + k.name + " cannot be resident (" +
                   (ce != cudaSuccess ? cudaGetErrorString(ce) : "occupancy 0") + ")";
            cudaLibraryUnload(m.lib);
            return UVU_ERR_UNSUPPORTED;
        }
        *k.occ = occ;
    }
    ce = cudaDeviceGetAttribute(&m.sm_count, cudaDevAttrMultiProcessorCount, dev);
    if (ce == cudaSuccess) {
        size_t bytes = 0;
        void* ptr = nullptr;
        ce = cudaLibraryGetGlobal(&ptr, &bytes, m.lib, "uvu_status_word");
        m.status_word = static_cast<unsigned*>(ptr);
    }
    if (ce != cudaSuccess) {
        *err = std::string("module set-up: ") + cudaGetErrorString(ce);
        cudaLibraryUnload(m.lib);
        return UVU_ERR_CUDA;
    }
    if (std::getenv("UVU_DEBUG")) {  // diagnostics of the loaded module (a debugging switch)
        std::fprintf(stderr, "[uvu] device %d sms %d occupancy fwd %d edge %d dx %d minb %d/%d/%d spills %zu/%zu/%zu\n", dev,
                     m.sm_count, m.occ_fwd, m.occ_edge, m.occ_dx, plan->minb_eff[0], plan->minb_eff[1],
                     plan->minb_eff[2], spill_bytes(plan->log, "uvu_fwd"), spill_bytes(plan->log, "uvu_bwd_edge"),
                     spill_bytes(plan->log, "uvu_bwd_dx"));
        for (const char* k : {"uvu_fwd", "uvu_bwd_edge", "uvu_bwd_dx"}) {
            const std::string key = std::string("Function properties for ") + k + "\n";
            const size_t at = plan->log.find(key);
            if (at != std::string::npos) {
                const size_t u = plan->log.find("Used ", at);
                const size_t e = plan->log.find('\n', u);
                std::fprintf(stderr, "[uvu]   %s: %s\n", k, plan->log.substr(u, e - u).c_str());
            }
        }
    }
    auto res = plan->modules.emplace(dev, m);
    *out = &res.first->second;
    return UVU_OK;
}

// Auxiliary modules (double backward, batched tensor product): emitted and compiled on the
// host on first use, then loaded once per device with the same launch set-up as the plan's own
// kernels (shared-memory size, carveout, occupancy, status word).  The register-budget retry of
// uvu_plan_create applies too: a pipelined kernel that spills under its budget is rebuilt for
// one resident block fewer.
static uvu_status compile_aux_locked(Plan* plan, int kind, std::string* err) {
    AuxBuild& A = plan->aux[kind];
    if (!A.cubin.empty()) return UVU_OK;
    for (int attempt = 0;; ++attempt) {
        A.source = emit_aux_source(plan, kind);
        CacheEntry e;
        uvu_status s = nvrtc_compile(A.source, &e, err);
        if (s != UVU_OK) return s;
        bool again = false;
        if (kind == AUX_RADIAL) {
            // a spilling fused radial forward forms fewer edges' weights at a time, then gives
            // up a resident block
            if (attempt < 4 && spill_bytes(e.log, kAuxKernelNames[kind][0]) > 32) {
                if (A.radial_ne > 1) A.radial_ne -= 1;
                else if (A.minb_eff[0] > 1) A.minb[0] = A.minb_eff[0] - 1;
                else attempt = 4;
                again = attempt < 4;
            }
        } else {
            for (int k = 0; k < 2 && attempt < 3; ++k)
                if (plan->pipelined_recv && A.minb_eff[k] > 1 && spill_bytes(e.log, kAuxKernelNames[kind][k]) > 32) {
                    A.minb[k] = A.minb_eff[k] - 1;
                    again = true;
                }
        }
        if (!again) {
            A.cubin = std::move(e.cubin);
            A.log = std::move(e.log);
            return UVU_OK;
        }
    }
}

uvu_status compile_aux(Plan* plan, int kind, std::string* err) {
    std::lock_guard<std::mutex> g(plan->mu);
    return compile_aux_locked(plan, kind, err);
}

uvu_status aux_module_for_current_device(Plan* plan, int kind, DeviceModule** out, std::string* err) {
    DeviceModule* m = nullptr;
    uvu_status s = module_for_current_device(plan, &m, err);
    if (s != UVU_OK) return s;
    std::lock_guard<std::mutex> g(plan->mu);
    s = compile_aux_locked(plan, kind, err);
    if (s != UVU_OK) return s;
    AuxBuild& A = plan->aux[kind];
    AuxLoaded& L = m->aux[kind];
    if (!L.lib) {
        cudaError_t ce = cudaLibraryLoadData(&L.lib, A.cubin.data(), nullptr, nullptr, 0, nullptr, nullptr, 0);
        for (int k = 0; k < 2 && ce == cudaSuccess; ++k) {
            if (!kAuxKernelNames[kind][k]) continue;  // one-kernel module
            ce = cudaLibraryGetKernel(&L.k[k], L.lib, kAuxKernelNames[kind][k]);
            const void* f = reinterpret_cast<const void*>(L.k[k]);
            if (ce == cudaSuccess && A.g[k].smem > 48 * 1024)
                ce = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, int(A.g[k].smem));
            if (ce == cudaSuccess && A.g[k].persistent)
                ce = cudaFuncSetAttribute(f, cudaFuncAttributePreferredSharedMemoryCarveout, int(cudaSharedmemCarveoutMaxShared));
            if (ce == cudaSuccess) ce = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&L.occ[k], f, A.g[k].threads, A.g[k].smem);
            if (ce == cudaSuccess && L.occ[k] < 1) ce = cudaErrorInvalidConfiguration;
        }
        if (ce == cudaSuccess && plan->pipelined_recv) {
            size_t bytes = 0;
            void* ptr = nullptr;
            ce = cudaLibraryGetGlobal(&ptr, &bytes, L.lib, "uvu_status_word");
            L.status_word = static_cast<unsigned*>(ptr);
        }
        if (ce != cudaSuccess) {
            *err = std::string("loading the ") + kAuxKernelNames[kind][0] + " module: " + cudaGetErrorString(ce);
            if (L.lib) cudaLibraryUnload(L.lib);
            L = AuxLoaded{};
            return UVU_ERR_CUDA;
        }
    }
    *out = m;
    return UVU_OK;
}

}  // namespace uvu
