// The C ABI (include/uvu.h): argument checks on the host, then asynchronous launches on the
// caller's stream.  Nothing here allocates device memory.
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <exception>
#include <limits>
#include <memory>
#include <string>

#include <nvtx3/nvToolsExt.h>

#include "plan.h"

struct uvu_plan_s {
    uvu::Plan p;
};

namespace uvu {
namespace {

// An NVTX range around each C-ABI call, named after the entry point (visible in Nsight traces;
// a no-op without a profiler attached).
struct Range {
    explicit Range(const char* name) { nvtxRangePushA(name); }
    ~Range() { nvtxRangePop(); }
    Range(const Range&) = delete;
    Range& operator=(const Range&) = delete;
};
#define UVU_RANGE(name) ::uvu::Range uvu_nvtx_range_(name)

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

uvu_status need(const void* p, const char* name) {
    if (!p) return fail(UVU_ERR_INVALID_ARGUMENT, std::string(name) + " is NULL");
    if (!aligned16(p)) return fail(UVU_ERR_INVALID_ARGUMENT, std::string(name) + " is not 16-byte aligned");
    return UVU_OK;
}

// Index arrays (int32) are read with scalar loads: 4-byte alignment is enough, which lets a
// caller pass a receiver sub-range (recv_offsets + r0) of a larger CSR.
uvu_status need_idx(const void* p, const char* name) {
    if (!p) return fail(UVU_ERR_INVALID_ARGUMENT, std::string(name) + " is NULL");
    if (reinterpret_cast<uintptr_t>(p) & 3u) return fail(UVU_ERR_INVALID_ARGUMENT, std::string(name) + " is not 4-byte aligned");
    return UVU_OK;
}

uvu_status opt(const void* p, const char* name) {
    if (p && !aligned16(p)) return fail(UVU_ERR_INVALID_ARGUMENT, std::string(name) + " is not 16-byte aligned");
    return UVU_OK;
}

uvu_status check_sizes(int64_t N, int64_t E) {
    if (N < 0 || E < 0) return fail(UVU_ERR_INVALID_ARGUMENT, "n_nodes and n_edges must be >= 0");
    if (N >= std::numeric_limits<int32_t>::max() || E >= std::numeric_limits<int32_t>::max())
        return fail(UVU_ERR_INVALID_ARGUMENT, "n_nodes and n_edges must be < 2^31 - 1 (int32 indices)");
    return UVU_OK;
}

#define UVU_TRY(expr)                         \
    do {                                      \
        uvu_status _s = (expr);               \
        if (_s != UVU_OK) return _s;          \
    } while (0)

// Grid of a launch: persistent kernels get the resident blocks (at most max_blocks), the others
// one block per owners_per_block owners.
int64_t grid_blocks(int occ, int sm_count, int64_t owners, const KernelGeom& g, int64_t max_blocks) {
    if (g.persistent) return std::min(std::min<int64_t>(owners * g.tiles, int64_t(occ) * sm_count), max_blocks);
    return (owners + g.owners_per_block - 1) / g.owners_per_block;
}

uvu_status launch(cudaKernel_t k, int occ, int sm_count, int64_t owners, const KernelGeom& g, void** args,
                  cudaStream_t st, const char* what, int64_t max_blocks = INT64_MAX) {
    if (owners <= 0) return UVU_OK;
    const int64_t blocks = grid_blocks(occ, sm_count, owners, g, max_blocks);
    cudaError_t e = cudaLaunchKernel(reinterpret_cast<const void*>(k), dim3(unsigned(blocks)),
                                     dim3(unsigned(g.threads)), args, g.smem, st);
    if (e != cudaSuccess) return cuda_fail(e, what);
    return UVU_OK;
}

Plan* get(uvu_plan_t h) { return h ? &h->p : nullptr; }

}  // namespace
}  // namespace uvu

using namespace uvu;

extern "C" uvu_status uvu_plan_create(const char* irreps_x, const char* irreps_sh, int lmax_out,
                                      uvu_dtype dtype, uvu_plan_t* plan_out) {
    UVU_RANGE("uvu_plan_create");
    if (!plan_out) return fail(UVU_ERR_INVALID_ARGUMENT, "plan_out is NULL");
    *plan_out = nullptr;
    if (!irreps_x || !irreps_sh) return fail(UVU_ERR_INVALID_ARGUMENT, "irreps string is NULL");
    if (dtype != UVU_F32 && dtype != UVU_F64) return fail(UVU_ERR_INVALID_ARGUMENT, "dtype must be UVU_F32 or UVU_F64");
    try {
        std::unique_ptr<uvu_plan_s> h(new uvu_plan_s);
        Plan& p = h->p;
        p.irreps_x = irreps_x;
        p.irreps_sh = irreps_sh;
        p.lmax_out = lmax_out;
        p.dtype = dtype;
        std::string err;
        uvu_status s = build_paths(&p, &err);
        if (s != UVU_OK) return fail(s, err);
        // Compile with a register budget sized for as many resident blocks per SM as the shared
        // memory allows (up to 4); a kernel that spills more than a call-site save under that
        // budget is recompiled for one block fewer.
        for (int attempt = 0; attempt < 4; ++attempt) {
            p.source = emit_source(&p);
            if (p.g_fwd.threads > 1024 || p.g_edge.threads > 1024 || p.g_dx.threads > 1024)
                return fail(UVU_ERR_UNSUPPORTED, "multiplicity x register groups exceeds 1024 threads per owner");
            s = compile_plan(&p, &err);
            if (s != UVU_OK) return fail(s, err);
            const char* names[3] = {"uvu_fwd", "uvu_bwd_edge", "uvu_bwd_dx"};
            // UVU_PIPE_SPILL_OK=n (a tuning switch): spill bytes accepted before a kernel gives up
            // a resident block (default 32, about one call-site save)
            size_t spill_ok = 32;
            if (const char* e2 = std::getenv("UVU_PIPE_SPILL_OK")) spill_ok = size_t(std::max(0, std::atoi(e2)));
            bool again = false;
            for (int k = 0; k < 3; ++k)
                if (p.minb_eff[k] > 1 && spill_bytes(p.log, names[k]) > spill_ok) {
                    p.minb[k] = p.minb_eff[k] - 1;
                    again = true;
                }
            if (!again) break;
        }
        *plan_out = h.release();
        return ok();
    } catch (const std::exception& e) {
        return fail(UVU_ERR_UNSUPPORTED, std::string("plan creation failed: ") + e.what());
    }
}

extern "C" uvu_status uvu_plan_destroy(uvu_plan_t plan) {
    UVU_RANGE("uvu_plan_destroy");
    if (!plan) return ok();
    for (auto& kv : plan->p.modules) {
        int cur = 0;
        if (cudaGetDevice(&cur) == cudaSuccess && cur != kv.first) cudaSetDevice(kv.first);
        cudaLibraryUnload(kv.second.lib);
        for (auto& a : kv.second.aux)
            if (a.lib) cudaLibraryUnload(a.lib);
        if (cur != kv.first) cudaSetDevice(cur);
    }
    delete plan;
    return ok();
}

extern "C" uvu_status uvu_plan_info(uvu_plan_t plan, int* mul_u, int* dim_x, int* dim_sh, int* dim_out,
                                    int* n_paths, int* paths_l1l2l3) {
    Plan* p = get(plan);
    if (!p) return fail(UVU_ERR_INVALID_ARGUMENT, "plan is NULL");
    if (mul_u) *mul_u = p->U;
    if (dim_x) *dim_x = p->Dx;
    if (dim_sh) *dim_sh = p->Dy;
    if (dim_out) *dim_out = p->Do;
    if (n_paths) *n_paths = p->P;
    if (paths_l1l2l3)
        for (int i = 0; i < p->P; ++i) {
            paths_l1l2l3[3 * i] = p->paths[i].l1;
            paths_l1l2l3[3 * i + 1] = p->paths[i].l2;
            paths_l1l2l3[3 * i + 2] = p->paths[i].l3;
        }
    return ok();
}

extern "C" uvu_status uvu_plan_cg(uvu_plan_t plan, int path, double* out) {
    Plan* p = get(plan);
    if (!p || !out) return fail(UVU_ERR_INVALID_ARGUMENT, "plan or out is NULL");
    if (path < 0 || path >= p->P) return fail(UVU_ERR_INVALID_ARGUMENT, "path index out of range");
    std::memcpy(out, p->paths[path].cg.data(), p->paths[path].cg.size() * sizeof(double));
    return ok();
}

extern "C" uvu_status uvu_plan_source(uvu_plan_t plan, const char** source, const char** log) {
    Plan* p = get(plan);
    if (!p) return fail(UVU_ERR_INVALID_ARGUMENT, "plan is NULL");
    if (source) *source = p->source.c_str();
    if (log) *log = p->log.c_str();
    return ok();
}

extern "C" uvu_status uvu_plan_module_source(uvu_plan_t plan, uvu_module module, const char** source, const char** log) {
    UVU_RANGE("uvu_plan_module_source");
    Plan* p = get(plan);
    if (!p) return fail(UVU_ERR_INVALID_ARGUMENT, "plan is NULL");
    if (module == UVU_MODULE_CONV) return uvu_plan_source(plan, source, log);
    const int kind = module == UVU_MODULE_HVP ? AUX_HVP : module == UVU_MODULE_TP ? AUX_TP
                   : module == UVU_MODULE_TP_SHARED ? AUX_TP_SHARED : -1;
    if (kind < 0) return fail(UVU_ERR_INVALID_ARGUMENT, "unknown module");
    std::string err;
    uvu_status s = compile_aux(p, kind, &err);
    if (s != UVU_OK) return fail(s, err);
    if (source) *source = p->aux[kind].source.c_str();
    if (log) *log = p->aux[kind].log.c_str();
    return ok();
}

extern "C" uvu_status uvu_csr_from_sorted_recv(int64_t n_nodes, int64_t n_edges, const int32_t* recv,
                                               int32_t* recv_offsets, uvu_stream_t stream) {
    UVU_RANGE("uvu_csr_from_sorted_recv");
    UVU_TRY(check_sizes(n_nodes, n_edges));
    if (!recv_offsets) return fail(UVU_ERR_INVALID_ARGUMENT, "recv_offsets is NULL");
    if (n_edges > 0 && !recv) return fail(UVU_ERR_INVALID_ARGUMENT, "recv is NULL");
    cudaError_t e = launch_csr_offsets(n_nodes, n_edges, recv, recv_offsets, stream);
    if (e != cudaSuccess) return cuda_fail(e, "csr offsets launch");
    return ok();
}

extern "C" uvu_status uvu_csr_transpose_workspace(int64_t n_nodes, int64_t n_edges, size_t* bytes) {
    UVU_TRY(check_sizes(n_nodes, n_edges));
    if (!bytes) return fail(UVU_ERR_INVALID_ARGUMENT, "bytes is NULL");
    *bytes = transpose_workspace_bytes(n_nodes, n_edges);
    return ok();
}

extern "C" uvu_status uvu_csr_transpose(int64_t n_nodes, int64_t n_edges, const int32_t* recv_offsets,
                                        const int32_t* src, int32_t* send_offsets, int32_t* send_eids,
                                        int32_t* send_recv, void* workspace, size_t workspace_bytes,
                                        uvu_stream_t stream) {
    UVU_RANGE("uvu_csr_transpose");
    UVU_TRY(check_sizes(n_nodes, n_edges));
    if (!send_offsets || !workspace) return fail(UVU_ERR_INVALID_ARGUMENT, "send_offsets or workspace is NULL");
    if (n_edges > 0 && (!recv_offsets || !src || !send_eids || !send_recv))
        return fail(UVU_ERR_INVALID_ARGUMENT, "graph pointer is NULL");
    if (!aligned16(workspace)) return fail(UVU_ERR_INVALID_ARGUMENT, "workspace is not 16-byte aligned");
    if (workspace_bytes < transpose_workspace_bytes(n_nodes, n_edges))
        return fail(UVU_ERR_INVALID_ARGUMENT, "workspace too small");
    cudaError_t e = launch_csr_transpose(n_nodes, n_edges, recv_offsets, src, send_offsets, send_eids,
                                         send_recv, workspace, stream);
    if (e != cudaSuccess) return cuda_fail(e, "csr transpose launch");
    return ok();
}

extern "C" uvu_status uvu_graph_validate(int64_t n_nodes, int64_t n_edges, const int32_t* recv_offsets,
                                         const int32_t* src, void* workspace, int64_t* n_bad,
                                         uvu_stream_t stream) {
    UVU_RANGE("uvu_graph_validate");
    UVU_TRY(check_sizes(n_nodes, n_edges));
    if (!recv_offsets || !workspace || !n_bad || (n_edges > 0 && !src))
        return fail(UVU_ERR_INVALID_ARGUMENT, "NULL argument");
    auto* bad = static_cast<unsigned long long*>(workspace);
    cudaError_t e = launch_graph_validate(n_nodes, n_edges, recv_offsets, src, bad, stream);
    if (e != cudaSuccess) return cuda_fail(e, "validate launch");
    unsigned long long h = 0;
    e = cudaMemcpyAsync(&h, bad, sizeof h, cudaMemcpyDeviceToHost, stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) return cuda_fail(e, "validate readback");
    *n_bad = int64_t(h);
    return ok();
}

extern "C" uvu_status uvu_conv_fwd(uvu_plan_t plan, int64_t n_nodes, int64_t n_edges, const void* x,
                                   const void* Y, const void* w, const int32_t* recv_offsets,
                                   const int32_t* src, void* out, uvu_stream_t stream) {
    UVU_RANGE("uvu_conv_fwd");
    Plan* p = get(plan);
    if (!p) return fail(UVU_ERR_INVALID_ARGUMENT, "plan is NULL");
    UVU_TRY(check_sizes(n_nodes, n_edges));
    if (n_nodes == 0) return ok();
    UVU_TRY(need(out, "out"));
    UVU_TRY(need_idx(recv_offsets, "recv_offsets"));
    if (n_edges > 0) {
        UVU_TRY(need(x, "x"));
        UVU_TRY(need(Y, "Y"));
        UVU_TRY(need(w, "w"));
        UVU_TRY(need_idx(src, "src"));
    }
    DeviceModule* m = nullptr;
    std::string err;
    uvu_status s = module_for_current_device(p, &m, &err);
    if (s != UVU_OK) return fail(s, err);
    long long N = n_nodes;
    void* args[] = {&N, &recv_offsets, &src, &x, &Y, &w, &out};
    UVU_TRY(launch(m->fwd, m->occ_fwd, m->sm_count, n_nodes, p->g_fwd, args, stream, "uvu_fwd launch"));
    return ok();
}

extern "C" uvu_status uvu_conv_bwd_edge(uvu_plan_t plan, int64_t n_nodes, int64_t n_edges, const void* x,
                                        const void* Y, const void* w, const int32_t* recv_offsets,
                                        const int32_t* src, const void* d_out, void* dY, void* dw,
                                        void* dx_atomic, void* dx_edge, uvu_stream_t stream) {
    UVU_RANGE("uvu_conv_bwd_edge");
    Plan* p = get(plan);
    if (!p) return fail(UVU_ERR_INVALID_ARGUMENT, "plan is NULL");
    UVU_TRY(check_sizes(n_nodes, n_edges));
    UVU_TRY(opt(dY, "dY"));
    UVU_TRY(opt(dw, "dw"));
    UVU_TRY(opt(dx_atomic, "dx"));
    UVU_TRY(opt(dx_edge, "dx_edge"));
    if (dx_edge && !p->staged_ok)
        return fail(UVU_ERR_UNSUPPORTED, "per-edge dx partials need the pipelined kernels or a single register group");
    if (n_nodes == 0 || (!dY && !dw && !dx_atomic && !dx_edge)) return ok();
    UVU_TRY(need_idx(recv_offsets, "recv_offsets"));
    if (n_edges > 0) {
        UVU_TRY(need(x, "x"));
        UVU_TRY(need(Y, "Y"));
        UVU_TRY(need(w, "w"));
        UVU_TRY(need_idx(src, "src"));
        UVU_TRY(need(d_out, "d_out"));
    }
    DeviceModule* m = nullptr;
    std::string err;
    uvu_status s = module_for_current_device(p, &m, &err);
    if (s != UVU_OK) return fail(s, err);
    if (dx_atomic) {
        cudaError_t e = cudaMemsetAsync(dx_atomic, 0, size_t(n_nodes) * p->U * p->Dx * p->elem(), stream);
        if (e != cudaSuccess) return cuda_fail(e, "dx memset");
    }
    if (n_edges == 0) return ok();
    long long N = n_nodes;
    void* args[] = {&N, &recv_offsets, &src, &x, &Y, &w, &d_out, &dY, &dw, &dx_atomic, &dx_edge};
    UVU_TRY(launch(m->bwd_edge, m->occ_edge, m->sm_count, n_nodes, p->g_edge, args, stream, "uvu_bwd_edge launch"));
    return ok();
}

extern "C" uvu_status uvu_conv_bwd_dx_reduce(uvu_plan_t plan, int64_t n_nodes, int64_t n_edges,
                                             const int32_t* send_offsets, const int32_t* send_eids,
                                             const void* dx_edge, void* dx, uvu_stream_t stream) {
    UVU_RANGE("uvu_conv_bwd_dx_reduce");
    Plan* p = get(plan);
    if (!p) return fail(UVU_ERR_INVALID_ARGUMENT, "plan is NULL");
    UVU_TRY(check_sizes(n_nodes, n_edges));
    if (n_nodes == 0) return ok();
    UVU_TRY(need(dx, "dx"));
    UVU_TRY(need_idx(send_offsets, "send_offsets"));
    if (n_edges > 0) {
        UVU_TRY(need_idx(send_eids, "send_eids"));
        UVU_TRY(need(dx_edge, "dx_edge"));
    }
    DeviceModule* m = nullptr;
    std::string err;
    uvu_status s = module_for_current_device(p, &m, &err);
    if (s != UVU_OK) return fail(s, err);
    long long N = n_nodes;
    void* args[] = {&N, &send_offsets, &send_eids, &dx_edge, &dx};
    const int64_t threads = n_nodes * (p->reduce_per_sender > 0 ? p->reduce_per_sender : p->U_pad);
    const KernelGeom g{256, 256, 0, false, 1};
    UVU_TRY(launch(m->bwd_dx_reduce, 1, m->sm_count, threads, g, args, stream, "uvu_bwd_dx_reduce launch"));
    return ok();
}

extern "C" uvu_status uvu_conv_bwd_workspace(uvu_plan_t plan, int64_t n_nodes, int64_t n_edges,
                                             uvu_dx_mode dx_mode, size_t* bytes) {
    Plan* p = get(plan);
    if (!p || !bytes) return fail(UVU_ERR_INVALID_ARGUMENT, "plan or bytes is NULL");
    UVU_TRY(check_sizes(n_nodes, n_edges));
    *bytes = dx_mode == UVU_DX_STAGED ? size_t(n_edges) * p->U * p->Dx * p->elem() : 0;
    return ok();
}

extern "C" uvu_status uvu_conv_bwd_dx(uvu_plan_t plan, int64_t n_nodes, int64_t n_edges, const void* Y,
                                      const void* w, const int32_t* send_offsets, const int32_t* send_eids,
                                      const int32_t* send_recv, const void* d_out, void* dx,
                                      uvu_stream_t stream) {
    UVU_RANGE("uvu_conv_bwd_dx");
    Plan* p = get(plan);
    if (!p) return fail(UVU_ERR_INVALID_ARGUMENT, "plan is NULL");
    UVU_TRY(check_sizes(n_nodes, n_edges));
    if (n_nodes == 0) return ok();
    UVU_TRY(need(dx, "dx"));
    UVU_TRY(need_idx(send_offsets, "send_offsets"));
    if (n_edges > 0) {
        UVU_TRY(need(Y, "Y"));
        UVU_TRY(need(w, "w"));
        UVU_TRY(need_idx(send_eids, "send_eids"));
        UVU_TRY(need_idx(send_recv, "send_recv"));
        UVU_TRY(need(d_out, "d_out"));
    }
    DeviceModule* m = nullptr;
    std::string err;
    uvu_status s = module_for_current_device(p, &m, &err);
    if (s != UVU_OK) return fail(s, err);
    long long N = n_nodes;
    void* args[] = {&N, &send_offsets, &send_eids, &send_recv, &Y, &w, &d_out, &dx};
    UVU_TRY(launch(m->bwd_dx, m->occ_dx, m->sm_count, n_nodes, p->g_dx, args, stream, "uvu_bwd_dx launch"));
    return ok();
}

extern "C" uvu_status uvu_conv_bwd(uvu_plan_t plan, int64_t n_nodes, int64_t n_edges, const void* x,
                                   const void* Y, const void* w, const int32_t* recv_offsets,
                                   const int32_t* src, const int32_t* send_offsets, const int32_t* send_eids,
                                   const int32_t* send_recv, const void* d_out, void* dx, void* dY, void* dw,
                                   uvu_dx_mode dx_mode, void* workspace, size_t workspace_bytes,
                                   uvu_stream_t stream) {
    UVU_RANGE("uvu_conv_bwd");
    if (dx_mode != UVU_DX_SENDER && dx_mode != UVU_DX_ATOMIC && dx_mode != UVU_DX_STAGED)
        return fail(UVU_ERR_INVALID_ARGUMENT, "dx_mode must be UVU_DX_SENDER, UVU_DX_ATOMIC or UVU_DX_STAGED");
    if (dx_mode == UVU_DX_ATOMIC)
        return uvu_conv_bwd_edge(plan, n_nodes, n_edges, x, Y, w, recv_offsets, src, d_out, dY, dw, dx, nullptr, stream);
    if (dx_mode == UVU_DX_STAGED && dx) {
        size_t need_bytes = 0;
        UVU_TRY(uvu_conv_bwd_workspace(plan, n_nodes, n_edges, dx_mode, &need_bytes));
        if (need_bytes && (!workspace || workspace_bytes < need_bytes))
            return fail(UVU_ERR_INVALID_ARGUMENT, "UVU_DX_STAGED needs a workspace of uvu_conv_bwd_workspace() bytes");
        UVU_TRY(opt(workspace, "workspace"));
        UVU_TRY(uvu_conv_bwd_edge(plan, n_nodes, n_edges, x, Y, w, recv_offsets, src, d_out, dY, dw, nullptr,
                                  need_bytes ? workspace : nullptr, stream));
        UVU_TRY(uvu_conv_bwd_dx_reduce(plan, n_nodes, n_edges, send_offsets, send_eids, workspace, dx, stream));
        return ok();
    }
    UVU_TRY(uvu_conv_bwd_edge(plan, n_nodes, n_edges, x, Y, w, recv_offsets, src, d_out, dY, dw, nullptr, nullptr,
                              stream));
    if (dx)
        UVU_TRY(uvu_conv_bwd_dx(plan, n_nodes, n_edges, Y, w, send_offsets, send_eids, send_recv, d_out, dx, stream));
    return ok();
}

extern "C" uvu_status uvu_plan_device_status(uvu_plan_t plan, unsigned* word, int reset) {
    UVU_RANGE("uvu_plan_device_status");
    Plan* p = get(plan);
    if (!p || !word) return fail(UVU_ERR_INVALID_ARGUMENT, "plan or word is NULL");
    DeviceModule* m = nullptr;
    std::string err;
    uvu_status s = module_for_current_device(p, &m, &err);
    if (s != UVU_OK) return fail(s, err);
    cudaError_t e = cudaMemcpy(word, m->status_word, sizeof(unsigned), cudaMemcpyDeviceToHost);
    for (auto& a : m->aux) {  // the auxiliary modules' own words
        if (e != cudaSuccess || !a.status_word) continue;
        unsigned w2 = 0;
        e = cudaMemcpy(&w2, a.status_word, sizeof(unsigned), cudaMemcpyDeviceToHost);
        *word |= w2;
    }
    if (e == cudaSuccess) {  // the tensor-core product kernels' word (shared by all plans)
        unsigned w3 = 0;
        e = tc_status(&w3, reset != 0);
        *word |= w3;
    }
    if (e == cudaSuccess && reset) {
        const unsigned zero = 0;
        e = cudaMemcpy(m->status_word, &zero, sizeof(unsigned), cudaMemcpyHostToDevice);
        for (auto& a : m->aux)
            if (e == cudaSuccess && a.status_word) e = cudaMemcpy(a.status_word, &zero, sizeof(unsigned), cudaMemcpyHostToDevice);
    }
    if (e != cudaSuccess) return cuda_fail(e, "status word copy");
    return ok();
}

extern "C" uvu_status uvu_conv_hvp_workspace(uvu_plan_t plan, int64_t n_nodes, int64_t n_edges, size_t* bytes) {
    Plan* p = get(plan);
    if (!p || !bytes) return fail(UVU_ERR_INVALID_ARGUMENT, "plan or bytes is NULL");
    UVU_TRY(check_sizes(n_nodes, n_edges));
    // per-edge grad_x partials: written by the pipelined kernels for any register grouping and by
    // the direct-load kernels with one group; otherwise grad_x is accumulated with atomics
    *bytes = (p->pipelined_recv || p->groups.size() == 1) ? size_t(n_edges) * p->U * p->Dx * p->elem() : 0;
    return ok();
}

extern "C" uvu_status uvu_conv_hvp(uvu_plan_t plan, int64_t n_nodes, int64_t n_edges, const void* x,
                                   const void* Y, const void* w, const int32_t* recv_offsets,
                                   const int32_t* src, const int32_t* send_offsets, const int32_t* send_eids,
                                   const void* d_out, const void* ax, const void* aY, const void* aw,
                                   void* grad_d_out, void* grad_x, void* grad_Y, void* grad_w, void* workspace,
                                   size_t workspace_bytes, uvu_stream_t stream) {
    UVU_RANGE("uvu_conv_hvp");
    Plan* p = get(plan);
    if (!p) return fail(UVU_ERR_INVALID_ARGUMENT, "plan is NULL");
    UVU_TRY(check_sizes(n_nodes, n_edges));
    for (auto& kv : {std::make_pair(ax, "ax"), std::make_pair(aY, "aY"), std::make_pair(aw, "aw"),
                     std::make_pair(static_cast<const void*>(grad_d_out), "grad_d_out"),
                     std::make_pair(static_cast<const void*>(grad_x), "grad_x"),
                     std::make_pair(static_cast<const void*>(grad_Y), "grad_Y"),
                     std::make_pair(static_cast<const void*>(grad_w), "grad_w")})
        UVU_TRY(opt(kv.first, kv.second));
    if (n_nodes == 0 || (!grad_d_out && !grad_x && !grad_Y && !grad_w)) return ok();
    UVU_TRY(need_idx(recv_offsets, "recv_offsets"));
    const bool need_edge = grad_x || grad_Y || grad_w;
    if (n_edges > 0) {
        UVU_TRY(need(x, "x"));
        UVU_TRY(need(Y, "Y"));
        UVU_TRY(need(w, "w"));
        UVU_TRY(need_idx(src, "src"));
        if (need_edge) UVU_TRY(need(d_out, "d_out"));
    }
    size_t ws_need = 0;
    UVU_TRY(uvu_conv_hvp_workspace(plan, n_nodes, n_edges, &ws_need));
    const bool staged = grad_x && ws_need > 0;
    if (grad_x) {
        UVU_TRY(need_idx(send_offsets, "send_offsets"));
        if (n_edges > 0 && staged) UVU_TRY(need_idx(send_eids, "send_eids"));
        if (staged && (!workspace || workspace_bytes < ws_need))
            return fail(UVU_ERR_INVALID_ARGUMENT, "grad_x needs a workspace of uvu_conv_hvp_workspace() bytes");
        UVU_TRY(opt(workspace, "workspace"));
    }
    DeviceModule* m = nullptr;
    std::string err;
    uvu_status s = aux_module_for_current_device(p, AUX_HVP, &m, &err);
    if (s != UVU_OK) return fail(s, err);
    const AuxLoaded& L = m->aux[AUX_HVP];
    const AuxBuild& A = p->aux[AUX_HVP];
    const int hm = (ax ? 1 : 0) | (aY ? 2 : 0) | (aw ? 4 : 0);
    long long N = n_nodes;
    if (grad_d_out) {
        void* args[] = {&N, &recv_offsets, &src, &x, &Y, &w, &ax, &aY, &aw, const_cast<int*>(&hm), &grad_d_out};
        UVU_TRY(launch(L.k[0], L.occ[0], m->sm_count, n_nodes, A.g[0], args, stream, "uvu_hvp_fwd launch"));
    }
    if (!need_edge) return ok();
    void* dx_atomic = (grad_x && !staged) ? grad_x : nullptr;
    void* dx_edge = staged ? workspace : nullptr;
    if (dx_atomic) {
        cudaError_t e = cudaMemsetAsync(dx_atomic, 0, size_t(n_nodes) * p->U * p->Dx * p->elem(), stream);
        if (e != cudaSuccess) return cuda_fail(e, "grad_x memset");
    }
    if (n_edges > 0) {
        void* args[] = {&N, &recv_offsets, &src, &x, &Y, &w, &d_out, &ax, &aY, &aw, const_cast<int*>(&hm),
                        &grad_Y, &grad_w, &dx_atomic, &dx_edge};
        UVU_TRY(launch(L.k[1], L.occ[1], m->sm_count, n_nodes, A.g[1], args, stream, "uvu_hvp_edge launch"));
    }
    if (staged) UVU_TRY(uvu_conv_bwd_dx_reduce(plan, n_nodes, n_edges, send_offsets, send_eids, workspace, grad_x, stream));
    return ok();
}

// ------------------------------------------------- receiver- vs sender-stationary forward

namespace uvu {
namespace {
// Bytes each forward moves through the memory system per launch (the data-movement model):
// receiver-stationary gathers an x row per edge and writes each out row once; sender-stationary
// reads each x row once, zero-fills out and read-modify-writes an out row per edge.
void fwd_model(const Plan* p, int64_t N, int64_t E, double* br, double* bs) {
    const double s = double(p->elem()), U = p->U;
    const double wY = double(E) * (p->P * U + p->Dy) * s;
    *br = wY + double(E) * U * p->Dx * s + double(N) * U * p->Do * s + 4.0 * (N + 1) + 4.0 * E;
    *bs = wY + double(N) * U * p->Dx * s + double(N) * U * p->Do * s + 2.0 * double(E) * U * p->Do * s +
          4.0 * (N + 1) + 8.0 * E;
}
}  // namespace
}  // namespace uvu

extern "C" uvu_status uvu_conv_fwd_model(uvu_plan_t plan, int64_t n_nodes, int64_t n_edges, uvu_fwd_mode* choice,
                                         double* bytes_receiver, double* bytes_sender) {
    Plan* p = get(plan);
    if (!p) return fail(UVU_ERR_INVALID_ARGUMENT, "plan is NULL");
    UVU_TRY(check_sizes(n_nodes, n_edges));
    double br = 0, bs = 0;
    fwd_model(p, n_nodes, n_edges, &br, &bs);
    if (choice) *choice = bs < br ? UVU_FWD_SENDER : UVU_FWD_RECEIVER;
    if (bytes_receiver) *bytes_receiver = br;
    if (bytes_sender) *bytes_sender = bs;
    return ok();
}

extern "C" uvu_status uvu_conv_fwd_sender(uvu_plan_t plan, int64_t n_nodes, int64_t n_edges, const void* x,
                                          const void* Y, const void* w, const int32_t* send_offsets,
                                          const int32_t* send_eids, const int32_t* send_recv, void* out,
                                          uvu_stream_t stream) {
    UVU_RANGE("uvu_conv_fwd_sender");
    Plan* p = get(plan);
    if (!p) return fail(UVU_ERR_INVALID_ARGUMENT, "plan is NULL");
    UVU_TRY(check_sizes(n_nodes, n_edges));
    if (n_nodes == 0) return ok();
    UVU_TRY(need(out, "out"));
    cudaError_t e = cudaMemsetAsync(out, 0, size_t(n_nodes) * p->U * p->Do * p->elem(), stream);
    if (e != cudaSuccess) return cuda_fail(e, "out memset");
    if (n_edges == 0) return ok();
    UVU_TRY(need(x, "x"));
    UVU_TRY(need(Y, "Y"));
    UVU_TRY(need(w, "w"));
    UVU_TRY(need_idx(send_offsets, "send_offsets"));
    UVU_TRY(need_idx(send_eids, "send_eids"));
    UVU_TRY(need_idx(send_recv, "send_recv"));
    DeviceModule* m = nullptr;
    std::string err;
    uvu_status s = module_for_current_device(p, &m, &err);
    if (s != UVU_OK) return fail(s, err);
    long long N = n_nodes;
    void* args[] = {&N, &send_offsets, &send_eids, &send_recv, &x, &Y, &w, &out};
    return launch(m->fwd_sender, 1, m->sm_count, n_nodes, p->g_fwd_sender, args, stream, "uvu_fwd_sender launch");
}

extern "C" uvu_status uvu_conv_fwd_mode(uvu_plan_t plan, uvu_fwd_mode mode, int64_t n_nodes, int64_t n_edges,
                                        const void* x, const void* Y, const void* w, const int32_t* recv_offsets,
                                        const int32_t* src, const int32_t* send_offsets, const int32_t* send_eids,
                                        const int32_t* send_recv, void* out, uvu_stream_t stream) {
    UVU_RANGE("uvu_conv_fwd_mode");
    if (mode == UVU_FWD_AUTO) UVU_TRY(uvu_conv_fwd_model(plan, n_nodes, n_edges, &mode, nullptr, nullptr));
    if (mode == UVU_FWD_RECEIVER) return uvu_conv_fwd(plan, n_nodes, n_edges, x, Y, w, recv_offsets, src, out, stream);
    if (mode == UVU_FWD_SENDER)
        return uvu_conv_fwd_sender(plan, n_nodes, n_edges, x, Y, w, send_offsets, send_eids, send_recv, out, stream);
    return fail(UVU_ERR_INVALID_ARGUMENT, "unknown forward mode");
}

// ------------------------------------------ channel mixing (factorised UVW -> UVU convolution)

namespace uvu {
namespace {
uvu_status mix_check(Plan* p, int64_t N, int W) {
    if (!p) return fail(UVU_ERR_INVALID_ARGUMENT, "plan is NULL");
    if (N < 0) return fail(UVU_ERR_INVALID_ARGUMENT, "n_nodes < 0");
    if (W < 1 || W > 4096) return fail(UVU_ERR_INVALID_ARGUMENT, "w_out must be in [1, 4096]");
    if (p->P > mix_max_paths()) return fail(UVU_ERR_UNSUPPORTED, "too many paths for the mixing kernels");
    return UVU_OK;
}
}  // namespace
}  // namespace uvu

extern "C" uvu_status uvu_mix_workspace(uvu_plan_t plan, int64_t n_nodes, int w_out, size_t* fwd_bytes,
                                        size_t* bwd_bytes) {
    Plan* p = get(plan);
    UVU_TRY(mix_check(p, n_nodes, w_out));
    if (fwd_bytes) *fwd_bytes = mix_workspace_bytes(*p, n_nodes, w_out, false);
    if (bwd_bytes) *bwd_bytes = mix_workspace_bytes(*p, n_nodes, w_out, true);
    return ok();
}

extern "C" uvu_status uvu_mix_fwd(uvu_plan_t plan, int64_t n_nodes, int w_out, const void* in, const void* M,
                                  void* out, void* workspace, size_t workspace_bytes, uvu_stream_t stream) {
    UVU_RANGE("uvu_mix_fwd");
    Plan* p = get(plan);
    UVU_TRY(mix_check(p, n_nodes, w_out));
    if (n_nodes == 0) return ok();
    UVU_TRY(need(in, "in"));
    UVU_TRY(need(M, "M"));
    UVU_TRY(need(out, "out"));
    UVU_TRY(need(workspace, "workspace"));
    if (workspace_bytes < mix_workspace_bytes(*p, n_nodes, w_out, false))
        return fail(UVU_ERR_INVALID_ARGUMENT, "workspace smaller than uvu_mix_workspace() reports for the forward");
    cudaError_t e = launch_mix_fwd(*p, n_nodes, w_out, in, M, out, workspace, stream);
    return e == cudaSuccess ? ok() : cuda_fail(e, "uvu_mix_fwd launch");
}

extern "C" uvu_status uvu_mix_bwd(uvu_plan_t plan, int64_t n_nodes, int w_out, const void* in, const void* M,
                                  const void* d_out, void* d_in, void* dM, void* workspace, size_t workspace_bytes,
                                  uvu_stream_t stream) {
    UVU_RANGE("uvu_mix_bwd");
    Plan* p = get(plan);
    UVU_TRY(mix_check(p, n_nodes, w_out));
    UVU_TRY(opt(d_in, "d_in"));
    UVU_TRY(opt(dM, "dM"));
    if (!d_in && !dM) return ok();
    if (n_nodes > 0) {
        UVU_TRY(need(d_out, "d_out"));
        if (d_in) UVU_TRY(need(M, "M"));
        if (dM) UVU_TRY(need(in, "in"));
        UVU_TRY(need(workspace, "workspace"));
        if (workspace_bytes < mix_workspace_bytes(*p, n_nodes, w_out, true))
            return fail(UVU_ERR_INVALID_ARGUMENT, "workspace smaller than uvu_mix_workspace() reports for the backward");
    }
    cudaError_t e = launch_mix_bwd(*p, n_nodes, w_out, in, M, d_out, d_in, dM, workspace, stream);
    return e == cudaSuccess ? ok() : cuda_fail(e, "uvu_mix_bwd launch");
}

extern "C" uvu_status uvu_conv_uvw_fwd(uvu_plan_t plan, int64_t n_nodes, int64_t n_edges, const void* x,
                                       const void* Y, const void* w, const int32_t* recv_offsets,
                                       const int32_t* src, const void* M, int w_out, void* uvu_out, void* out,
                                       void* workspace, size_t workspace_bytes, uvu_stream_t stream) {
    UVU_RANGE("uvu_conv_uvw_fwd");
    UVU_TRY(mix_check(get(plan), n_nodes, w_out));
    UVU_TRY(uvu_conv_fwd(plan, n_nodes, n_edges, x, Y, w, recv_offsets, src, uvu_out, stream));
    return uvu_mix_fwd(plan, n_nodes, w_out, uvu_out, M, out, workspace, workspace_bytes, stream);
}

// ------------------------------------------------------------- batched tensor product (no graph)

namespace uvu {
namespace {
// Grid cap of the batch-shared-weight edge kernel: bounds the rows of its partial-dw workspace.
constexpr int64_t kTpMaxBlocks = 2048;

uvu_status tp_check(Plan* p, int64_t batch) {
    if (!p) return fail(UVU_ERR_INVALID_ARGUMENT, "plan is NULL");
    if (batch < 0 || batch > INT32_MAX - 1) return fail(UVU_ERR_INVALID_ARGUMENT, "batch must be in [0, 2^31 - 1)");
    if (!p->pipelined_recv)
        return fail(UVU_ERR_UNSUPPORTED, "the batched tensor product needs a plan whose kernels are pipelined (U >= 32)");
    return UVU_OK;
}
}  // namespace
}  // namespace uvu

extern "C" uvu_status uvu_tp_bwd_workspace(uvu_plan_t plan, int64_t batch, int w_shared, size_t* bytes) {
    Plan* p = get(plan);
    if (!bytes) return fail(UVU_ERR_INVALID_ARGUMENT, "bytes is NULL");
    UVU_TRY(tp_check(p, batch));
    *bytes = w_shared ? size_t(std::min<int64_t>(batch, kTpMaxBlocks)) * p->P * p->U * sizeof(double) : 0;
    return ok();
}

extern "C" uvu_status uvu_tp_fwd(uvu_plan_t plan, int64_t batch, const void* x, const void* y, const void* w,
                                 int w_shared, void* out, uvu_stream_t stream) {
    UVU_RANGE("uvu_tp_fwd");
    Plan* p = get(plan);
    UVU_TRY(tp_check(p, batch));
    if (batch == 0) return ok();
    UVU_TRY(need(out, "out"));
    UVU_TRY(need(x, "x"));
    UVU_TRY(need(y, "y"));
    UVU_TRY(need(w, "w"));
    const int kind = w_shared ? AUX_TP_SHARED : AUX_TP;
    DeviceModule* m = nullptr;
    std::string err;
    uvu_status s = aux_module_for_current_device(p, kind, &m, &err);
    if (s != UVU_OK) return fail(s, err);
    long long N = batch;
    const int32_t* none = nullptr;
    void* args[] = {&N, &none, &none, &x, &y, &w, &out};
    return launch(m->aux[kind].k[0], m->aux[kind].occ[0], m->sm_count, batch, p->aux[kind].g[0], args, stream,
                  "uvu_tp_fwd launch");
}

extern "C" uvu_status uvu_tp_bwd(uvu_plan_t plan, int64_t batch, const void* x, const void* y, const void* w,
                                 int w_shared, const void* d_out, void* dx, void* dy, void* dw, void* workspace,
                                 size_t workspace_bytes, uvu_stream_t stream) {
    UVU_RANGE("uvu_tp_bwd");
    Plan* p = get(plan);
    UVU_TRY(tp_check(p, batch));
    UVU_TRY(opt(dx, "dx"));
    UVU_TRY(opt(dy, "dy"));
    UVU_TRY(opt(dw, "dw"));
    if (!dx && !dy && !dw) return ok();
    const size_t wsz = size_t(p->P) * p->U * p->elem();
    if (batch == 0) {  // a shared dw over an empty batch is zero
        if (dw && w_shared) {
            cudaError_t e = cudaMemsetAsync(dw, 0, wsz, stream);
            if (e != cudaSuccess) return cuda_fail(e, "dw memset");
        }
        return ok();
    }
    UVU_TRY(need(x, "x"));
    UVU_TRY(need(y, "y"));
    UVU_TRY(need(w, "w"));
    UVU_TRY(need(d_out, "d_out"));
    size_t ws_need = 0;
    UVU_TRY(uvu_tp_bwd_workspace(plan, batch, w_shared, &ws_need));
    const bool partials = w_shared && dw;
    if (partials) {
        if (!workspace || workspace_bytes < ws_need)
            return fail(UVU_ERR_INVALID_ARGUMENT, "a shared-weight dw needs a workspace of uvu_tp_bwd_workspace() bytes");
        UVU_TRY(need(workspace, "workspace"));
    }
    const int kind = w_shared ? AUX_TP_SHARED : AUX_TP;
    DeviceModule* m = nullptr;
    std::string err;
    uvu_status s = aux_module_for_current_device(p, kind, &m, &err);
    if (s != UVU_OK) return fail(s, err);
    const AuxLoaded& L = m->aux[kind];
    const AuxBuild& A = p->aux[kind];
    long long N = batch;
    const int32_t* none = nullptr;
    void* dw_arg = partials ? workspace : dw;
    void* dx_atomic = nullptr;
    void* args[] = {&N, &none, &none, &x, &y, &w, &d_out, &dy, &dw_arg, &dx_atomic, &dx};
    UVU_TRY(launch(L.k[1], L.occ[1], m->sm_count, batch, A.g[1], args, stream, "uvu_tp_edge launch", kTpMaxBlocks));
    if (partials) {
        const int64_t rows = grid_blocks(L.occ[1], m->sm_count, batch, A.g[1], kTpMaxBlocks);
        cudaError_t e = launch_column_sum(workspace, rows, int64_t(p->P) * p->U, dw, p->dtype == UVU_F64, stream);
        if (e != cudaSuccess) return cuda_fail(e, "dw column sum launch");
    }
    return ok();
}

// ------------------------------------------------------------------ fused radial weights
namespace uvu {
namespace {
// Fixes (or checks) the plan's hidden width for the fused radial forward.
uvu_status radial_prepare(Plan* p, int hidden) {
    if (hidden < 4 || hidden > 256 || hidden % 4)
        return fail(UVU_ERR_INVALID_ARGUMENT, "hidden must be a multiple of 4 in [4, 256]");
    std::lock_guard<std::mutex> g(p->mu);
    AuxBuild& A = p->aux[AUX_RADIAL];
    if (A.radial_h == 0) {
        A.radial_h = hidden;
        // UVU_RAD_NE / UVU_RAD_MINB (tuning switches): edges whose weights a thread forms
        // together; cap on resident blocks per SM the register budget is sized for
        if (const char* e = std::getenv("UVU_RAD_NE")) A.radial_ne = std::max(1, std::min(8, std::atoi(e)));
        if (const char* e = std::getenv("UVU_RAD_MINB")) A.minb[0] = std::max(1, std::min(8, std::atoi(e)));
    } else if (A.radial_h != hidden) {
        return fail(UVU_ERR_UNSUPPORTED, "this plan's fused radial forward was built for hidden width " +
                                             std::to_string(A.radial_h));
    }
    return UVU_OK;
}
}  // namespace
}  // namespace uvu

extern "C" uvu_status uvu_radial_hidden(uvu_plan_t plan, int64_t n_edges, const void* r, double r_cut, int p_env,
                                        int n_layers, const int* widths, const void* weights, void* h,
                                        uvu_stream_t stream) {
    UVU_RANGE("uvu_radial_hidden");
    Plan* p = get(plan);
    if (!p) return fail(UVU_ERR_INVALID_ARGUMENT, "plan is NULL");
    UVU_TRY(check_sizes(0, n_edges));
    if (!(r_cut > 0) || !std::isfinite(r_cut)) return fail(UVU_ERR_INVALID_ARGUMENT, "r_cut must be positive and finite");
    if (p_env < 1 || p_env > 16) return fail(UVU_ERR_INVALID_ARGUMENT, "p_env must be in [1, 16]");
    if (n_layers < 1 || n_layers > kRadialMaxLayers) return fail(UVU_ERR_INVALID_ARGUMENT, "n_layers must be in [1, 4]");
    if (!widths) return fail(UVU_ERR_INVALID_ARGUMENT, "widths is NULL");
    RadialNet net;
    net.n_layers = n_layers;
    if (widths[0] < 1 || widths[0] > 64) return fail(UVU_ERR_INVALID_ARGUMENT, "widths[0] (n_basis) must be in [1, 64]");
    for (int i = 0; i <= n_layers; ++i) {
        if (i > 0 && (widths[i] < 4 || widths[i] > 128 || widths[i] % 4))
            return fail(UVU_ERR_INVALID_ARGUMENT, "hidden widths must be multiples of 4 in [4, 128]");
        net.widths[i] = widths[i];
        net.max_width = std::max(net.max_width, widths[i]);
    }
    if (n_edges == 0) return ok();
    UVU_TRY(need(r, "r"));
    UVU_TRY(need(weights, "weights"));
    UVU_TRY(need(h, "h"));
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return cuda_fail(e, "device query");
    e = launch_radial_hidden(n_edges, r, r_cut, p_env, net, weights, h, p->dtype == UVU_F64, sms,
                             static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "radial network launch");
    return ok();
}

extern "C" uvu_status uvu_radial_module_source(uvu_plan_t plan, int hidden, const char** source, const char** log) {
    UVU_RANGE("uvu_radial_module_source");
    Plan* p = get(plan);
    if (!p) return fail(UVU_ERR_INVALID_ARGUMENT, "plan is NULL");
    UVU_TRY(radial_prepare(p, hidden));
    std::string err;
    uvu_status s = compile_aux(p, AUX_RADIAL, &err);
    if (s != UVU_OK) return fail(s, err);
    if (source) *source = p->aux[AUX_RADIAL].source.c_str();
    if (log) *log = p->aux[AUX_RADIAL].log.c_str();
    return ok();
}

extern "C" uvu_status uvu_conv_fwd_radial(uvu_plan_t plan, int64_t n_nodes, int64_t n_edges, const void* x,
                                          const void* Y, const void* h, int hidden, const void* w_last,
                                          const int32_t* recv_offsets, const int32_t* src, void* out,
                                          uvu_stream_t stream) {
    UVU_RANGE("uvu_conv_fwd_radial");
    Plan* p = get(plan);
    if (!p) return fail(UVU_ERR_INVALID_ARGUMENT, "plan is NULL");
    UVU_TRY(check_sizes(n_nodes, n_edges));
    UVU_TRY(radial_prepare(p, hidden));
    if (n_nodes == 0) return ok();
    UVU_TRY(need(out, "out"));
    UVU_TRY(need_idx(recv_offsets, "recv_offsets"));
    UVU_TRY(need(w_last, "w_last"));
    if (n_edges > 0) {
        UVU_TRY(need(x, "x"));
        UVU_TRY(need(Y, "Y"));
        UVU_TRY(need(h, "h"));
        UVU_TRY(need_idx(src, "src"));
    }
    DeviceModule* m = nullptr;
    std::string err;
    uvu_status s = aux_module_for_current_device(p, AUX_RADIAL, &m, &err);
    if (s != UVU_OK) return fail(s, err);
    const AuxLoaded& L = m->aux[AUX_RADIAL];
    const AuxBuild& A = p->aux[AUX_RADIAL];
    // grid: whole channel slices, each with the resident blocks' share (at most one block per
    // A.radial_rpb receivers)
    const int64_t nsl = int64_t(A.radial_nsl) * A.radial_gblk;
    const int64_t want = (n_nodes + A.radial_rpb - 1) / A.radial_rpb;
    const int64_t per_slice = std::max<int64_t>(1, std::min<int64_t>(want, int64_t(L.occ[0]) * m->sm_count / nsl));
    long long N = n_nodes;
    void* args[] = {&N, &recv_offsets, &src, &x, &Y, &h, &w_last, &out};
    cudaError_t e = cudaLaunchKernel(reinterpret_cast<const void*>(L.k[0]), dim3(unsigned(nsl * per_slice)),
                                     dim3(unsigned(A.g[0].threads)), args, A.g[0].smem, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "uvu_fwd_radial launch");
    return ok();
}

extern "C" uvu_status uvu_fma_rate_probe(uvu_dtype dtype, int blocks, int iters, void* out, double* fmas,
                                         uvu_stream_t stream) {
    UVU_RANGE("uvu_fma_rate_probe");
    if (dtype != UVU_F32 && dtype != UVU_F64) return fail(UVU_ERR_INVALID_ARGUMENT, "unknown dtype");
    if (blocks < 1 || blocks > (1 << 20) || iters < 1 || iters > (1 << 24))
        return fail(UVU_ERR_INVALID_ARGUMENT, "blocks must be in [1, 2^20] and iters in [1, 2^24]");
    UVU_TRY(need(out, "out"));
    cudaError_t e = launch_fma_probe(dtype == UVU_F64, blocks, iters, out, static_cast<cudaStream_t>(stream), fmas);
    if (e != cudaSuccess) return cuda_fail(e, "fma probe launch");
    return ok();
}

// ------------------------------------------------------- radial network: last layer, gradients
namespace uvu {
namespace {
uvu_status radial_net(int n_layers, const int* widths, RadialNet* net) {
    if (n_layers < 1 || n_layers > kRadialMaxLayers) return fail(UVU_ERR_INVALID_ARGUMENT, "n_layers must be in [1, 4]");
    if (!widths) return fail(UVU_ERR_INVALID_ARGUMENT, "widths is NULL");
    net->n_layers = n_layers;
    if (widths[0] < 1 || widths[0] > 64) return fail(UVU_ERR_INVALID_ARGUMENT, "widths[0] (n_basis) must be in [1, 64]");
    for (int i = 0; i <= n_layers; ++i) {
        if (i > 0 && (widths[i] < 4 || widths[i] > 128 || widths[i] % 4))
            return fail(UVU_ERR_INVALID_ARGUMENT, "hidden widths must be multiples of 4 in [4, 128]");
        net->widths[i] = widths[i];
        net->max_width = std::max(net->max_width, widths[i]);
    }
    return UVU_OK;
}
int sm_count_now() {
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    return sms;
}
}  // namespace
}  // namespace uvu

extern "C" uvu_status uvu_radial_weights_workspace(uvu_plan_t plan, int hidden, size_t* bytes) {
    Plan* p = get(plan);
    if (!p || !bytes) return fail(UVU_ERR_INVALID_ARGUMENT, "plan or bytes is NULL");
    if (hidden < 4 || hidden > 256 || hidden % 4) return fail(UVU_ERR_INVALID_ARGUMENT, "hidden must be a multiple of 4 in [4, 256]");
    *bytes = dense_product_workspace(hidden, p->P * p->U, p->dtype == UVU_F64);
    return ok();
}

extern "C" uvu_status uvu_radial_weights(uvu_plan_t plan, int64_t n_edges, const void* h, int hidden,
                                         const void* w_last, void* w, void* workspace, size_t workspace_bytes,
                                         uvu_stream_t stream) {
    UVU_RANGE("uvu_radial_weights");
    Plan* p = get(plan);
    if (!p) return fail(UVU_ERR_INVALID_ARGUMENT, "plan is NULL");
    UVU_TRY(check_sizes(0, n_edges));
    if (hidden < 4 || hidden > 256 || hidden % 4) return fail(UVU_ERR_INVALID_ARGUMENT, "hidden must be a multiple of 4 in [4, 256]");
    if (n_edges == 0) return ok();
    UVU_TRY(need(h, "h"));
    UVU_TRY(need(w_last, "w_last"));
    UVU_TRY(need(w, "w"));
    const int PU = p->P * p->U;
    if (!workspace || workspace_bytes < dense_product_workspace(hidden, PU, p->dtype == UVU_F64) ||
        (reinterpret_cast<uintptr_t>(workspace) & 15u))
        return fail(UVU_ERR_INVALID_ARGUMENT, "workspace is NULL, misaligned or smaller than uvu_radial_weights_workspace()");
    cudaError_t e = launch_dense_product(p->dtype == UVU_F64, n_edges, hidden, PU, h, w_last, false, w, workspace,
                                         workspace_bytes, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "radial last layer launch");
    return ok();
}

extern "C" uvu_status uvu_radial_weights_bwd_workspace(uvu_plan_t plan, int64_t n_edges, int hidden, size_t* bytes) {
    Plan* p = get(plan);
    if (!p || !bytes) return fail(UVU_ERR_INVALID_ARGUMENT, "plan or bytes is NULL");
    UVU_TRY(check_sizes(0, n_edges));
    if (hidden < 4 || hidden > 256 || hidden % 4) return fail(UVU_ERR_INVALID_ARGUMENT, "hidden must be a multiple of 4 in [4, 256]");
    const int PU = p->P * p->U;
    // dh = dw W_last^T is the product with K = P U and N = hidden (the forward's transpose)
    const size_t a = (dense_product_workspace(PU, hidden, p->dtype == UVU_F64) + 255) / 256 * 256;
    *bytes = a + dense_reduction_workspace(n_edges, hidden, PU);
    return ok();
}

extern "C" uvu_status uvu_radial_weights_bwd(uvu_plan_t plan, int64_t n_edges, const void* h, int hidden,
                                             const void* w_last, const void* dw, void* dh, void* dw_last,
                                             void* workspace, size_t workspace_bytes, uvu_stream_t stream) {
    UVU_RANGE("uvu_radial_weights_bwd");
    Plan* p = get(plan);
    if (!p) return fail(UVU_ERR_INVALID_ARGUMENT, "plan is NULL");
    UVU_TRY(check_sizes(0, n_edges));
    if (hidden < 4 || hidden > 256 || hidden % 4) return fail(UVU_ERR_INVALID_ARGUMENT, "hidden must be a multiple of 4 in [4, 256]");
    UVU_TRY(opt(dh, "dh"));
    UVU_TRY(opt(dw_last, "dw_last"));
    const bool f64 = p->dtype == UVU_F64;
    const int PU = p->P * p->U;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (n_edges == 0) {
        if (dw_last) {
            cudaError_t e = cudaMemsetAsync(dw_last, 0, size_t(hidden) * PU * p->elem(), st);
            if (e != cudaSuccess) return cuda_fail(e, "memset");
        }
        return ok();
    }
    if (!dh && !dw_last) return ok();
    UVU_TRY(need(dw, "dw"));
    UVU_TRY(need(w_last, "w_last"));
    if (dw_last) UVU_TRY(need(h, "h"));
    size_t need_bytes = 0;
    UVU_TRY(uvu_radial_weights_bwd_workspace(plan, n_edges, hidden, &need_bytes));
    if (!workspace || workspace_bytes < need_bytes || (reinterpret_cast<uintptr_t>(workspace) & 15u))
        return fail(UVU_ERR_INVALID_ARGUMENT, "workspace is NULL, misaligned or smaller than uvu_radial_weights_bwd_workspace()");
    char* ws = static_cast<char*>(workspace);
    const size_t a = (dense_product_workspace(PU, hidden, f64) + 255) / 256 * 256;
    cudaError_t e = cudaSuccess;
    if (dh) e = launch_dense_product(f64, n_edges, PU, hidden, dw, w_last, true, dh, ws, a, st);
    if (e == cudaSuccess && dw_last) e = launch_dense_reduction(f64, n_edges, hidden, PU, h, dw, dw_last, ws + a, st);
    if (e != cudaSuccess) return cuda_fail(e, "radial last-layer gradient launch");
    return ok();
}

extern "C" uvu_status uvu_radial_hidden_bwd_workspace(uvu_plan_t plan, int64_t n_edges, int n_layers, const int* widths,
                                                      size_t* bytes) {
    Plan* p = get(plan);
    if (!p || !bytes) return fail(UVU_ERR_INVALID_ARGUMENT, "plan or bytes is NULL");
    UVU_TRY(check_sizes(0, n_edges));
    RadialNet net;
    UVU_TRY(radial_net(n_layers, widths, &net));
    if (!radial_hidden_bwd_supported(net, p->dtype == UVU_F64))
        return fail(UVU_ERR_UNSUPPORTED, "the radial network is too wide for the reverse pass's shared memory");
    *bytes = radial_hidden_bwd_workspace(n_edges, net, p->dtype == UVU_F64, std::max(1, sm_count_now()));
    return ok();
}

extern "C" uvu_status uvu_radial_hidden_bwd(uvu_plan_t plan, int64_t n_edges, const void* r, double r_cut, int p_env,
                                            int n_layers, const int* widths, const void* weights, const void* dh,
                                            void* dr, void* dweights, void* workspace, size_t workspace_bytes,
                                            uvu_stream_t stream) {
    UVU_RANGE("uvu_radial_hidden_bwd");
    Plan* p = get(plan);
    if (!p) return fail(UVU_ERR_INVALID_ARGUMENT, "plan is NULL");
    UVU_TRY(check_sizes(0, n_edges));
    if (!(r_cut > 0) || !std::isfinite(r_cut)) return fail(UVU_ERR_INVALID_ARGUMENT, "r_cut must be positive and finite");
    if (p_env < 1 || p_env > 16) return fail(UVU_ERR_INVALID_ARGUMENT, "p_env must be in [1, 16]");
    RadialNet net;
    UVU_TRY(radial_net(n_layers, widths, &net));
    const bool f64 = p->dtype == UVU_F64;
    if (!radial_hidden_bwd_supported(net, f64))
        return fail(UVU_ERR_UNSUPPORTED, "the radial network is too wide for the reverse pass's shared memory");
    UVU_TRY(need(weights, "weights"));
    UVU_TRY(need(dweights, "dweights"));
    const int sms = std::max(1, sm_count_now());
    if (n_edges > 0) {
        UVU_TRY(need(r, "r"));
        UVU_TRY(need(dh, "dh"));
        UVU_TRY(need(dr, "dr"));
        const size_t nb = radial_hidden_bwd_workspace(n_edges, net, f64, sms);
        if (!workspace || workspace_bytes < nb || (reinterpret_cast<uintptr_t>(workspace) & 15u))
            return fail(UVU_ERR_INVALID_ARGUMENT, "workspace is NULL, misaligned or smaller than uvu_radial_hidden_bwd_workspace()");
    }
    cudaError_t e = launch_radial_hidden_bwd(n_edges, r, r_cut, p_env, net, weights, dh, dr, dweights, workspace, f64, sms,
                                             static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "radial network reverse pass launch");
    return ok();
}
