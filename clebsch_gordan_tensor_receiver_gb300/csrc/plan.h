// Internal declarations of the UVU convolution library (not part of the C ABI).
#pragma once

#include <cuda_runtime.h>

#include <cstdint>
#include <map>
#include <memory>
#include <mutex>
#include <string>
#include <vector>

#include "uvu.h"

namespace uvu {

struct Irrep {
    int mul;
    int l;
    int parity;  // +1 even, -1 odd
};

// One non-zero of a real CG tensor.
struct Nz {
    int m1, m2, m3;  // 0 .. 2l
    double c;
};

struct PathInfo {
    int l1, l2, l3, parity;
    int ix, iy;              // index of the x irrep / SH irrep
    int xoff, yoff, ooff;    // block offsets inside a channel's x row, an edge's Y row, a channel's out row
    std::vector<double> cg;  // dense (2l1+1)(2l2+1)(2l3+1), row-major (m1, m2, m3)
    std::vector<Nz> nz;      // non-zeros of cg
};

// Launch geometry of one generated kernel.
struct KernelGeom {
    int threads = 0;           // threads per block
    int owners_per_block = 0;  // receivers (or senders) per block (non-persistent kernels)
    size_t smem = 0;           // dynamic shared memory bytes
    bool persistent = false;   // grid = resident blocks, owners assigned round-robin
    int tiles = 1;             // work items per owner (channel tiles) for persistent kernels
};

// Auxiliary modules of a plan, emitted and compiled on their first use, each with a
// receiver-ordered "forward" kernel and an "edge" kernel: the double backward, and the batched
// (non-convolution) tensor product with per-sample or batch-shared weights.
// The fused-radial-weight forward (AUX_RADIAL) has one kernel only.
enum AuxKind { AUX_HVP = 0, AUX_TP = 1, AUX_TP_SHARED = 2, AUX_RADIAL = 3, AUX_COUNT = 4 };
extern const char* const kAuxKernelNames[AUX_COUNT][2];

struct AuxBuild {  // host side, per plan
    std::string source, log;
    std::vector<char> cubin;
    KernelGeom g[2];
    int minb[2] = {4, 4};      // register-budget caps (blocks per SM), lowered on spills
    int minb_eff[2] = {1, 1};  // value used by the last emission
    // fused radial forward: hidden width the module is built for (0 = not yet), edges whose
    // weights a thread forms together (lowered on spills), layout chosen at emission
    int radial_h = 0;
    int radial_ne = 3;
    bool radial_wsm = false;   // last-layer slice staged in shared memory
    int radial_nsl = 1;        // channel slices of 32
    int radial_rpb = 1;        // receivers per block per round
    int radial_gblk = 1;       // blocks per channel slice and receiver set (path runs, split form)
};

// Radial network of the fused-weight forward (radial.cu): widths[0] = n_basis, then the hidden
// layers' widths (multiples of 4), each layer followed by SiLU.
constexpr int kRadialMaxLayers = 4;
struct RadialNet {
    int n_layers = 0;
    int max_width = 0;
    int widths[kRadialMaxLayers + 1] = {};
};

struct AuxLoaded {  // per device
    cudaLibrary_t lib = nullptr;
    cudaKernel_t k[2] = {nullptr, nullptr};
    int occ[2] = {1, 1};
    unsigned* status_word = nullptr;  // the module's own uvu_status_word (pipelined kernels only)
};

struct DeviceModule {
    cudaLibrary_t lib = nullptr;
    cudaKernel_t fwd = nullptr, bwd_edge = nullptr, bwd_dx = nullptr, bwd_dx_reduce = nullptr, fwd_sender = nullptr;
    int sm_count = 0;
    int occ_fwd = 1, occ_edge = 1, occ_dx = 1;  // resident blocks per SM
    unsigned* status_word = nullptr;            // device address of uvu_status_word
    AuxLoaded aux[AUX_COUNT];
};

struct Plan {
    std::string irreps_x, irreps_sh;
    int lmax_out = 0;
    uvu_dtype dtype = UVU_F32;
    int U = 0, Dx = 0, Dy = 0, Do = 0, P = 0;
    int U_pad = 0;  // channel slots per owner in the generated kernels
    std::vector<Irrep> xs, ys;
    std::vector<PathInfo> paths;
    std::vector<std::vector<int>> groups;  // path ids per register group
    KernelGeom g_fwd, g_edge, g_dx, g_fwd_sender;
    int reduce_per_sender = 0;  // threads of uvu_bwd_dx_reduce per sender (set by the generator)
    int edge_chunk = 0;  // edges per dY reduction chunk in the edge kernel
    bool pipelined_recv = false, pipelined_dx = false;
    bool staged_ok = false;   // the edge kernel can write per-edge dx partials (staged dx)
    bool rebalanced = false;  // register groups re-split for the pipelined kernels
    // Upper bound on resident blocks per SM that the register budget is sized for, per kernel
    // (fwd, edge, dx); lowered one block at a time for a kernel whose budget makes ptxas spill.
    int minb[3] = {4, 4, 4};
    int minb_eff[3] = {1, 1, 1};  // value used by the last emission
    std::string source, log;
    std::vector<char> cubin;
    AuxBuild aux[AUX_COUNT];
    std::mutex mu;
    std::map<int, DeviceModule> modules;  // per device ordinal
    size_t elem() const { return dtype == UVU_F64 ? 8 : 4; }
};

// cg.cpp
std::vector<double> real_cg_dense(int l1, int l2, int l3);

// irreps.cpp
bool parse_irreps(const char* s, std::vector<Irrep>* out, std::string* err);
uvu_status build_paths(Plan* plan, std::string* err);

// codegen.cpp
std::string emit_source(Plan* plan);
std::string emit_aux_source(Plan* plan, int kind);
void balance_groups(Plan* plan, int ng);

// jit.cpp
uvu_status compile_plan(Plan* plan, std::string* err);
size_t spill_bytes(const std::string& log, const char* kernel);
uvu_status module_for_current_device(Plan* plan, DeviceModule** out, std::string* err);
uvu_status compile_aux(Plan* plan, int kind, std::string* err);  // host only
uvu_status aux_module_for_current_device(Plan* plan, int kind, DeviceModule** out, std::string* err);

// status.cpp
uvu_status fail(uvu_status s, const std::string& msg);
uvu_status ok();
uvu_status cuda_fail(cudaError_t e, const char* what);
const char* g_last_message_cstr();

}  // namespace uvu

namespace uvu {
// graph.cu
size_t transpose_workspace_bytes(int64_t N, int64_t E);
cudaError_t launch_fma_probe(bool f64, int blocks, int iters, void* out, cudaStream_t st, double* fmas);
cudaError_t launch_csr_offsets(int64_t N, int64_t E, const int32_t* recv, int32_t* off, cudaStream_t st);
cudaError_t launch_csr_transpose(int64_t N, int64_t E, const int32_t* roff, const int32_t* src,
                                 int32_t* soff, int32_t* eids, int32_t* srecv, void* ws, cudaStream_t st);
cudaError_t launch_graph_validate(int64_t N, int64_t E, const int32_t* off, const int32_t* src,
                                  unsigned long long* bad, cudaStream_t st);
// tp.cu
cudaError_t launch_column_sum(const void* part, int64_t rows, int64_t cols, void* out, bool f64, cudaStream_t st);
// radial.cu
size_t radial_hidden_smem(const RadialNet& net, bool f64);
cudaError_t launch_radial_hidden(int64_t E, const void* r, double r_cut, int p_env, const RadialNet& net, const void* W,
                                 void* h, bool f64, int sm_count, cudaStream_t st);
size_t radial_hidden_bwd_workspace(int64_t E, const RadialNet& net, bool f64, int sm_count);
bool radial_hidden_bwd_supported(const RadialNet& net, bool f64);
cudaError_t launch_radial_hidden_bwd(int64_t E, const void* r, double r_cut, int p_env, const RadialNet& net,
                                     const void* W, const void* dh, void* dr, void* dW, void* ws, bool f64,
                                     int sm_count, cudaStream_t st);
// tcgemm.cu: fp32 products on the tensor cores (3xTF32, see tcgemm.cu)
constexpr int kTcMaxSeg = 128;
struct TcJobs;
bool tc_gemm_supported(const TcJobs& J);
size_t tc_gemm_workspace(const TcJobs& J);
cudaError_t launch_tc_gemm(TcJobs& J, cudaStream_t st);
cudaError_t tc_status(unsigned* word, bool reset);
// mix.cu
cudaError_t launch_dense_product(bool f64, int64_t rows, int K, int Nc, const void* A, const void* B, bool b_kcont,
                                 void* C, void* ws, size_t ws_bytes, cudaStream_t st);
size_t dense_product_workspace(int K, int Nc, bool f64);
size_t dense_reduction_workspace(int64_t rows, int Mr, int Nc);
cudaError_t launch_dense_reduction(bool f64, int64_t rows, int Mr, int Nc, const void* A, const void* G, void* C, void* ws,
                                   cudaStream_t st);
int mix_max_paths();
size_t mix_workspace_bytes(const Plan& p, int64_t N, int W, bool bwd);
cudaError_t launch_mix_fwd(const Plan& p, int64_t N, int W, const void* in, const void* M, void* out, void* ws,
                           cudaStream_t st);
cudaError_t launch_mix_bwd(const Plan& p, int64_t N, int W, const void* in, const void* M, const void* g, void* d_in,
                           void* dM, void* ws, cudaStream_t st);
}  // namespace uvu
