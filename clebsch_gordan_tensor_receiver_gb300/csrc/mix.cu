// Per-path channel mixing that reduces a factorised UVW convolution to the UVU one
// ("Receiver-streaming convolutions for channel-wise UVU tensor products", replies: UVW cases
// that can be reduced to UVU).  With per-edge weights W_e[p,u,w] = w[e,p,u] M[p,u,w], the
// mixing M is the same on every edge and commutes with the sum over a receiver's edges:
//     out[r,w,ooff(p)+m3] = sum_u M[p,u,w] in[r,u,ooff(p)+m3]        in = the UVU output.
//
// In the convolution's layout [N][U][D_out] a path's components are a few values inside each
// 55-106-wide row, so a direct product gathers D_out-strided values.  The kernels here first copy
// the operand to a component-major layout [D_out][N][U] (one pass, coalesced both ways through a
// shared-memory tile); a path p is then the contiguous matrix of rows (ooff(p)+m, r), and the
// mixing is one dense product per path, A_p [d3*N x U] times M[p] [U x W], written component-major
// and copied back.  The input gradient is the same product with M[p] transposed, and
// dM[p] = A_p^T G_p is a product over the rows, split into fixed row chunks summed in fp64 (fp32
// within 16 rows) and added in chunk order (deterministic).  In fp32 plans the two products with
// K = U or W run on the tensor cores (tcgemm.cu: 3xTF32, fp32 accuracy), reading M directly as the
// k-contiguous operand for the input gradient; dM, a sum over d3 N rows, stays on the compensated
// CUDA-core kernel, whose fp32 steps of 16 rows keep the elementwise tolerance that the tensor
// memory's accumulation did not.
#include <algorithm>
#include <cstdint>

#include "plan.h"
#include "tcgemm.h"

namespace uvu {
namespace {

constexpr int kMaxPaths = 128;

// ----------------------------------------------------------------------------- layout copies

// out[b][n][a] = in[n][a][b]  (to component-major: a = channel, b = component), or the inverse
// out[n][a][b] = in[b][n][a] when INV.  Block = (node n, TA consecutive channels a0..): the
// node's [TA][B] slab (contiguous in the node-major layout) passes through shared memory with
// an odd row pitch, so that the component-major side's accesses (lane = channel, stride pitch)
// hit distinct banks.  The node-major side is one contiguous run: copied linearly (16-byte
// vectors when aligned) when B is odd (pitch == B), else row by row (lane = component).
template <typename T, bool INV>
__global__ void __launch_bounds__(256) relayout(int64_t N, int A, int B, int TA, const T* __restrict__ in,
                                                T* __restrict__ out) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    T* s = reinterpret_cast<T*>(smem_raw);
    const int pitch = B | 1;
    const int64_t n = blockIdx.x;
    const int a0 = blockIdx.y * TA;
    const int na = min(TA, A - a0);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int64_t nm = (n * A + a0) * B;  // node-major start of the slab
    const int cnt = na * B;
    constexpr int V = 16 / int(sizeof(T));
    const bool vec = pitch == B && ((reinterpret_cast<uintptr_t>(INV ? static_cast<const void*>(out + nm)
                                                                     : static_cast<const void*>(in + nm)) & 15) == 0);
    if (!INV) {
        if (pitch == B) {
            if (vec) {
                const int nv = cnt / V;
                for (int i = tid; i < nv; i += 256)
                    reinterpret_cast<uint4*>(s)[i] = __ldg(reinterpret_cast<const uint4*>(in + nm) + i);
                for (int e = nv * V + tid; e < cnt; e += 256) s[e] = in[nm + e];
            } else {
                for (int e = tid; e < cnt; e += 256) s[e] = in[nm + e];
            }
        } else {
            for (int a = warp; a < na; a += 8)
                for (int b = lane; b < B; b += 32) s[a * pitch + b] = in[nm + int64_t(a) * B + b];
        }
        __syncthreads();
        for (int b = warp; b < B; b += 8) {
            T* o = out + (int64_t(b) * N + n) * A + a0;
            for (int a = lane; a < na; a += 32) o[a] = s[a * pitch + b];
        }
    } else {
        for (int b = warp; b < B; b += 8) {
            const T* q = in + (int64_t(b) * N + n) * A + a0;
            for (int a = lane; a < na; a += 32) s[a * pitch + b] = q[a];
        }
        __syncthreads();
        if (pitch == B) {
            if (vec) {
                const int nv = cnt / V;
                for (int i = tid; i < nv; i += 256) reinterpret_cast<uint4*>(out + nm)[i] = reinterpret_cast<const uint4*>(s)[i];
                for (int e = nv * V + tid; e < cnt; e += 256) out[nm + e] = s[e];
            } else {
                for (int e = tid; e < cnt; e += 256) out[nm + e] = s[e];
            }
        } else {
            for (int a = warp; a < na; a += 8)
                for (int b = lane; b < B; b += 32) out[nm + int64_t(a) * B + b] = s[a * pitch + b];
        }
    }
}

// Mt[p][w][u] = M[p][u][w]
template <typename T>
__global__ void transpose_M(int P, int U, int W, const T* __restrict__ M, T* __restrict__ Mt) {
    const int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
    if (i >= int64_t(P) * U * W) return;
    const int64_t p = i / (int64_t(U) * W), rem = i % (int64_t(U) * W);
    const int u = int(rem / W), w = int(rem % W);
    Mt[(p * W + w) * U + u] = M[i];
}

// ------------------------------------------------------------------- per-path dense products

struct SegTab {
    int n;
    int64_t row0[kMaxPaths];   // first row of the path in the component-major operand (ooff * N)
    int64_t rows[kMaxPaths];   // d3 * N
    int tile0[kMaxPaths + 1];  // prefix of row tiles
};

constexpr int kTM = 128, kTN = 128, kTK = 8;

// C[row][c] = sum_k A[row][k] Bp[k][c] for the rows of each path (Bp = Bmat + p K Nc), A and C
// row-major, row = component-major row index.  256 threads with 8 x 8 outputs each (rows
// tr*4 + {0..3} and 64 + tr*4 + {0..3}, columns likewise: conflict-free shared-memory reads);
// k advances in chunks of 8, the next chunk loaded into registers during the current one.
template <typename T>
__global__ void __launch_bounds__(256) seg_gemm(int K, int Nc, SegTab tab, const T* __restrict__ A,
                                                const T* __restrict__ Bmat, T* __restrict__ C) {
    __shared__ __align__(16) T sA[2][kTK][kTM];
    __shared__ __align__(16) T sB[2][kTK][kTN];
    int pi = 0;
    while (pi + 1 < tab.n && int(blockIdx.x) >= tab.tile0[pi + 1]) ++pi;
    const int64_t rbeg = tab.row0[pi] + int64_t(int(blockIdx.x) - tab.tile0[pi]) * kTM;
    const int64_t rend = tab.row0[pi] + tab.rows[pi];
    const int c0 = blockIdx.y * kTN;
    const T* Bp = Bmat + size_t(pi) * K * Nc;
    const int tid = threadIdx.x, tr = tid / 16, tc = tid % 16;
    // loader roles: A row (tid / 2) with k half (tid % 2) * 4; B k row (tid / 32) with columns (tid % 32) * 4
    const int la_r = tid / 2, la_k = (tid % 2) * 4;
    const int lb_k = tid / 32, lb_c = (tid % 32) * 4;
    T ra[4], rb[4];
    auto load = [&](int k0) {
        const int64_t row = rbeg + la_r;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int k = k0 + la_k + i;
            ra[i] = (row < rend && k < K) ? A[row * K + k] : T(0);
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int k = k0 + lb_k, c = c0 + lb_c + i;
            rb[i] = (k < K && c < Nc) ? Bp[size_t(k) * Nc + c] : T(0);
        }
    };
    auto store = [&](int buf) {
#pragma unroll
        for (int i = 0; i < 4; ++i) sA[buf][la_k + i][la_r] = ra[i];
#pragma unroll
        for (int i = 0; i < 4; ++i) sB[buf][lb_k][lb_c + i] = rb[i];
    };
    T acc[8][8];
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[i][j] = 0;
    load(0);
    store(0);
    __syncthreads();
    int buf = 0;
    for (int k0 = 0; k0 < K; k0 += kTK) {
        const bool more = k0 + kTK < K;
        if (more) load(k0 + kTK);
#pragma unroll
        for (int k = 0; k < kTK; ++k) {
            T a[8], b[8];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                a[i] = sA[buf][k][tr * 4 + i];
                a[4 + i] = sA[buf][k][64 + tr * 4 + i];
                b[i] = sB[buf][k][tc * 4 + i];
                b[4 + i] = sB[buf][k][64 + tc * 4 + i];
            }
#pragma unroll
            for (int i = 0; i < 8; ++i)
#pragma unroll
                for (int j = 0; j < 8; ++j) acc[i][j] = fma(a[i], b[j], acc[i][j]);
        }
        if (more) {
            store(buf ^ 1);
            __syncthreads();
            buf ^= 1;
        }
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int64_t row = rbeg + (i < 4 ? tr * 4 + i : 64 + tr * 4 + i - 4);
        if (row >= rend) continue;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const int c = c0 + (j < 4 ? tc * 4 + j : 64 + tc * 4 + j - 4);
            if (c < Nc) C[row * Nc + c] = acc[i][j];
        }
    }
}

// dM partials: part[ch][p][u][w] = sum over the rows of chunk ch of path p of A[row][u] G[row][w].
// Block tile 64 u x 64 w, 256 threads with 4 x 4 outputs each.  Rows go in steps of 16 summed in
// the plan's type; the step sums are added with Kahan compensation, and into fp64 registers every
// 16 steps.  A plain fp32 sum of a chunk lost digits where the terms cancel, and an fp64 add after
// every step cost more than the products (FP64 runs at a small fraction of FP32 here).  Stored as
// fp64; chunks past a path's rows store zero.
constexpr int kRowChunk = 1024, kDT = 64, kDR = 16;
template <typename T>
__global__ void __launch_bounds__(256) seg_dM(int U, int W, SegTab tab, const T* __restrict__ A, const T* __restrict__ G,
                                              double* __restrict__ part) {
    __shared__ __align__(16) T sA[kDR][kDT];
    __shared__ __align__(16) T sG[kDR][kDT];
    const int ntw = (W + kDT - 1) / kDT;
    const int u0 = (blockIdx.x / ntw) * kDT, w0 = (blockIdx.x % ntw) * kDT;
    const int pi = blockIdx.y, ch = blockIdx.z;
    const int64_t rbeg = tab.row0[pi] + int64_t(ch) * kRowChunk;
    const int64_t rend = min(tab.row0[pi] + tab.rows[pi], rbeg + kRowChunk);
    const int tid = threadIdx.x, tr = tid / 16, tc = tid % 16;
    double acc[4][4] = {};
    T ksum[4][4] = {}, kcomp[4][4] = {};
    int nstep = 0;
    for (int64_t r0 = rbeg; r0 < rend; r0 += kDR) {
        // 16 rows x 64 columns of each operand: 4 consecutive columns per thread
        {
            const int lr = tid / 16, lc = (tid % 16) * 4;
            const int64_t row = r0 + lr;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int u = u0 + lc + i, w = w0 + lc + i;
                sA[lr][lc + i] = (row < rend && u < U) ? A[row * U + u] : T(0);
                sG[lr][lc + i] = (row < rend && w < W) ? G[row * W + w] : T(0);
            }
        }
        __syncthreads();
        T part_acc[4][4] = {};
#pragma unroll
        for (int k = 0; k < kDR; ++k) {
            T a[4], b[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                a[i] = sA[k][tr + 16 * i];
                b[i] = sG[k][tc + 16 * i];
            }
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) part_acc[i][j] = fma(a[i], b[j], part_acc[i][j]);
        }
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const T y = part_acc[i][j] - kcomp[i][j];
                const T t = ksum[i][j] + y;
                kcomp[i][j] = (t - ksum[i][j]) - y;
                ksum[i][j] = t;
            }
        if (++nstep == 16 || r0 + kDR >= rend) {
            nstep = 0;
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    acc[i][j] += double(ksum[i][j]) - double(kcomp[i][j]);
                    ksum[i][j] = T(0);
                    kcomp[i][j] = T(0);
                }
        }
        __syncthreads();
    }
    double* pr = part + (size_t(ch) * tab.n + pi) * size_t(U) * W;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int u = u0 + tr + 16 * i;
        if (u >= U) continue;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int w = w0 + tc + 16 * j;
            if (w < W) pr[size_t(u) * W + w] = acc[i][j];
        }
    }
}

// fp32 form of seg_dM for 4-aligned widths.  Block tile 64 u x 128 w; warp tu (of 8) owns
// u = u0 + 8 tu + i (i < 8), lane tw owns w = w0 + 4 tw + j (j < 4): per row the warp's lanes
// share two 16-byte reads of A (broadcast) and read G as one contiguous 512-byte row (no bank
// conflicts), 32 FMAs (16 paired) per three shared-memory reads.  Rows in steps of 32 through a four-stage
// cp.async ring.  Each step's fp32 sums are added with Kahan compensation (which carries the
// chunk to fp32-round-off accuracy without fp64 registers), and the chunk's sum
// (sum - lost part) is stored as fp64, like seg_dM.
constexpr int kFU = 64, kFW = 128, kFR = 32, kFS = 4;
constexpr int kFStage = kFR * (kFU + kFW);  // floats per stage
constexpr int kFSmem = kFS * kFStage * 4;
__device__ __forceinline__ unsigned long long f2pack(float a, float b) {
    unsigned long long r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
    return r;
}
__device__ __forceinline__ void f2unpack(unsigned long long v, float& a, float& b) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(v));
}
// (a0, a1) * (b0, b1) + (c0, c1), each half rounded as a scalar fma
__device__ __forceinline__ unsigned long long f2fma(unsigned long long a, unsigned long long b, unsigned long long c) {
    unsigned long long d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
__device__ __forceinline__ void cp_async16(void* dst, const void* src, bool valid) {
    const unsigned d = unsigned(__cvta_generic_to_shared(dst));
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(d), "l"(src), "r"(valid ? 16 : 0) : "memory");
}
// Two resident blocks per SM (a 128-register budget; ptxas spills 80 bytes of the 160 it would
// use at one block): measured faster than one block at 160 registers (radial dW_last 1.61 ->
// 1.41 ms, mixing dM 0.390 -> 0.365 ms on MACE-medium), the extra warps hiding the ring's waits.
__global__ void __launch_bounds__(256, 2) seg_dM_f32(int U, int W, SegTab tab, const float* __restrict__ A,
                                                     const float* __restrict__ G, double* __restrict__ part) {
    extern __shared__ __align__(16) float fsm[];  // kFS stages of [kFR][kFU] A rows then [kFR][kFW] G rows
    const int ntw = (W + kFW - 1) / kFW;
    const int u0 = (blockIdx.x / ntw) * kFU, w0 = (blockIdx.x % ntw) * kFW;
    const int pi = blockIdx.y, ch = blockIdx.z;
    const int64_t rbeg = tab.row0[pi] + int64_t(ch) * kRowChunk;
    const int64_t rend = min(tab.row0[pi] + tab.rows[pi], rbeg + kRowChunk);
    const int tid = threadIdx.x, tw = tid & 31, tu = tid >> 5;
    float ks[8][4], kc[8][4];
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) ks[i][j] = kc[i][j] = 0.f;
    const int nsteps = rbeg < rend ? int((rend - rbeg + kFR - 1) / kFR) : 0;
    // step st: 32 rows of A (16 vectors per row) and of G (32 vectors per row) into its stage;
    // rows past the chunk and columns past the width read as zeros.  Every thread commits one
    // group per call, empty past the last step, so that the group count stays uniform.
    auto load = [&](int st) {
        if (st < nsteps) {
            float* sa = fsm + (st % kFS) * kFStage;
            float* sg = sa + kFR * kFU;
            const int64_t r0 = rbeg + int64_t(st) * kFR;
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                const int f = tid + 256 * i, row = f >> 4, c4 = f & 15;
                const int64_t gr = r0 + row;
                const int u = u0 + 4 * c4;
                const bool ok = gr < rend && u < U;
                cp_async16(sa + row * kFU + 4 * c4, ok ? A + gr * U + u : A, ok);
            }
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int f = tid + 256 * i, row = f >> 5, c4 = f & 31;
                const int64_t gr = r0 + row;
                const int w = w0 + 4 * c4;
                const bool ok = gr < rend && w < W;
                cp_async16(sg + row * kFW + 4 * c4, ok ? G + gr * W + w : G, ok);
            }
        }
        asm volatile("cp.async.commit_group;" ::: "memory");
    };
#pragma unroll
    for (int st = 0; st < kFS - 1; ++st) load(st);
    for (int st = 0; st < nsteps; ++st) {
        asm volatile("cp.async.wait_group %0;" ::"n"(kFS - 2) : "memory");
        __syncthreads();     // step st has landed for every thread; step st - 1's stage is free
        load(st + kFS - 1);  // into the stage step st - 1 used
        const float* sa = fsm + (st % kFS) * kFStage;
        const float* sg = sa + kFR * kFU;
        // step sums of (u 2i, u 2i + 1) pairs with paired FMAs (the same per-half rounding as
        // scalar fmaf): half the FMA instructions
        unsigned long long acc2[4][4];
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j) acc2[i][j] = 0ull;
#pragma unroll 8
        for (int k = 0; k < kFR; ++k) {
            const float4 a0 = *reinterpret_cast<const float4*>(sa + k * kFU + 8 * tu);
            const float4 a1 = *reinterpret_cast<const float4*>(sa + k * kFU + 8 * tu + 4);
            const float4 b = *reinterpret_cast<const float4*>(sg + k * kFW + 4 * tw);
            const unsigned long long ap[4] = {f2pack(a0.x, a0.y), f2pack(a0.z, a0.w), f2pack(a1.x, a1.y),
                                              f2pack(a1.z, a1.w)};
            const unsigned long long bp[4] = {f2pack(b.x, b.x), f2pack(b.y, b.y), f2pack(b.z, b.z), f2pack(b.w, b.w)};
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) acc2[i][j] = f2fma(ap[i], bp[j], acc2[i][j]);
        }
        float acc[8][4];
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j) f2unpack(acc2[i][j], acc[2 * i][j], acc[2 * i + 1][j]);
#pragma unroll
        for (int i = 0; i < 8; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const float y = acc[i][j] - kc[i][j];
                const float t = ks[i][j] + y;
                kc[i][j] = (t - ks[i][j]) - y;
                ks[i][j] = t;
            }
    }
    asm volatile("cp.async.wait_group 0;" ::: "memory");
    double* pr = part + (size_t(ch) * tab.n + pi) * size_t(U) * W;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int u = u0 + 8 * tu + i;
        if (u >= U) continue;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int w = w0 + 4 * tw + j;
            if (w < W) pr[size_t(u) * W + w] = double(ks[i][j]) - double(kc[i][j]);
        }
    }
}

// Launch of the fp32 form; its dynamic shared memory (above the 48 KB default) is set once per
// process.
cudaError_t launch_dM_f32(int U, int W, const SegTab& tab, unsigned nseg, unsigned nch, const float* A, const float* G,
                          double* part, cudaStream_t st) {
    static const cudaError_t e0 = cudaFuncSetAttribute(seg_dM_f32, cudaFuncAttributeMaxDynamicSharedMemorySize, kFSmem);
    if (e0 != cudaSuccess) return e0;
    const unsigned t = unsigned(((U + kFU - 1) / kFU) * ((W + kFW - 1) / kFW));
    seg_dM_f32<<<dim3(t, nseg, nch), 256, kFSmem, st>>>(U, W, tab, A, G, part);
    return cudaGetLastError();
}

// the fp32 form takes 16-byte vectors of both operands
bool dM_f32_ok(int U, int W, const void* A, const void* G) {
    return U % 4 == 0 && W % 4 == 0 && (reinterpret_cast<uintptr_t>(A) & 15u) == 0 &&
           (reinterpret_cast<uintptr_t>(G) & 15u) == 0;
}

// ----------------------------------------------------------------------------------- host side

SegTab make_seg(const Plan& p, int64_t N, int64_t* tiles) {
    SegTab t{};
    t.n = p.P;
    int64_t tl = 0;
    for (int i = 0; i < p.P && i < kMaxPaths; ++i) {
        t.row0[i] = int64_t(p.paths[i].ooff) * N;
        t.rows[i] = int64_t(2 * p.paths[i].l3 + 1) * N;
        t.tile0[i] = int(tl);
        tl += (t.rows[i] + kTM - 1) / kTM;
    }
    t.tile0[p.P] = int(tl);
    if (tiles) *tiles = tl;
    return t;
}

int64_t max_chunks(const Plan& p, int64_t N) {
    int64_t m = 1;
    for (int i = 0; i < p.P; ++i) m = std::max<int64_t>(m, (int64_t(2 * p.paths[i].l3 + 1) * N + kRowChunk - 1) / kRowChunk);
    return m;
}

template <typename T>
cudaError_t relayout_launch(int64_t N, int A, int B, bool inv, const void* in, void* out, cudaStream_t st) {
    // channel tile: the whole row of channels when its slab fits 32 KB of shared memory (one
    // contiguous node-major run per block), else a multiple of 32 channels that does
    const size_t row = size_t(B | 1) * sizeof(T);
    int TA = int(std::min<size_t>(size_t(A), std::max<size_t>(32, (32768 / row) / 32 * 32)));
    if (TA < A) TA = std::max(32, TA / 32 * 32);
    const size_t smem = size_t(TA) * row;
    dim3 grid(unsigned(N), unsigned((A + TA - 1) / TA));
    cudaError_t e;
    if (inv) {
        auto k = relayout<T, true>;
        e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
        if (e == cudaSuccess) k<<<grid, 256, smem, st>>>(N, A, B, TA, static_cast<const T*>(in), static_cast<T*>(out));
    } else {
        auto k = relayout<T, false>;
        e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
        if (e == cudaSuccess) k<<<grid, 256, smem, st>>>(N, A, B, TA, static_cast<const T*>(in), static_cast<T*>(out));
    }
    return e != cudaSuccess ? e : cudaGetLastError();
}

// The per-path products as tensor-core jobs: segment p = the rows of path p in the
// component-major operand A [Do N][K]; B_p [K][Nc] n-contiguous, or, with b_kcont, the product
// with B_p^T of a [Nc][K] block (k contiguous) so that M needs no transposed copy.
TcJobs tc_product_jobs(const Plan& p, int64_t N, int K, int Nc, const float* A, const float* B, bool b_kcont, float* C,
                       void* bpack, size_t bpack_bytes) {
    TcJobs J{};
    J.bpack = bpack;
    J.bpack_bytes = bpack_bytes;
    J.nseg = p.P;
    for (int i = 0; i < p.P && i < kTcMaxSeg; ++i) {
        J.row0[i] = int64_t(p.paths[i].ooff) * N;
        J.rows[i] = int64_t(2 * p.paths[i].l3 + 1) * N;
    }
    J.K = K;
    J.N = Nc;
    J.b_kcont = b_kcont ? 1 : 0;
    J.A = A;
    J.lda = K;
    J.B = B;
    J.sbk = b_kcont ? 1 : Nc;
    J.sbn = b_kcont ? K : 1;
    J.b_seg_stride = int64_t(K) * Nc;
    J.C = C;
    J.ldc = Nc;
    return J;
}

// in [N][K][Do] -> out [N][Nc][Do] through component-major copies in ws: [Do N K] then [Do N Nc],
// then bp_bytes of room for the tensor-core path's pre-split B (0: CUDA cores only)
template <typename T>
cudaError_t mix_product(const Plan& p, int64_t N, int K, int Nc, const void* in, const void* Bmat, void* out,
                        void* ws, size_t bp_bytes, cudaStream_t st) {
    T* inT = static_cast<T*>(ws);
    T* outT = reinterpret_cast<T*>(static_cast<char*>(ws) + (size_t(N) * p.Do * K * sizeof(T) + 255) / 256 * 256);
    cudaError_t e = relayout_launch<T>(N, K, p.Do, false, in, inT, st);
    if (e != cudaSuccess) return e;
    int64_t tiles = 0;
    const SegTab tab = make_seg(p, N, &tiles);
    if (tiles > INT32_MAX) return cudaErrorInvalidConfiguration;
    bool done = false;
    if (sizeof(T) == 4 && bp_bytes) {
        // fp32: the per-path products on the tensor cores (3xTF32), B_p = Bmat + p K Nc, its
        // pre-split tiles after the two component-major copies in ws
        void* bp = reinterpret_cast<char*>(outT) + (size_t(N) * p.Do * Nc * sizeof(T) + 255) / 256 * 256;
        TcJobs J = tc_product_jobs(p, N, K, Nc, reinterpret_cast<const float*>(inT),
                                   reinterpret_cast<const float*>(Bmat), false, reinterpret_cast<float*>(outT), bp,
                                   bp_bytes);
        if (tc_gemm_supported(J)) {
            if ((e = launch_tc_gemm(J, st)) != cudaSuccess) return e;
            done = true;
        }
    }
    if (!done) {
        seg_gemm<T><<<dim3(unsigned(tiles), unsigned((Nc + kTN - 1) / kTN)), 256, 0, st>>>(
            K, Nc, tab, inT, static_cast<const T*>(Bmat), outT);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    return relayout_launch<T>(N, Nc, p.Do, true, outT, out, st);
}

}  // namespace

int mix_max_paths() { return kMaxPaths; }

// ------------------------------------------------- single dense products (radial last layer)

// C[rows][Nc] = A[rows][K] B, with B [K][Nc] (b_kcont = 0) or given as the [Nc][K] block B^T
// (b_kcont = 1).  fp32: the tensor cores when the shapes allow; otherwise (fp64, other shapes) the
// register-tiled CUDA-core product, which needs B as [K][Nc] (a transposed copy in `ws`,
// K * Nc elements, for b_kcont).
namespace {
TcJobs dense_jobs(int64_t rows, int K, int Nc, const void* A, const void* B, bool b_kcont, void* C, void* ws,
                  size_t ws_bytes) {
    TcJobs J{};
    J.nseg = 1;
    J.row0[0] = 0;
    J.rows[0] = rows;
    J.K = K;
    J.N = Nc;
    J.b_kcont = b_kcont ? 1 : 0;
    J.A = static_cast<const float*>(A);
    J.lda = K;
    J.B = static_cast<const float*>(B);
    J.sbk = b_kcont ? 1 : Nc;
    J.sbn = b_kcont ? K : 1;
    J.b_seg_stride = 0;
    J.C = static_cast<float*>(C);
    J.ldc = Nc;
    J.bpack = ws;
    J.bpack_bytes = ws_bytes;
    return J;
}
}  // namespace

cudaError_t launch_dense_product(bool f64, int64_t rows, int K, int Nc, const void* A, const void* B, bool b_kcont,
                                 void* C, void* ws, size_t ws_bytes, cudaStream_t st) {
    if (rows <= 0 || Nc <= 0) return cudaSuccess;
    if (ws_bytes < dense_product_workspace(K, Nc, f64)) return cudaErrorInvalidValue;
    if (!f64) {
        TcJobs J = dense_jobs(rows, K, Nc, A, B, b_kcont, C, ws, ws_bytes);
        if (tc_gemm_supported(J)) return launch_tc_gemm(J, st);
    }
    const void* Bn = B;
    cudaError_t e;
    if (b_kcont) {  // [Nc][K] -> [K][Nc]
        const int64_t n = int64_t(K) * Nc;
        const unsigned nb = unsigned((n + 255) / 256);
        if (f64) transpose_M<double><<<nb, 256, 0, st>>>(1, Nc, K, static_cast<const double*>(B), static_cast<double*>(ws));
        else transpose_M<float><<<nb, 256, 0, st>>>(1, Nc, K, static_cast<const float*>(B), static_cast<float*>(ws));
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
        Bn = ws;
    }
    SegTab tab{};
    tab.n = 1;
    tab.row0[0] = 0;
    tab.rows[0] = rows;
    tab.tile0[0] = 0;
    const int64_t tiles = (rows + kTM - 1) / kTM;
    if (tiles > INT32_MAX) return cudaErrorInvalidConfiguration;
    tab.tile0[1] = int(tiles);
    const dim3 grid(unsigned(tiles), unsigned((Nc + kTN - 1) / kTN));
    if (f64) seg_gemm<double><<<grid, 256, 0, st>>>(K, Nc, tab, static_cast<const double*>(A), static_cast<const double*>(Bn), static_cast<double*>(C));
    else seg_gemm<float><<<grid, 256, 0, st>>>(K, Nc, tab, static_cast<const float*>(A), static_cast<const float*>(Bn), static_cast<float*>(C));
    return cudaGetLastError();
}

// the tensor-core path's pre-split B tiles, or the CUDA-core path's transposed B
size_t dense_product_workspace(int K, int Nc, bool f64) {
    const size_t t = size_t(K) * Nc * (f64 ? 8 : 4);
    if (f64) return t;
    TcJobs J = dense_jobs(1, K, Nc, nullptr, nullptr, false, nullptr, nullptr, 0);
    return std::max(t, tc_gemm_workspace(J));
}

// C[Mr][Nc] = sum over rows of A[row][m] G[row][n]: fp32 steps of 16 rows, Kahan-compensated,
// fp64 partials per chunk of kRowChunk rows (in `ws`) added in chunk order -- deterministic.
size_t dense_reduction_workspace(int64_t rows, int Mr, int Nc) {
    const int64_t C = std::max<int64_t>(1, (rows + kRowChunk - 1) / kRowChunk);
    return size_t(C) * Mr * Nc * sizeof(double);
}

cudaError_t launch_dense_reduction(bool f64, int64_t rows, int Mr, int Nc, const void* A, const void* G, void* C, void* ws,
                                   cudaStream_t st) {
    if (Mr <= 0 || Nc <= 0) return cudaSuccess;
    if (rows <= 0) return cudaMemsetAsync(C, 0, size_t(Mr) * Nc * (f64 ? 8 : 4), st);
    SegTab tab{};
    tab.n = 1;
    tab.row0[0] = 0;
    tab.rows[0] = rows;
    const int64_t nch = (rows + kRowChunk - 1) / kRowChunk;
    if (!f64 && dM_f32_ok(Mr, Nc, A, G)) {
        cudaError_t e0 = launch_dM_f32(Mr, Nc, tab, 1u, unsigned(nch), static_cast<const float*>(A),
                                       static_cast<const float*>(G), static_cast<double*>(ws), st);
        if (e0 != cudaSuccess) return e0;
        return launch_column_sum(ws, nch, int64_t(Mr) * Nc, C, f64, st);
    }
    const unsigned tiles = unsigned(((Mr + kDT - 1) / kDT) * ((Nc + kDT - 1) / kDT));
    const dim3 grid(tiles, 1u, unsigned(nch));
    if (f64)
        seg_dM<double><<<grid, 256, 0, st>>>(Mr, Nc, tab, static_cast<const double*>(A), static_cast<const double*>(G),
                                              static_cast<double*>(ws));
    else
        seg_dM<float><<<grid, 256, 0, st>>>(Mr, Nc, tab, static_cast<const float*>(A), static_cast<const float*>(G),
                                             static_cast<double*>(ws));
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    return launch_column_sum(ws, nch, int64_t(Mr) * Nc, C, f64, st);
}

namespace {
size_t r256(size_t b) { return (b + 255) / 256 * 256; }
}  // namespace

// Workspace regions (each starting on a 256-byte boundary).  Forward: [in | out] component-major.
// Backward: [g | d_in] component-major (the input-gradient product; g alone for dM), in
// component-major, M transposed, fp64 dM partials.
// Pre-split M tiles of the tensor-core products (fp32 plans): forward (K = U, N = W) and input
// gradient (K = W, N = U).
size_t tc_pack_bytes(const Plan& p, int64_t N, int W, bool bwd) {
    if (p.dtype != UVU_F32) return 0;
    TcJobs J = tc_product_jobs(p, N, bwd ? W : p.U, bwd ? p.U : W, nullptr, nullptr, bwd, nullptr, nullptr, 0);
    return tc_gemm_workspace(J);
}

size_t mix_workspace_bytes(const Plan& p, int64_t N, int W, bool bwd) {
    const size_t s = p.elem(), ND = size_t(N) * p.Do;
    const size_t U = size_t(p.U);
    if (!bwd) return r256(ND * U * s) + r256(ND * W * s) + r256(tc_pack_bytes(p, N, W, false));
    return r256(ND * W * s) + r256(ND * U * s) + r256(ND * U * s) + r256(size_t(p.P) * U * W * s) +
           r256(size_t(max_chunks(p, N)) * p.P * U * W * sizeof(double)) + r256(tc_pack_bytes(p, N, W, true));
}

cudaError_t launch_mix_fwd(const Plan& p, int64_t N, int W, const void* in, const void* M, void* out, void* ws,
                           cudaStream_t st) {
    if (N == 0) return cudaSuccess;
    return p.dtype == UVU_F64 ? mix_product<double>(p, N, p.U, W, in, M, out, ws, 0, st)
                              : mix_product<float>(p, N, p.U, W, in, M, out, ws, tc_pack_bytes(p, N, W, false), st);
}

cudaError_t launch_mix_bwd(const Plan& p, int64_t N, int W, const void* in, const void* M, const void* g, void* d_in,
                           void* dM, void* ws, cudaStream_t st) {
    const size_t s = p.elem(), ND = size_t(N) * p.Do;
    const size_t PUW = size_t(p.P) * p.U * W;
    if (N == 0) return dM ? cudaMemsetAsync(dM, 0, PUW * s, st) : cudaSuccess;
    char* base = static_cast<char*>(ws);
    void* prod_ws = base;                                // [gT | d_inT], then gT alone for dM
    void* inT = base + r256(ND * W * s) + r256(ND * p.U * s);
    void* Mt = static_cast<char*>(inT) + r256(ND * p.U * s);
    void* part = static_cast<char*>(Mt) + r256(PUW * s);
    const bool f64 = p.dtype == UVU_F64;
    cudaError_t e = cudaSuccess;
    bool d_in_done = false;
    if (d_in && !f64) {
        // tensor cores: d_in_p = g_p M_p^T with M read as the k-contiguous operand (no transposed copy)
        float* gT = static_cast<float*>(prod_ws);
        float* dT = reinterpret_cast<float*>(base + r256(ND * W * s));
        void* bp = static_cast<char*>(part) + r256(size_t(max_chunks(p, N)) * PUW * sizeof(double));
        TcJobs J = tc_product_jobs(p, N, W, p.U, gT, static_cast<const float*>(M), true, dT, bp, tc_pack_bytes(p, N, W, true));
        if (tc_gemm_supported(J)) {
            if ((e = relayout_launch<float>(N, W, p.Do, false, g, gT, st)) != cudaSuccess) return e;
            if ((e = launch_tc_gemm(J, st)) != cudaSuccess) return e;
            if ((e = relayout_launch<float>(N, p.U, p.Do, true, dT, d_in, st)) != cudaSuccess) return e;
            d_in_done = true;
        }
    }
    if (d_in && !d_in_done) {
        const unsigned nb = unsigned((PUW + 255) / 256);
        if (f64) transpose_M<double><<<nb, 256, 0, st>>>(p.P, p.U, W, static_cast<const double*>(M), static_cast<double*>(Mt));
        else transpose_M<float><<<nb, 256, 0, st>>>(p.P, p.U, W, static_cast<const float*>(M), static_cast<float*>(Mt));
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
        e = f64 ? mix_product<double>(p, N, W, p.U, g, Mt, d_in, prod_ws, 0, st)
                : mix_product<float>(p, N, W, p.U, g, Mt, d_in, prod_ws, 0, st);
        if (e != cudaSuccess) return e;
    }
    if (dM) {
        void* gT = prod_ws;
        e = f64 ? relayout_launch<double>(N, p.U, p.Do, false, in, inT, st)
                : relayout_launch<float>(N, p.U, p.Do, false, in, inT, st);
        if (e != cudaSuccess) return e;
        e = f64 ? relayout_launch<double>(N, W, p.Do, false, g, gT, st)
                : relayout_launch<float>(N, W, p.Do, false, g, gT, st);
        if (e != cudaSuccess) return e;
        const SegTab tab = make_seg(p, N, nullptr);
        const int64_t C = max_chunks(p, N);
        const unsigned tiles = unsigned(((p.U + kDT - 1) / kDT) * ((W + kDT - 1) / kDT));
        dim3 grid(tiles, unsigned(p.P), unsigned(C));
        if (!f64 && dM_f32_ok(p.U, W, inT, gT)) {
            if ((e = launch_dM_f32(p.U, W, tab, unsigned(p.P), unsigned(C), static_cast<const float*>(inT),
                                   static_cast<const float*>(gT), static_cast<double*>(part), st)) != cudaSuccess)
                return e;
        } else if (f64)
            seg_dM<double><<<grid, 256, 0, st>>>(p.U, W, tab, static_cast<const double*>(inT),
                                                  static_cast<const double*>(gT), static_cast<double*>(part));
        else
            seg_dM<float><<<grid, 256, 0, st>>>(p.U, W, tab, static_cast<const float*>(inT),
                                                 static_cast<const float*>(gT), static_cast<double*>(part));
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
        e = launch_column_sum(part, C, int64_t(PUW), dM, f64, st);
    }
    return e;
}

}  // namespace uvu
