// Per-path channel mixing that reduces a factorised UVW convolution to the UVU one
// ("Receiver-streaming convolutions for channel-wise UVU tensor products", replies: UVW cases
// that can be reduced to UVU).  With per-edge weights W_e[p,u,w] = w[e,p,u] M[p,u,w], the
// mixing M is the same on every edge and commutes with the sum over a receiver's edges:
//     out[r,w,ooff(p)+m3] = sum_u M[p,u,w] in[r,u,ooff(p)+m3]        in = the UVU output.
// Three kernels: the mixing, its input gradient (the same contraction with M transposed) and
// dM[p,u,w] = sum_r sum_m3 in[r,u,ooff+m3] g[r,w,ooff+m3], the last one over fixed receiver
// chunks into fp64 partial rows that are then added in chunk order (deterministic).
#include "plan.h"

namespace uvu {
namespace {

constexpr int kMaxD3 = 9;   // 2 l3 + 1 for l3 <= 4
constexpr int kMT = 128;    // threads per block of the row kernels
constexpr int kMaxPaths = 128;

struct PathTab {
    int n;
    int ooff[kMaxPaths];
    int d3[kMaxPaths];
};

// out[r, c0 + t, :] for RB receivers per block, channels c0 .. c0 + kMT - 1 of the output side:
//   out[r, c, ooff+m] = sum_k A(p, k, c) in[r, k, ooff+m],  A(p, k, c) = M[(p K + k) ldk + c] when
// k runs over the input channels (forward: K = U, C = W, A = M), or M[(p C + c) ldk + k] for the
// input gradient (K = W, C = U, A = M transposed).
template <typename T, int RB, bool TRANS>
__global__ void __launch_bounds__(kMT) mix_rows(int64_t N, int K, int C, int Do, PathTab tab,
                                                const T* __restrict__ in, const T* __restrict__ M,
                                                T* __restrict__ out) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    T* s_in = reinterpret_cast<T*>(smem_raw);            // [RB][K][Do]
    T* s_out = s_in + size_t(RB) * K * Do;               // [RB][kMT][Do]
    const int64_t r0 = int64_t(blockIdx.x) * RB;
    const int c0 = blockIdx.y * kMT, tc = threadIdx.x, c = c0 + tc;
    const int nr = int(N - r0 < RB ? N - r0 : int64_t(RB));
    const int nc = min(kMT, C - c0);
    for (int64_t i = threadIdx.x; i < int64_t(nr) * K * Do; i += kMT) s_in[i] = in[r0 * K * Do + i];
    __syncthreads();
    if (c < C) {
        for (int pi = 0; pi < tab.n; ++pi) {
            const int o = tab.ooff[pi], d = tab.d3[pi];
            T acc[RB][kMaxD3];
#pragma unroll
            for (int rb = 0; rb < RB; ++rb)
#pragma unroll
                for (int m = 0; m < kMaxD3; ++m) acc[rb][m] = 0;
            for (int k = 0; k < K; ++k) {
                const T a = TRANS ? __ldg(M + (size_t(pi) * C + c) * K + k) : __ldg(M + (size_t(pi) * K + k) * C + c);
#pragma unroll
                for (int rb = 0; rb < RB; ++rb) {
                    const T* row = s_in + (size_t(rb) * K + k) * Do + o;
#pragma unroll
                    for (int m = 0; m < kMaxD3; ++m)
                        if (m < d) acc[rb][m] = fma(a, row[m], acc[rb][m]);
                }
            }
#pragma unroll
            for (int rb = 0; rb < RB; ++rb)
#pragma unroll
                for (int m = 0; m < kMaxD3; ++m)
                    if (m < d) s_out[(size_t(rb) * kMT + tc) * Do + o + m] = acc[rb][m];
        }
    }
    __syncthreads();
    // the block's output rows [r][c0 .. c0 + nc)[0 .. Do) are contiguous: coalesced copy-out
    for (int rb = 0; rb < nr; ++rb) {
        T* dst = out + ((r0 + rb) * C + c0) * Do;
        const T* srcp = s_out + size_t(rb) * kMT * Do;
        for (int i = threadIdx.x; i < nc * Do; i += kMT) dst[i] = srcp[i];
    }
}

// dM partials: block (u-tile, w-tile) x path x receiver chunk; 16 x 16 threads, each owning a
// 4 x 4 (u, w) register tile; rows of in and g for the tile staged in shared memory per receiver.
constexpr int kTile = 64;
template <typename T>
__global__ void __launch_bounds__(256) mix_dM(int64_t N, int U, int W, int Do, PathTab tab, int64_t chunk,
                                              const T* __restrict__ in, const T* __restrict__ g,
                                              double* __restrict__ part) {
    __shared__ T s_a[kTile][kMaxD3 + 1];
    __shared__ T s_b[kTile][kMaxD3 + 1];
    const int nwt = (W + kTile - 1) / kTile;
    const int u0 = (blockIdx.x / nwt) * kTile, w0 = (blockIdx.x % nwt) * kTile;
    const int pi = blockIdx.y;
    const int64_t ck = blockIdx.z;
    const int o = tab.ooff[pi], d = tab.d3[pi];
    const int ty = threadIdx.x / 16, tx = threadIdx.x % 16;
    // sums over up to 16 receivers in the plan's type, added into fp64 (FP64 FMAs are slow on
    // this part; a long fp32 sum loses digits where the terms cancel)
    double acc[4][4] = {};
    T acc_c[4][4] = {};
    int nacc = 0;
    const int64_t r_end = min(N, (ck + 1) * chunk);
    for (int64_t r = ck * chunk; r < r_end; ++r) {
        for (int i = threadIdx.x; i < kTile * d; i += 256) {
            const int row = i / d, m = i - row * d;
            const int u = u0 + row, w = w0 + row;
            s_a[row][m] = u < U ? in[(r * U + u) * Do + o + m] : T(0);
            s_b[row][m] = w < W ? g[(r * W + w) * Do + o + m] : T(0);
        }
        __syncthreads();
        for (int m = 0; m < d; ++m) {
            T a[4], b[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) a[i] = s_a[ty * 4 + i][m];
#pragma unroll
            for (int j = 0; j < 4; ++j) b[j] = s_b[tx * 4 + j][m];
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) acc_c[i][j] = fma(a[i], b[j], acc_c[i][j]);
        }
        __syncthreads();
        if (++nacc == 16 || r + 1 == r_end) {
            nacc = 0;
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    acc[i][j] += double(acc_c[i][j]);
                    acc_c[i][j] = T(0);
                }
        }
    }
    double* pr = part + (size_t(ck) * tab.n + pi) * size_t(U) * W;
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int u = u0 + ty * 4 + i, w = w0 + tx * 4 + j;
            if (u < U && w < W) pr[size_t(u) * W + w] = acc[i][j];
        }
}

PathTab make_tab(const Plan& p) {
    PathTab t{};
    t.n = p.P;
    for (int i = 0; i < p.P && i < kMaxPaths; ++i) {
        t.ooff[i] = p.paths[i].ooff;
        t.d3[i] = 2 * p.paths[i].l3 + 1;
    }
    return t;
}

template <typename T, bool TRANS>
cudaError_t rows_launch(const Plan& p, int64_t N, int K, int C, const void* in, const void* M, void* out, cudaStream_t st) {
    const PathTab tab = make_tab(p);
    const int Do = p.Do;
    // two receivers per block when their rows fit in shared memory, else one
    const size_t per = (size_t(K) + kMT) * Do * sizeof(T);
    const bool two = 2 * per <= 200 * 1024;
    const size_t smem = (two ? 2 : 1) * per;
    if (smem > 227 * 1024) return cudaErrorInvalidConfiguration;
    const int rb = two ? 2 : 1;
    dim3 grid(unsigned((N + rb - 1) / rb), unsigned((C + kMT - 1) / kMT));
    const T* a = static_cast<const T*>(in);
    const T* m = static_cast<const T*>(M);
    T* o = static_cast<T*>(out);
    cudaError_t e;
    if (two) {
        auto k = mix_rows<T, 2, TRANS>;
        e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
        if (e == cudaSuccess) k<<<grid, kMT, smem, st>>>(N, K, C, Do, tab, a, m, o);
    } else {
        auto k = mix_rows<T, 1, TRANS>;
        e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
        if (e == cudaSuccess) k<<<grid, kMT, smem, st>>>(N, K, C, Do, tab, a, m, o);
    }
    return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace

int mix_max_paths() { return kMaxPaths; }
int mix_max_d3() { return kMaxD3; }

size_t mix_dM_chunks(int64_t N) { return size_t(std::min<int64_t>(std::max<int64_t>(N, 1), 32)); }

cudaError_t launch_mix_fwd(const Plan& p, int64_t N, int W, const void* in, const void* M, void* out, cudaStream_t st) {
    if (N == 0) return cudaSuccess;
    return p.dtype == UVU_F64 ? rows_launch<double, false>(p, N, p.U, W, in, M, out, st)
                              : rows_launch<float, false>(p, N, p.U, W, in, M, out, st);
}

cudaError_t launch_mix_bwd_in(const Plan& p, int64_t N, int W, const void* g, const void* M, void* d_in, cudaStream_t st) {
    if (N == 0) return cudaSuccess;
    return p.dtype == UVU_F64 ? rows_launch<double, true>(p, N, W, p.U, g, M, d_in, st)
                              : rows_launch<float, true>(p, N, W, p.U, g, M, d_in, st);
}

cudaError_t launch_mix_bwd_M(const Plan& p, int64_t N, int W, const void* in, const void* g, void* part, void* dM,
                             cudaStream_t st) {
    const int64_t cols = int64_t(p.P) * p.U * W;
    if (N == 0) return cudaMemsetAsync(dM, 0, size_t(cols) * p.elem(), st);
    const PathTab tab = make_tab(p);
    const int64_t C = int64_t(mix_dM_chunks(N));
    const int64_t chunk = (N + C - 1) / C;
    const unsigned tiles = unsigned(((p.U + kTile - 1) / kTile) * ((W + kTile - 1) / kTile));
    dim3 grid(tiles, unsigned(p.P), unsigned(C));
    double* pr = static_cast<double*>(part);
    if (p.dtype == UVU_F64)
        mix_dM<double><<<grid, 256, 0, st>>>(N, p.U, W, p.Do, tab, chunk, static_cast<const double*>(in),
                                              static_cast<const double*>(g), pr);
    else
        mix_dM<float><<<grid, 256, 0, st>>>(N, p.U, W, p.Do, tab, chunk, static_cast<const float*>(in),
                                             static_cast<const float*>(g), pr);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    return launch_column_sum(part, C, cols, dM, p.dtype == UVU_F64, st);
}

}  // namespace uvu
