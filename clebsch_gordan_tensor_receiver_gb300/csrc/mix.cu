// Per-path channel mixing that reduces a factorised UVW convolution to the UVU one
// ("Receiver-streaming convolutions for channel-wise UVU tensor products", replies: UVW cases
// that can be reduced to UVU).  With per-edge weights W_e[p,u,w] = w[e,p,u] M[p,u,w], the
// mixing M is the same on every edge and commutes with the sum over a receiver's edges:
//     out[r,w,ooff(p)+m3] = sum_u M[p,u,w] in[r,u,ooff(p)+m3]        in = the UVU output.
// Two kernels: the mixing and its input gradient (one tiled product kernel, M or M transposed) and
// dM[p,u,w] = sum_r sum_m3 in[r,u,ooff+m3] g[r,w,ooff+m3], the last one over fixed receiver
// chunks into fp64 partial rows that are then added in chunk order (deterministic).
#include "plan.h"

namespace uvu {
namespace {

constexpr int kMaxD3 = 9;   // 2 l3 + 1 for l3 <= 4
constexpr int kMaxPaths = 128;

struct PathTab {
    int n;
    int ooff[kMaxPaths];
    int d3[kMaxPaths];
};

// The mixing and its input gradient are, per path p, a dense product
//   out_p[q, c] = sum_k in_p[q, k] B_p[k, c],   q = (r, m) over N x (2 l3 + 1) rows,
// with in_p[q, k] = in[r, k, ooff + m] and B_p = M[p] (forward: K = U, C = W) or M[p]^T (input
// gradient: K = W, C = U).  One block computes a 64-row x 128-column tile of one path with 256
// threads, each owning a 4 x 8 register tile; k advances in chunks of 32 staged in shared memory
// (rows of `in` gathered as (r, m) pairs, M read along its contiguous index).
constexpr int kRows = 64, kCols = 128, kK = 32;

struct TileTab {
    int n;
    int ooff[kMaxPaths];
    int d3[kMaxPaths];
    int tile0[kMaxPaths + 1];  // first row-tile index of each path (prefix over paths)
};

template <typename T, bool TRANS>
__global__ void __launch_bounds__(256) mix_gemm(int64_t N, int K, int C, int Do, TileTab tab,
                                                const T* __restrict__ in, const T* __restrict__ M,
                                                T* __restrict__ out) {
    __shared__ __align__(16) T sA[kK][kRows];   // A transposed: [k][q]
    __shared__ __align__(16) T sB[kK][kCols];   // [k][c]
    int pi = 0;
    while (pi + 1 < tab.n && int(blockIdx.x) >= tab.tile0[pi + 1]) ++pi;
    const int o = tab.ooff[pi], d = tab.d3[pi];
    const int64_t nq = N * d;
    const int64_t q0 = int64_t(int(blockIdx.x) - tab.tile0[pi]) * kRows;
    const int c0 = blockIdx.y * kCols;
    const int tr = threadIdx.x / 16, tc = threadIdx.x % 16;
    T acc[4][8];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[i][j] = 0;
    // The next k-chunk's elements are loaded into registers while the current one is computed
    // (8 of A and 16 of B per thread).  Both tiles are staged with the row / column index
    // fastest across threads (conflict-free shared-memory writes); M is small and L2-resident.
    T ra[kRows * kK / 256], rb[kK * kCols / 256];
    auto load = [&](int k0) {
#pragma unroll
        for (int t = 0; t < kRows * kK / 256; ++t) {
            const int e = threadIdx.x + t * 256;
            const int qi = e % kRows, ki = e / kRows;
            const int64_t q = q0 + qi;
            const int k = k0 + ki;
            T v = 0;
            if (q < nq && k < K) {
                const int64_t r = q / d;
                const int m = int(q - r * d);
                v = in[(r * K + k) * Do + o + m];
            }
            ra[t] = v;
        }
#pragma unroll
        for (int t = 0; t < kK * kCols / 256; ++t) {
            const int e = threadIdx.x + t * 256;
            const int ci = e % kCols, ki = e / kCols;
            const int k = k0 + ki, c = c0 + ci;
            T v = 0;
            if (k < K && c < C) v = TRANS ? M[(size_t(pi) * C + c) * K + k] : M[(size_t(pi) * K + k) * C + c];
            rb[t] = v;
        }
    };
    auto store = [&]() {
#pragma unroll
        for (int t = 0; t < kRows * kK / 256; ++t) {
            const int e = threadIdx.x + t * 256;
            sA[e / kRows][e % kRows] = ra[t];
        }
#pragma unroll
        for (int t = 0; t < kK * kCols / 256; ++t) {
            const int e = threadIdx.x + t * 256;
            sB[e / kCols][e % kCols] = rb[t];
        }
    };
    load(0);
    for (int k0 = 0; k0 < K; k0 += kK) {
        store();
        __syncthreads();
        if (k0 + kK < K) load(k0 + kK);
#pragma unroll 8
        for (int ki = 0; ki < kK; ++ki) {
            T a[4], b[8];
#pragma unroll
            for (int i = 0; i < 4; ++i) a[i] = sA[ki][tr * 4 + i];
#pragma unroll
            for (int j = 0; j < 8; ++j) b[j] = sB[ki][tc * 8 + j];
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 8; ++j) acc[i][j] = fma(a[i], b[j], acc[i][j]);
        }
        __syncthreads();
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int64_t q = q0 + tr * 4 + i;
        if (q >= nq) continue;
        const int64_t r = q / d;
        const int m = int(q - r * d);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const int c = c0 + tc * 8 + j;
            if (c < C) out[(r * C + c) * Do + o + m] = acc[i][j];
        }
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
    TileTab tab{};
    tab.n = p.P;
    int64_t tiles = 0;
    for (int i = 0; i < p.P && i < kMaxPaths; ++i) {
        tab.ooff[i] = p.paths[i].ooff;
        tab.d3[i] = 2 * p.paths[i].l3 + 1;
        tab.tile0[i] = int(tiles);
        tiles += (N * tab.d3[i] + kRows - 1) / kRows;
    }
    tab.tile0[p.P] = int(tiles);
    if (tiles > INT32_MAX) return cudaErrorInvalidConfiguration;
    dim3 grid(unsigned(tiles), unsigned((C + kCols - 1) / kCols));
    mix_gemm<T, TRANS><<<grid, 256, 0, st>>>(N, K, C, p.Do, tab, static_cast<const T*>(in), static_cast<const T*>(M),
                                             static_cast<T*>(out));
    return cudaGetLastError();
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
