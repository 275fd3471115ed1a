// Radial network of the fused-weight convolution: edge lengths -> hidden features h [E][H].
//
// "Receiver-streaming convolutions for channel-wise UVU tensor products" (replies) has the
// radial weights materialised by a separate network before the convolution and names fusing
// that network into the convolution as the next step.  The network here is the radial network of
// MACE-style potentials: n_basis order-zero spherical Bessel functions of the edge length times a
// polynomial cutoff envelope, then fully connected layers without biases, each followed by SiLU.
// Its last linear layer (hidden -> P x U weights) is not applied here: the fused forward kernel
// applies it per (edge, channel) in registers, so the per-edge weights never reach global memory.
//
// One block takes tiles of 64 edges.  The activations of a tile live in shared memory, feature-
// major ([feature][edge]), so that a thread reads four consecutive edges with one vector load;
// each thread computes a 4 x 4 block (edges x output features) of a layer from four edges'
// inputs and four features' weights per input feature.  The weights of all layers are copied
// into shared memory once per block when they fit in 64 KB (8-64-64-64: 35 KB), else read
// through the read-only cache.
#include <algorithm>
#include <cmath>

#include "plan.h"

namespace uvu {
namespace {

constexpr int kTE = 64;       // edges per tile
constexpr int kThreads = 256;

template <typename T> struct Q4 { T a, b, c, d; };
__device__ __forceinline__ Q4<float> lds4(const float* p) {
    const float4 v = *reinterpret_cast<const float4*>(p);
    return {v.x, v.y, v.z, v.w};
}
__device__ __forceinline__ Q4<double> lds4(const double* p) {
    const double2 u = reinterpret_cast<const double2*>(p)[0], v = reinterpret_cast<const double2*>(p)[1];
    return {u.x, u.y, v.x, v.y};
}
__device__ __forceinline__ Q4<float> ldg4(const float* p) {
    const float4 v = __ldg(reinterpret_cast<const float4*>(p));
    return {v.x, v.y, v.z, v.w};
}
__device__ __forceinline__ Q4<double> ldg4(const double* p) {
    const double2 u = __ldg(reinterpret_cast<const double2*>(p)), v = __ldg(reinterpret_cast<const double2*>(p) + 1);
    return {u.x, u.y, v.x, v.y};
}
__device__ __forceinline__ void st4(float* p, float a, float b, float c, float d) {
    *reinterpret_cast<float4*>(p) = make_float4(a, b, c, d);
}
__device__ __forceinline__ void st4(double* p, double a, double b, double c, double d) {
    reinterpret_cast<double2*>(p)[0] = make_double2(a, b);
    reinterpret_cast<double2*>(p)[1] = make_double2(c, d);
}
__device__ __forceinline__ float silu(float v) { return v / (1.0f + expf(-v)); }
__device__ __forceinline__ double silu(double v) { return v / (1.0 + exp(-v)); }
__device__ __forceinline__ float sin_t(float v) { return sinf(v); }
__device__ __forceinline__ double sin_t(double v) { return sin(v); }
__device__ __forceinline__ float sqrt_t(float v) { return sqrtf(v); }
__device__ __forceinline__ double sqrt_t(double v) { return sqrt(v); }

// W_SM: the layers' weights (n_w values) are copied into shared memory once per block, ahead of
// the activation buffers; otherwise they are read through the read-only cache.
template <typename T, bool W_SM>
__global__ void __launch_bounds__(kThreads) radial_hidden_kernel(long long E, const T* __restrict__ r, T r_cut, int p_env,
                                                                 RadialNet net, const T* __restrict__ Wg, int n_w,
                                                                 T* __restrict__ h) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    T* const wsm = reinterpret_cast<T*>(smem_raw);
    T* const bufA = wsm + (W_SM ? (n_w + 3) / 4 * 4 : 0);
    T* const bufB = bufA + size_t(net.max_width) * kTE;
    const int tid = threadIdx.x;
    if (W_SM) {
        for (int i = tid; i < n_w; i += kThreads) wsm[i] = Wg[i];
        __syncthreads();
    }
    const T* const W = W_SM ? wsm : Wg;
    const int nb = net.widths[0], H = net.widths[net.n_layers];
    const T pi_over_rc = T(3.14159265358979323846) / r_cut;
    const T norm = sqrt_t(T(2) / r_cut);
    const T p = T(p_env);
    const T c1 = (p + 1) * (p + 2) / 2, c2 = p * (p + 2), c3 = p * (p + 1) / 2;
    for (long long t0 = (long long)blockIdx.x * kTE; t0 < E; t0 += (long long)gridDim.x * kTE) {
        // enveloped Bessel basis of the tile's edges; edges past E get zeros
        for (int i = tid; i < nb * kTE; i += kThreads) {
            const int n = i / kTE, e = i - n * kTE;
            T b = 0;
            if (t0 + e < E) {
                const T rr = r[t0 + e];
                const T s = rr / r_cut;
                if (s < T(1)) {
                    T sp = 1;
                    for (int k = 0; k < p_env; ++k) sp *= s;
                    const T env = T(1) - c1 * sp + c2 * sp * s - c3 * sp * s * s;
                    b = norm * sin_t(T(n + 1) * pi_over_rc * rr) / rr * env;
                }
            }
            bufA[n * kTE + e] = b;
        }
        __syncthreads();
        const T* Wl = W;
        for (int l = 0; l < net.n_layers; ++l) {
            const int hin = net.widths[l], hout = net.widths[l + 1];
            const T* in = (l & 1) ? bufB : bufA;
            T* outb = (l & 1) ? bufA : bufB;
            const bool last = l + 1 == net.n_layers;
            const int nq = hout / 4;
            for (int t = tid; t < (kTE / 4) * nq; t += kThreads) {
                const int eq = t % (kTE / 4), q = t / (kTE / 4);
                T acc[4][4] = {};
#pragma unroll 2
                for (int k = 0; k < hin; ++k) {
                    const Q4<T> a = lds4(in + k * kTE + 4 * eq);
                    const Q4<T> w = W_SM ? lds4(Wl + size_t(k) * hout + 4 * q) : ldg4(Wl + size_t(k) * hout + 4 * q);
                    const T av[4] = {a.a, a.b, a.c, a.d}, wv[4] = {w.a, w.b, w.c, w.d};
#pragma unroll
                    for (int i = 0; i < 4; ++i)
#pragma unroll
                        for (int j = 0; j < 4; ++j) acc[i][j] = fma(av[i], wv[j], acc[i][j]);
                }
#pragma unroll
                for (int i = 0; i < 4; ++i)
#pragma unroll
                    for (int j = 0; j < 4; ++j) acc[i][j] = silu(acc[i][j]);
                if (last) {  // h rows of the tile's edges, four features per vector store
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const long long e = t0 + 4 * eq + i;
                        if (e < E) st4(h + e * H + 4 * q, acc[i][0], acc[i][1], acc[i][2], acc[i][3]);
                    }
                } else {
#pragma unroll
                    for (int j = 0; j < 4; ++j) st4(outb + (4 * q + j) * kTE + 4 * eq, acc[0][j], acc[1][j], acc[2][j], acc[3][j]);
                }
            }
            Wl += size_t(hin) * hout;
            __syncthreads();
        }
    }
}

}  // namespace

namespace {
int weight_count(const RadialNet& net) {
    int n = 0;
    for (int l = 0; l < net.n_layers; ++l) n += net.widths[l] * net.widths[l + 1];
    return n;
}
// weights staged in shared memory when they take at most this many bytes
constexpr size_t kWeightSmemMax = 64 * 1024;

// Persistent grid: the blocks that are resident at once (a whole number per SM), each looping
// over tiles.
template <typename T, bool W_SM>
cudaError_t launch_t(int64_t E, const void* r, double r_cut, int p_env, const RadialNet& net, const void* W, void* h,
                     size_t smem, int sm_count, cudaStream_t st) {
    auto k = radial_hidden_kernel<T, W_SM>;
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
    int per_sm = 0;
    if (e == cudaSuccess) e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k, kThreads, smem);
    if (e != cudaSuccess) return e;
    const int64_t tiles = (E + kTE - 1) / kTE;
    const unsigned blocks = unsigned(std::min<int64_t>(tiles, int64_t(std::max(1, sm_count)) * std::max(1, per_sm)));
    k<<<blocks, kThreads, smem, st>>>(E, static_cast<const T*>(r), T(r_cut), p_env, net, static_cast<const T*>(W),
                                      weight_count(net), static_cast<T*>(h));
    return cudaGetLastError();
}
}  // namespace

size_t radial_hidden_smem(const RadialNet& net, bool f64) {
    const size_t es = f64 ? 8 : 4;
    const size_t wb = size_t(weight_count(net) + 3) / 4 * 4 * es;
    return 2 * size_t(net.max_width) * kTE * es + (wb <= kWeightSmemMax ? wb : 0);
}

cudaError_t launch_radial_hidden(int64_t E, const void* r, double r_cut, int p_env, const RadialNet& net, const void* W,
                                 void* h, bool f64, int sm_count, cudaStream_t st) {
    if (E <= 0) return cudaSuccess;
    const size_t es = f64 ? 8 : 4;
    const bool wsm = size_t(weight_count(net) + 3) / 4 * 4 * es <= kWeightSmemMax;
    const size_t smem = radial_hidden_smem(net, f64);
    if (f64)
        return wsm ? launch_t<double, true>(E, r, r_cut, p_env, net, W, h, smem, sm_count, st)
                   : launch_t<double, false>(E, r, r_cut, p_env, net, W, h, smem, sm_count, st);
    return wsm ? launch_t<float, true>(E, r, r_cut, p_env, net, W, h, smem, sm_count, st)
               : launch_t<float, false>(E, r, r_cut, p_env, net, W, h, smem, sm_count, st);
}

}  // namespace uvu
