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

// ------------------------------------------------------------------------ reverse pass
// Gradients of <dh, h(r)> with respect to the edge lengths r (for forces) and to the layers'
// weights W_1 .. W_L.  Per tile of TE edges the block recomputes the forward pass into shared
// memory (each layer's activation a_l and its sigmoid s_l = 1 / (1 + exp(-z_l)), from which
// silu'(z_l) = s_l + a_l (1 - s_l)), then walks back:
//     dz_l = g_l * silu'(z_l),   dW_l += a_(l-1)^T dz_l,   g_(l-1) = dz_l W_l^T,
// and finally dr = sum_n g_0[n] d/dr (b_n(r) f(r / r_cut)).  The layer gradients are sums over
// all edges: each block keeps its own running sums in global scratch as compensated fp32 pairs
// (sum, lost low part), updated tile by tile with four-edge partial products by the one thread
// that owns each entry, and a second kernel adds the blocks' pairs in fp64 in block order, so
// the result is deterministic.
namespace uvu {
namespace {

template <typename T>
__device__ __forceinline__ T sigm(T v) { return T(1) / (T(1) + (sizeof(T) == 4 ? T(expf(float(-v))) : T(exp(double(-v))))); }

__device__ __forceinline__ float cos_t(float v) { return cosf(v); }
__device__ __forceinline__ double cos_t(double v) { return cos(v); }

// Kahan step: (s, c) += v
template <typename T>
__device__ __forceinline__ void kahan(T& s, T& c, T v) {
    const T y = v - c;
    const T t = s + y;
    c = (t - s) - y;
    s = t;
}

struct BwdLayout {  // element offsets inside the block's shared memory
    int wt;          // W_l^T blocks, [hout][hin rounded up to 4], zero-padded
    int act[kRadialMaxLayers + 1];
    int sig[kRadialMaxLayers + 1];
    int gA, gB;
    int total;
    int w_off[kRadialMaxLayers + 1];   // offset of W_l in the weight array (row-major [hin][hout])
    int wt_off[kRadialMaxLayers + 1];  // offset of W_l^T inside the wt region
    int w_sm;        // W (as given) staged at offset 0 when nonzero
};

// REG: every layer has at most kThreads 4 x 4 blocks of dW and there are at most kRegLayers
// layers, so each thread keeps its blocks' compensated sums in registers over all its tiles
// (written once at the end) instead of reloading them from the block's scratch row per tile.
constexpr int kRegLayers = 3;
template <typename T, int TE, bool REG>
__global__ void __launch_bounds__(kThreads, 1) radial_hidden_bwd_kernel(long long E, const T* __restrict__ r, T r_cut,
                                                                        int p_env, RadialNet net, BwdLayout L,
                                                                        const T* __restrict__ Wg, int n_w,
                                                                        const T* __restrict__ dh, T* __restrict__ dr,
                                                                        T* __restrict__ acc) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    T* const S = reinterpret_cast<T*>(smem_raw);
    const int tid = threadIdx.x;
    const int nl = net.n_layers, nb = net.widths[0], H = net.widths[nl];
    // weights as given (row-major per layer) and transposed, zero-padded to 4-multiples of hin
    if (L.w_sm)
        for (int i = tid; i < n_w; i += kThreads) S[i] = Wg[i];
    for (int l = 1; l <= nl; ++l) {
        const int hin = net.widths[l - 1], hout = net.widths[l], hinp = (hin + 3) / 4 * 4;
        for (int i = tid; i < hout * hinp; i += kThreads) {
            const int j = i / hinp, k = i - j * hinp;
            S[L.wt + L.wt_off[l] + i] = k < hin ? Wg[L.w_off[l] + k * hout + j] : T(0);
        }
    }
    __syncthreads();
    const T pi_over_rc = T(3.14159265358979323846) / r_cut;
    const T norm = sqrt_t(T(2) / r_cut);
    const T p = T(p_env);
    const T c1 = (p + 1) * (p + 2) / 2, c2 = p * (p + 2), c3 = p * (p + 1) / 2;
    const T d1 = p * (p + 1) * (p + 2) / 2;  // f'(s) = -d1 s^(p-1) + 2 d1 s^p - d1 s^(p+1)
    T* const accb = acc + (size_t)blockIdx.x * n_w * 2;
    bool first = true;
    T rs[kRegLayers][4][4], rc[kRegLayers][4][4];  // REG: this thread's dW block per layer (sum, lost part)
    if (REG) {
#pragma unroll
        for (int l = 0; l < kRegLayers; ++l)
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) rs[l][i][j] = rc[l][i][j] = T(0);
    }
    for (long long t0 = (long long)blockIdx.x * TE; t0 < E; t0 += (long long)gridDim.x * TE) {
        // ---- forward: a_0 = enveloped basis (rows padded to a multiple of 4 with zeros)
        const int nbp = (nb + 3) / 4 * 4;
        for (int i = tid; i < nbp * TE; i += kThreads) {
            const int n = i / TE, e = i - n * TE;
            T b = 0;
            if (n < nb && t0 + e < E) {
                const T rr = r[t0 + e];
                const T s = rr / r_cut;
                if (s < T(1)) {
                    T sp = 1;
                    for (int k = 0; k < p_env; ++k) sp *= s;
                    b = norm * sin_t(T(n + 1) * pi_over_rc * rr) / rr * (T(1) - c1 * sp + c2 * sp * s - c3 * sp * s * s);
                }
            }
            S[L.act[0] + i] = b;
        }
        __syncthreads();
        for (int l = 1; l <= nl; ++l) {
            const int hin = net.widths[l - 1], hout = net.widths[l];
            const T* in = S + L.act[l - 1];
            const T* W = L.w_sm ? S + L.w_off[l] : Wg + L.w_off[l];
            for (int t = tid; t < (TE / 4) * (hout / 4); t += kThreads) {
                const int eq = t % (TE / 4), q = t / (TE / 4);
                T z[4][4] = {};
                for (int k = 0; k < hin; ++k) {
                    const Q4<T> a = lds4(in + k * TE + 4 * eq);
                    const Q4<T> w = L.w_sm ? lds4(W + size_t(k) * hout + 4 * q) : ldg4(W + size_t(k) * hout + 4 * q);
                    const T av[4] = {a.a, a.b, a.c, a.d}, wv[4] = {w.a, w.b, w.c, w.d};
#pragma unroll
                    for (int i = 0; i < 4; ++i)
#pragma unroll
                        for (int j = 0; j < 4; ++j) z[i][j] = fma(av[i], wv[j], z[i][j]);
                }
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    T a4[4], s4[4];
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        s4[i] = sigm(z[i][j]);
                        a4[i] = z[i][j] * s4[i];
                    }
                    st4(S + L.act[l] + (4 * q + j) * TE + 4 * eq, a4[0], a4[1], a4[2], a4[3]);
                    st4(S + L.sig[l] + (4 * q + j) * TE + 4 * eq, s4[0], s4[1], s4[2], s4[3]);
                }
            }
            __syncthreads();
        }
        // ---- backward: g_L = dh rows of the tile (feature-major)
        T* g = S + L.gA;
        T* g2 = S + L.gB;
        for (int i = tid; i < H * TE; i += kThreads) {
            const int k = i / TE, e = i - k * TE;
            g[i] = t0 + e < E ? dh[(t0 + e) * H + k] : T(0);
        }
        __syncthreads();
        for (int l = nl; l >= 1; --l) {
            const int hin = net.widths[l - 1], hout = net.widths[l], hinp = (hin + 3) / 4 * 4;
            // dz_l = g * silu'(z_l), in place
            for (int i = tid; i < hout * TE; i += kThreads) {
                const T s = S[L.sig[l] + i], a = S[L.act[l] + i];
                g[i] *= s + a * (T(1) - s);
            }
            __syncthreads();
            // dW_l += a_(l-1)^T dz_l: 4 x 4 blocks (k, j) per thread, sixteen edges per partial.  The
            // edge groups are visited starting at jb (mod TE/4) so that the lanes of a warp, which
            // differ in jb, read different shared-memory banks (a fixed order per thread).
            const T* ain = S + L.act[l - 1];
            auto block = [&](int kb, int jb, T (&s)[4][4], T (&c)[4][4]) {
                // groups of (up to) 16 edges summed in the working precision, each group's sum added
                // with compensation
                constexpr int G4 = TE / 4 < 4 ? TE / 4 : 4;
                for (int e0 = 0; e0 < TE / 4; e0 += G4) {
                    T v[4][4];
#pragma unroll
                    for (int i = 0; i < 4; ++i)
#pragma unroll
                        for (int j = 0; j < 4; ++j) v[i][j] = T(0);
#pragma unroll
                    for (int e = e0; e < e0 + G4; ++e) {
                        const int e4 = (e + jb) & (TE / 4 - 1);
                        Q4<T> av[4], dv[4];
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            av[i] = lds4(ain + (4 * kb + i) * TE + 4 * e4);
                            dv[i] = lds4(g + (4 * jb + i) * TE + 4 * e4);
                        }
#pragma unroll
                        for (int i = 0; i < 4; ++i)
#pragma unroll
                            for (int j = 0; j < 4; ++j) {
                                v[i][j] = fma(av[i].a, dv[j].a, v[i][j]);
                                v[i][j] = fma(av[i].b, dv[j].b, v[i][j]);
                                v[i][j] = fma(av[i].c, dv[j].c, v[i][j]);
                                v[i][j] = fma(av[i].d, dv[j].d, v[i][j]);
                            }
                    }
#pragma unroll
                    for (int i = 0; i < 4; ++i)
#pragma unroll
                        for (int j = 0; j < 4; ++j) kahan(s[i][j], c[i][j], v[i][j]);
                }
            };
            if (REG) {
                const int b = tid;
                if (b < (hinp / 4) * (hout / 4)) {
#pragma unroll
                    for (int ll = 0; ll < kRegLayers; ++ll)
                        if (ll == l - 1) block(b / (hout / 4), b % (hout / 4), rs[ll], rc[ll]);
                }
            } else {
                for (int b = tid; b < (hinp / 4) * (hout / 4); b += kThreads) {
                    const int kb = b / (hout / 4), jb = b - kb * (hout / 4);
                    T s[4][4], c[4][4];
#pragma unroll
                    for (int i = 0; i < 4; ++i)
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            const int k = 4 * kb + i;
                            const size_t o = (size_t(L.w_off[l]) + size_t(k) * hout + 4 * jb + j) * 2;
                            const bool ok = k < hin && !first;
                            s[i][j] = ok ? accb[o] : T(0);
                            c[i][j] = ok ? accb[o + 1] : T(0);
                        }
                    block(kb, jb, s, c);
#pragma unroll
                    for (int i = 0; i < 4; ++i)
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            const int k = 4 * kb + i;
                            if (k < hin) {
                                const size_t o = (size_t(L.w_off[l]) + size_t(k) * hout + 4 * jb + j) * 2;
                                accb[o] = s[i][j];
                                accb[o + 1] = c[i][j];
                            }
                        }
                }
            }
            // g_(l-1) = dz_l W_l^T: 4 edges x 4 inputs per thread
            const T* WT = S + L.wt + L.wt_off[l];
            for (int t = tid; t < (TE / 4) * (hinp / 4); t += kThreads) {
                const int eq = t % (TE / 4), q = t / (TE / 4);
                T o4[4][4] = {};
                for (int j = 0; j < hout; ++j) {
                    const Q4<T> d = lds4(g + j * TE + 4 * eq);
                    const Q4<T> w = lds4(WT + size_t(j) * hinp + 4 * q);
                    const T dv[4] = {d.a, d.b, d.c, d.d}, wv[4] = {w.a, w.b, w.c, w.d};
#pragma unroll
                    for (int i = 0; i < 4; ++i)
#pragma unroll
                        for (int k = 0; k < 4; ++k) o4[i][k] = fma(dv[i], wv[k], o4[i][k]);
                }
#pragma unroll
                for (int k = 0; k < 4; ++k) st4(g2 + (4 * q + k) * TE + 4 * eq, o4[0][k], o4[1][k], o4[2][k], o4[3][k]);
            }
            __syncthreads();
            T* tmp = g;
            g = g2;
            g2 = tmp;
        }
        // ---- dr = sum_n g_0[n] (b_n' f + b_n f' / r_cut)
        for (int e = tid; e < TE; e += kThreads) {
            if (t0 + e >= E) continue;
            const T rr = r[t0 + e];
            const T s = rr / r_cut;
            T acc_r = 0;
            if (s < T(1)) {
                T sp = 1;
                for (int k = 0; k < p_env - 1; ++k) sp *= s;  // s^(p-1)
                const T f = T(1) - c1 * sp * s + c2 * sp * s * s - c3 * sp * s * s * s;
                const T fd = (-d1 * sp + T(2) * d1 * sp * s - d1 * sp * s * s) / r_cut;
                for (int n = 0; n < nb; ++n) {
                    const T kk = T(n + 1) * pi_over_rc;
                    const T sn = sin_t(kk * rr), cs = cos_t(kk * rr);
                    const T b = norm * sn / rr;
                    const T bd = norm * (kk * cs / rr - sn / (rr * rr));
                    acc_r = fma(g[n * TE + e], bd * f + b * fd, acc_r);
                }
            }
            dr[t0 + e] = acc_r;
        }
        __syncthreads();
        first = false;
    }
    if (REG) {  // this thread's blocks (zeros for a block without any tile)
        for (int l = 1; l <= nl; ++l) {
            const int hin = net.widths[l - 1], hout = net.widths[l], hinp = (hin + 3) / 4 * 4;
            const int b = tid;
            if (b >= (hinp / 4) * (hout / 4)) continue;
            const int kb = b / (hout / 4), jb = b % (hout / 4);
#pragma unroll
            for (int ll = 0; ll < kRegLayers; ++ll) {
                if (ll != l - 1) continue;
#pragma unroll
                for (int i = 0; i < 4; ++i)
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const int k = 4 * kb + i;
                        if (k < hin) {
                            const size_t o = (size_t(L.w_off[l]) + size_t(k) * hout + 4 * jb + j) * 2;
                            accb[o] = rs[ll][i][j];
                            accb[o + 1] = rc[ll][i][j];
                        }
                    }
            }
        }
    } else if (first) {  // a block without any tile still owns its (zero) row of pairs
        for (int i = tid; i < 2 * n_w; i += kThreads) accb[i] = T(0);
    }
}

// out[i] = sum over blocks b, in order, of (sum - lost part) of entry i, in fp64
template <typename T>
__global__ void kahan_column_sum(const T* __restrict__ acc, int nblk, int n_w, T* __restrict__ out) {
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= n_w) return;
    double a = 0;
    for (int b = 0; b < nblk; ++b) {
        const T* q = acc + ((size_t)b * n_w + i) * 2;
        a += double(q[0]) - double(q[1]);
    }
    out[i] = T(a);
}

BwdLayout bwd_layout(const RadialNet& net, int TE, bool w_sm) {
    BwdLayout L{};
    int o = 0, wo = 0, wto = 0;
    L.w_sm = w_sm ? 1 : 0;
    for (int l = 1; l <= net.n_layers; ++l) {
        L.w_off[l] = wo;
        wo += net.widths[l - 1] * net.widths[l];
        L.wt_off[l] = wto;
        wto += net.widths[l] * ((net.widths[l - 1] + 3) / 4 * 4);
    }
    if (w_sm) o = (wo + 3) / 4 * 4;
    L.wt = o;
    o += (wto + 3) / 4 * 4;
    L.act[0] = o;
    o += (net.widths[0] + 3) / 4 * 4 * TE;
    for (int l = 1; l <= net.n_layers; ++l) {
        L.act[l] = o;
        o += net.widths[l] * TE;
        L.sig[l] = o;
        o += net.widths[l] * TE;
    }
    const int mw = std::max(net.max_width, (net.widths[0] + 3) / 4 * 4);
    L.gA = o;
    o += mw * TE;
    L.gB = o;
    o += mw * TE;
    L.total = o;
    return L;
}

constexpr size_t kBwdSmemMax = 220 * 1024;

// tile size and weight staging of the reverse pass: the largest tile (64, 32 or 16 edges) whose
// shared memory fits, with the weights staged when they also fit
bool bwd_config(const RadialNet& net, bool f64, int* te, bool* w_sm, size_t* smem) {
    const size_t es = f64 ? 8 : 4;
    for (int wsm = 1; wsm >= 0; --wsm)
        for (int t : {64, 32, 16}) {
            const BwdLayout L = bwd_layout(net, t, wsm != 0);
            if (size_t(L.total) * es <= kBwdSmemMax) {
                *te = t;
                *w_sm = wsm != 0;
                *smem = size_t(L.total) * es;
                return true;
            }
        }
    return false;
}

template <typename T, int TE>
cudaError_t launch_bwd_t(int64_t E, const void* r, double r_cut, int p_env, const RadialNet& net, const BwdLayout& L,
                         const void* W, const void* dh, void* dr, void* dW, void* ws, size_t smem, int blocks,
                         cudaStream_t st) {
    bool reg = net.n_layers <= kRegLayers;
    for (int l = 1; l <= net.n_layers; ++l)
        reg = reg && ((net.widths[l - 1] + 3) / 4) * (net.widths[l] / 4) <= kThreads;
    auto k = reg ? radial_hidden_bwd_kernel<T, TE, true> : radial_hidden_bwd_kernel<T, TE, false>;
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
    if (e != cudaSuccess) return e;
    const int n_w = weight_count(net);
    k<<<blocks, kThreads, smem, st>>>(E, static_cast<const T*>(r), T(r_cut), p_env, net, L, static_cast<const T*>(W), n_w,
                                      static_cast<const T*>(dh), static_cast<T*>(dr), static_cast<T*>(ws));
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    kahan_column_sum<T><<<(n_w + 255) / 256, 256, 0, st>>>(static_cast<const T*>(ws), blocks, n_w, static_cast<T*>(dW));
    return cudaGetLastError();
}

}  // namespace

// Blocks of the reverse pass: one per SM (its shared memory allows no more), at most one per tile.
int radial_bwd_blocks(int64_t E, const RadialNet& net, bool f64, int sm_count) {
    int te = 64;
    bool wsm = false;
    size_t smem = 0;
    if (!bwd_config(net, f64, &te, &wsm, &smem)) return 0;
    const int64_t tiles = (E + te - 1) / te;
    return int(std::max<int64_t>(1, std::min<int64_t>(tiles, std::max(1, sm_count))));
}

size_t radial_hidden_bwd_workspace(int64_t E, const RadialNet& net, bool f64, int sm_count) {
    const int b = radial_bwd_blocks(E, net, f64, sm_count);
    return size_t(std::max(b, 1)) * weight_count(net) * 2 * (f64 ? 8 : 4);
}

bool radial_hidden_bwd_supported(const RadialNet& net, bool f64) {
    int te;
    bool wsm;
    size_t smem;
    return bwd_config(net, f64, &te, &wsm, &smem);
}

cudaError_t launch_radial_hidden_bwd(int64_t E, const void* r, double r_cut, int p_env, const RadialNet& net,
                                     const void* W, const void* dh, void* dr, void* dW, void* ws, bool f64,
                                     int sm_count, cudaStream_t st) {
    int te = 64;
    bool wsm = false;
    size_t smem = 0;
    if (!bwd_config(net, f64, &te, &wsm, &smem)) return cudaErrorInvalidValue;
    const BwdLayout L = bwd_layout(net, te, wsm);
    const int blocks = radial_bwd_blocks(E, net, f64, sm_count);
    if (E <= 0) {  // no edges: zero layer gradients
        return cudaMemsetAsync(dW, 0, size_t(weight_count(net)) * (f64 ? 8 : 4), st);
    }
#define UVU_BWD(T, TE_) launch_bwd_t<T, TE_>(E, r, r_cut, p_env, net, L, W, dh, dr, dW, ws, smem, blocks, st)
    if (f64) {
        if (te == 64) return UVU_BWD(double, 64);
        if (te == 32) return UVU_BWD(double, 32);
        return UVU_BWD(double, 16);
    }
    if (te == 64) return UVU_BWD(float, 64);
    if (te == 32) return UVU_BWD(float, 32);
    return UVU_BWD(float, 16);
#undef UVU_BWD
}

}  // namespace uvu
