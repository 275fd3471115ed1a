// Arithmetic-rate probe: independent fused multiply-add chains, so that the timed kernel is
// bound by the FP32 (or FP64) pipe alone.  Its rate is the denominator of the ALU fractions the
// benchmark reports next to the HBM fractions (the convolution's fp32 intensity sits near the
// FP32 ridge and the fp64 workload is bound by the FP64 pipe).
//
// Each thread runs kChains independent chains a <- a * b + c with |b| < 1, so the values stay
// finite and normal for any iteration count; the chains' sum is stored so that no chain is dead
// code.  One launch performs grid * block * iters * kChains FMAs (2 flop each).
#include <cuda_runtime.h>

#include <cstdint>

#include "plan.h"

namespace uvu {
namespace {

constexpr int kChains = 8;
constexpr int kProbeThreads = 256;

template <typename T>
__global__ void __launch_bounds__(kProbeThreads) fma_chain_kernel(int iters, T* __restrict__ out) {
    const int gid = blockIdx.x * blockDim.x + threadIdx.x;
    T a[kChains];
#pragma unroll
    for (int i = 0; i < kChains; ++i) a[i] = T(1) + T(gid % 97) * T(1e-3) + T(i) * T(1e-2);
    const T b = T(0.99999), c = T(1e-6);
#pragma unroll 1
    for (int it = 0; it < iters; it += 4) {
#pragma unroll
        for (int r = 0; r < 4; ++r)
#pragma unroll
            for (int i = 0; i < kChains; ++i) a[i] = fma(a[i], b, c);
    }
    T s = 0;
#pragma unroll
    for (int i = 0; i < kChains; ++i) s += a[i];
    out[gid] = s;
}

}  // namespace

cudaError_t launch_fma_probe(bool f64, int blocks, int iters, void* out, cudaStream_t st, double* fmas) {
    const int it = (iters + 3) / 4 * 4;
    if (f64)
        fma_chain_kernel<double><<<blocks, kProbeThreads, 0, st>>>(it, static_cast<double*>(out));
    else
        fma_chain_kernel<float><<<blocks, kProbeThreads, 0, st>>>(it, static_cast<float*>(out));
    if (fmas) *fmas = double(blocks) * kProbeThreads * double(it) * kChains;
    return cudaGetLastError();
}

}  // namespace uvu
