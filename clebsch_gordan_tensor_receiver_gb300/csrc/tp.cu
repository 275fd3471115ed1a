// Batched (non-convolution) tensor product: the final step of dw for weights shared by the
// whole batch.  The generated edge kernel leaves one fp64 partial dw [P][U] per block (each
// block's fixed set of samples, summed in sample order); this kernel adds the block rows in
// ascending block order in fp64, one thread per (path, channel) column, and rounds once to the
// plan's type, so the result does not depend on timing.
#include "plan.h"

namespace uvu {
namespace {

template <typename T>
__global__ void column_sum_kernel(const double* __restrict__ part, int64_t rows, int64_t cols, T* __restrict__ out) {
    const int64_t c = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
    if (c >= cols) return;
    double acc = 0;
    for (int64_t r = 0; r < rows; ++r) acc += part[r * cols + c];
    out[c] = T(acc);
}

}  // namespace

cudaError_t launch_column_sum(const void* part, int64_t rows, int64_t cols, void* out, bool f64, cudaStream_t st) {
    // part: fp64 [rows][cols]; out: [cols] of the plan's type (fp64 if f64)
    if (cols <= 0) return cudaSuccess;
    const int threads = 256;
    const unsigned blocks = unsigned((cols + threads - 1) / threads);
    if (f64)
        column_sum_kernel<double><<<blocks, threads, 0, st>>>(static_cast<const double*>(part), rows, cols,
                                                              static_cast<double*>(out));
    else
        column_sum_kernel<float><<<blocks, threads, 0, st>>>(static_cast<const double*>(part), rows, cols,
                                                             static_cast<float*>(out));
    return cudaGetLastError();
}

}  // namespace uvu
