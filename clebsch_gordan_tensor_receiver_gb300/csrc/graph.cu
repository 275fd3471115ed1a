// Graph preparation kernels: receiver CSR from receiver-sorted edges, the transposed (sender)
// CSR, and an on-device validity check.
//
// "Receiver-streaming convolutions for channel-wise UVU tensor products" (opening post,
// benchmark paragraph) runs on prepared receiver-sorted edge lists and keeps graph construction
// out of the timed region; these kernels are that preparation.  Every output word is written by
// exactly one thread and the sender order is fixed (ascending edge id), so the result is
// bit-exact regardless of scheduling.
#include <cuda_runtime.h>

#include <climits>
#include <cstdint>
#include <map>
#include <mutex>
#include <string>

#include "plan.h"

namespace uvu {
namespace {

constexpr int kThreads = 256;

int grid_for(int64_t n) {
    int64_t b = (n + kThreads - 1) / kThreads;
    if (b < 1) b = 1;
    if (b > 152 * 32) b = 152 * 32;  // grid-stride loops cover the rest
    return int(b);
}

// offsets[r] = #{e : recv[e] < r}.  The thread owning edge e writes every offset in
// (recv[e-1], recv[e]]; the last edge also writes (recv[E-1], N].  Every write is clamped to
// [0, N], so a receiver id outside [0, N) or a decreasing recv (a broken precondition) leaves an
// invalid CSR, which uvu_graph_validate reports, and never a write outside recv_offsets.
__global__ void csr_offsets_kernel(int64_t N, int64_t E, const int32_t* __restrict__ recv,
                                   int32_t* __restrict__ off) {
    const int64_t stride = int64_t(gridDim.x) * blockDim.x;
    for (int64_t e = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; e < E; e += stride) {
        const int64_t r = recv[e] < N ? int64_t(recv[e]) : N;
        const int64_t prev = e == 0 ? -1 : int64_t(recv[e - 1]);
        for (int64_t k = (prev + 1 > 0 ? prev + 1 : 0); k <= r; ++k) off[k] = int32_t(e);
        if (e == E - 1)
            for (int64_t k = (r + 1 > 0 ? r + 1 : 0); k <= N; ++k) off[k] = int32_t(E);
    }
}

__global__ void fill_kernel(int32_t* __restrict__ p, int64_t n, int32_t v) {
    const int64_t stride = int64_t(gridDim.x) * blockDim.x;
    for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < n; i += stride) p[i] = v;
}

__global__ void count_senders_kernel(int64_t E, const int32_t* __restrict__ src, int32_t* __restrict__ cnt) {
    const int64_t stride = int64_t(gridDim.x) * blockDim.x;
    for (int64_t e = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; e < E; e += stride)
        atomicAdd(cnt + src[e], 1);
}

// Exclusive scan of cnt[0..N) into off[0..N], one block: each thread scans a contiguous slice.
__global__ void scan_kernel(int64_t N, const int32_t* __restrict__ cnt, int32_t* __restrict__ off) {
    __shared__ int64_t part[1024];
    const int t = threadIdx.x, T = blockDim.x;
    const int64_t per = (N + T - 1) / T;
    const int64_t b = int64_t(t) * per, e = (b + per < N) ? b + per : N;
    int64_t s = 0;
    for (int64_t i = b; i < e; ++i) s += cnt[i];
    part[t] = s;
    __syncthreads();
    if (t == 0) {
        int64_t run = 0;
        for (int i = 0; i < T; ++i) {
            const int64_t v = part[i];
            part[i] = run;
            run += v;
        }
        off[N] = int32_t(run);
    }
    __syncthreads();
    int64_t run = part[t];
    for (int64_t i = b; i < e; ++i) {
        off[i] = int32_t(run);
        run += cnt[i];
    }
}

// Unordered scatter of edge ids into their sender segments (cursor starts at zero).
__global__ void scatter_kernel(int64_t E, const int32_t* __restrict__ src, const int32_t* __restrict__ soff,
                               int32_t* __restrict__ cursor, int32_t* __restrict__ tmp) {
    const int64_t stride = int64_t(gridDim.x) * blockDim.x;
    for (int64_t e = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; e < E; e += stride) {
        const int32_t s = src[e];
        const int32_t pos = atomicAdd(cursor + s, 1);
        tmp[soff[s] + pos] = int32_t(e);
    }
}

__device__ __forceinline__ int32_t receiver_of(int64_t N, const int32_t* __restrict__ roff, int32_t e) {
    // largest r with roff[r] <= e (the receiver whose segment holds e)
    int64_t lo = 0, hi = N - 1;
    while (lo < hi) {
        const int64_t mid = (lo + hi + 1) >> 1;
        if (roff[mid] <= e) lo = mid;
        else hi = mid - 1;
    }
    return int32_t(lo);
}

// Sender segments up to this many edges are ordered by rank counting (each entry counts the
// smaller ids of its segment: d^2 comparisons, cheap for the usual degrees); longer segments
// (hub senders) are sorted in place by sort_segments_kernel instead, O(d log^2 d).
constexpr int32_t kRankMax = 64;

// Place each unordered entry of a short segment at its rank (edge ids are distinct, so the rank
// is unique): the result lists each sender's edges in ascending edge id.  Entries of long
// segments are copied unordered, to be sorted next.
__global__ void rank_place_kernel(int64_t E, const int32_t* __restrict__ src, const int32_t* __restrict__ soff,
                                  const int32_t* __restrict__ tmp, int32_t* __restrict__ eids) {
    const int64_t stride = int64_t(gridDim.x) * blockDim.x;
    for (int64_t k = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; k < E; k += stride) {
        const int32_t e = tmp[k];
        const int32_t s = src[e];
        const int32_t b = soff[s], t = soff[s + 1];
        if (t - b > kRankMax) {
            eids[k] = e;
            continue;
        }
        int32_t rank = 0;
        for (int32_t j = b; j < t; ++j) rank += tmp[j] < e;
        eids[b + rank] = e;
    }
}

// Ascending sort of every segment longer than kRankMax, one block per segment (blocks stride
// over the senders).  Bitonic network in the form whose comparators all put the smaller value
// at the lower index (the first step of each merge compares i with its mirror in the block of
// size k), so the segment behaves as if padded with +infinity up to the next power of two and
// comparators that reach past its end do nothing.
__global__ void sort_segments_kernel(int64_t N, const int32_t* __restrict__ soff, int32_t* __restrict__ eids) {
    for (int64_t s = blockIdx.x; s < N; s += gridDim.x) {
        const int32_t b = soff[s], d = soff[s + 1] - b;
        if (d <= kRankMax) continue;
        int32_t* a = eids + b;
        int32_t n2 = 1;
        while (n2 < d) n2 <<= 1;
        for (int32_t k = 2; k <= n2; k <<= 1) {
            for (int32_t j = k >> 1; j > 0; j >>= 1) {
                __syncthreads();
                // n2 / 2 comparators per step, each on one pair (lo < hi)
                for (int32_t t = threadIdx.x; t < (n2 >> 1); t += blockDim.x) {
                    const int32_t lo = (t / j) * (2 * j) + (t % j);
                    const int32_t hi = (j == (k >> 1)) ? ((lo / k) * k + (k - 1 - (lo % k))) : lo + j;
                    if (hi < d) {
                        const int32_t x = a[lo], y = a[hi];
                        if (y < x) {
                            a[lo] = y;
                            a[hi] = x;
                        }
                    }
                }
            }
        }
        __syncthreads();
    }
}

// send_recv[k] = receiver of send_eids[k], by binary search in the receiver CSR.
__global__ void send_recv_kernel(int64_t N, int64_t E, const int32_t* __restrict__ roff,
                                 const int32_t* __restrict__ eids, int32_t* __restrict__ srecv) {
    const int64_t stride = int64_t(gridDim.x) * blockDim.x;
    for (int64_t k = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; k < E; k += stride)
        srecv[k] = receiver_of(N, roff, eids[k]);
}

__global__ void validate_kernel(int64_t N, int64_t E, const int32_t* __restrict__ off,
                                const int32_t* __restrict__ src, unsigned long long* bad) {
    const int64_t stride = int64_t(gridDim.x) * blockDim.x;
    unsigned long long local = 0;
    const int64_t n = N + 1 > E ? N + 1 : E;
    for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < n; i += stride) {
        if (i <= N) {
            if (i == 0 && off[0] != 0) ++local;
            if (i == N && off[N] != E) ++local;
            if (i < N && off[i + 1] < off[i]) ++local;
        }
        if (i < E && (src[i] < 0 || src[i] >= N)) ++local;
    }
    if (local) atomicAdd(bad, local);
}

}  // namespace

size_t transpose_workspace_bytes(int64_t N, int64_t E) {
    const size_t a = (size_t(N + 1) * 4 + 255) / 256 * 256;
    const size_t b = (size_t(E > 0 ? E : 1) * 4 + 255) / 256 * 256;
    return a + b;
}

cudaError_t launch_csr_offsets(int64_t N, int64_t E, const int32_t* recv, int32_t* off, cudaStream_t st) {
    if (E == 0) {
        fill_kernel<<<grid_for(N + 1), kThreads, 0, st>>>(off, N + 1, 0);
    } else {
        csr_offsets_kernel<<<grid_for(E), kThreads, 0, st>>>(N, E, recv, off);
    }
    return cudaGetLastError();
}

cudaError_t launch_csr_transpose(int64_t N, int64_t E, const int32_t* roff, const int32_t* src,
                                 int32_t* soff, int32_t* eids, int32_t* srecv, void* ws, cudaStream_t st) {
    int32_t* cnt = static_cast<int32_t*>(ws);
    int32_t* tmp = reinterpret_cast<int32_t*>(static_cast<char*>(ws) + (size_t(N + 1) * 4 + 255) / 256 * 256);
    fill_kernel<<<grid_for(N + 1), kThreads, 0, st>>>(cnt, N + 1, 0);
    if (E > 0) count_senders_kernel<<<grid_for(E), kThreads, 0, st>>>(E, src, cnt);
    scan_kernel<<<1, 1024, 0, st>>>(N, cnt, soff);
    if (E > 0) {
        fill_kernel<<<grid_for(N + 1), kThreads, 0, st>>>(cnt, N + 1, 0);
        scatter_kernel<<<grid_for(E), kThreads, 0, st>>>(E, src, soff, cnt, tmp);
        rank_place_kernel<<<grid_for(E), kThreads, 0, st>>>(E, src, soff, tmp, eids);
        sort_segments_kernel<<<152 * 4, 512, 0, st>>>(N, soff, eids);
        send_recv_kernel<<<grid_for(E), kThreads, 0, st>>>(N, E, roff, eids, srecv);
    }
    return cudaGetLastError();
}

cudaError_t launch_graph_validate(int64_t N, int64_t E, const int32_t* off, const int32_t* src,
                                  unsigned long long* bad, cudaStream_t st) {
    cudaError_t e = cudaMemsetAsync(bad, 0, sizeof(unsigned long long), st);
    if (e != cudaSuccess) return e;
    const int64_t n = N + 1 > E ? N + 1 : E;
    validate_kernel<<<grid_for(n), kThreads, 0, st>>>(N, E, off, src, bad);
    return cudaGetLastError();
}

}  // namespace uvu

// ---------------------------------------------------------------------------------------------
// Allocation-free transpose.  Some callers cannot hand this library a workspace: a plugin whose
// host runtime owns every byte of device memory and only passes it input and output buffers, or
// a latency-critical path that must not take an allocator lock or risk an out-of-memory failure
// in the middle of a run.  For them the transpose's scratch (per-sender counters plus the
// unordered edge list) lives in one fixed array compiled into the library.  The array exists on
// every GPU that loads the library for as long as the process runs.  Each call re-initialises
// what it reads (the counters are zeroed and the edge list is fully rewritten), so the contents
// left by the previous call do not matter; calls whose work overlaps on the GPU share the array
// and therefore race.
namespace uvu {
namespace {

constexpr size_t kNoAllocScratchBytes = size_t(16) << 20;  // 16 MiB
static __device__ __align__(256) unsigned char uvu_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_noalloc_mu;
std::map<int, void*> g_noalloc_ptr;  // device ordinal -> address found by the last lookup there

// The array's device address on the current device.  In host code `uvu_noalloc_scratch` names a
// host-side stand-in, so the address must come from the runtime (cudaGetSymbolAddress, with that
// device current, its return code checked).  The lookup is repeated on every call made outside
// stream capture, so a context torn down and recreated in between (cudaDeviceReset, a new primary
// context) never leaves a stale address behind.  While `stream` is capturing, the lookup (which
// may load the library's module) is not made: the address found by the last call on this device
// is used, and a capture before any call on the device is refused.
uvu_status noalloc_scratch(cudaStream_t stream, void** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    e = cudaStreamIsCapturing(stream, &cap);
    if (e != cudaSuccess) return cuda_fail(e, "cudaStreamIsCapturing");
    std::lock_guard<std::mutex> g(g_noalloc_mu);
    if (cap != cudaStreamCaptureStatusNone) {
        auto it = g_noalloc_ptr.find(dev);
        if (it == g_noalloc_ptr.end())
            return fail(UVU_ERR_INVALID_ARGUMENT,
                        "uvu_csr_transpose_noalloc: the first call on a device must come before stream capture");
        *out = it->second;
        return UVU_OK;
    }
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, uvu_noalloc_scratch);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(uvu_noalloc_scratch)");
    g_noalloc_ptr[dev] = p;
    *out = p;
    return UVU_OK;
}

}  // namespace
}  // namespace uvu

extern "C" uvu_status uvu_csr_transpose_noalloc(int64_t n_nodes, int64_t n_edges, const int32_t* recv_offsets,
                                                const int32_t* src, int32_t* send_offsets, int32_t* send_eids,
                                                int32_t* send_recv, uvu_stream_t stream) {
    using namespace uvu;
    if (n_nodes < 0 || n_edges < 0 || n_nodes >= INT32_MAX || n_edges >= INT32_MAX)
        return fail(UVU_ERR_INVALID_ARGUMENT, "n_nodes and n_edges must be in [0, 2^31 - 1)");
    if (!send_offsets) return fail(UVU_ERR_INVALID_ARGUMENT, "send_offsets is NULL");
    if (n_edges > 0 && (!recv_offsets || !src || !send_eids || !send_recv))
        return fail(UVU_ERR_INVALID_ARGUMENT, "graph pointer is NULL");
    const size_t need = transpose_workspace_bytes(n_nodes, n_edges);
    if (need > kNoAllocScratchBytes)
        return fail(UVU_ERR_UNSUPPORTED,
                    "graph needs " + std::to_string(need) + " bytes of transpose scratch; the built-in scratch holds " +
                        std::to_string(kNoAllocScratchBytes) + " bytes (4(N+1) + 4E rounded up); use uvu_csr_transpose "
                        "with a caller workspace");
    void* ws = nullptr;
    uvu_status s = noalloc_scratch(reinterpret_cast<cudaStream_t>(stream), &ws);
    if (s != UVU_OK) return s;
    cudaError_t e = launch_csr_transpose(n_nodes, n_edges, recv_offsets, src, send_offsets, send_eids, send_recv,
                                         ws, stream);
    if (e != cudaSuccess) return cuda_fail(e, "csr transpose launch");
    return ok();
}
