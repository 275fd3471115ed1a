// Dense fp32 products on the 5th-generation tensor cores (tcgen05) with fp32 accuracy.
//
// The dense contractions next to the convolution -- the channel mixing that reduces a factorised
// UVW convolution to the UVU one, and the last linear layer of the radial network (with its two
// gradients) -- are ordinary matrix products.  A single TF32 product keeps 11 significant bits,
// far outside the fp32 tolerance, so each operand is split as x = hi + lo with hi = x rounded to
// TF32 and lo = (x - hi) rounded to TF32 (|lo| <= 2^-11 |x|, so hi + lo holds x to about 2^-22),
// and the product is accumulated as hi*hi + hi*lo + lo*hi ("3xTF32"; the dropped lo*lo term is
// below 2^-22 of each product).  Accumulation is fp32 in tensor memory.
//
// One CTA computes one 128 x BN tile of C (BN = 128 or 64): 8 warps load 16-wide K chunks of A
// and B from global memory (16-byte loads, the next chunk in flight while the current one is
// stored), split them and store hi and lo parts into shared memory in the canonical K-major
// no-swizzle layout of the MMA (8-row x 16-byte core matrices); one thread issues the MMAs
// (M = 128, N = BN, K = 8 per instruction) and commits them to the stage's mbarrier, which frees
// the stage three chunks later.  The accumulator lives in tensor memory.  Measured on GB300: an
// accumulation there loses more than a round-to-nearest fp32 add (a 35,000-term reduction was off
// by 3e-3 where fp32 sums in registers stay near 1e-4), so long K is split over up to eight
// accumulators of at most 256 K each, added in registers by the epilogue in a fixed order, and
// sums over tens of thousands of rows are left to compensated CUDA-core kernels.  The epilogue
// reads the accumulators with tcgen05.ld, each warp 32 lanes (rows) x BN/2 columns.  Every
// mbarrier wait is bounded (about two seconds on the global timer); on expiry the CTA sets
// tc_status_word, skips its remaining work, frees its tensor memory and returns.
//
//   C[row][n] = sum_k A[row][k] B_s[k][n] over the rows of each segment s (A row-major, K
//   contiguous; B_s = B + s * b_seg_stride, either n- or k-contiguous).
#include <cuda_runtime.h>

#include <cstdint>

#include "plan.h"
#include "tcgemm.h"

namespace uvu {
namespace {

constexpr int kThreads = 256;
constexpr int kBM = 128, kBNmax = 128, kBK = 16, kNST = 3;
constexpr int kSBO = 528;                       // bytes between 8-row core-matrix groups (512 + 16)
constexpr int kTileBytes = 16 * kSBO;           // one 128-row x 16-k operand tile
constexpr int kStageBytes = 4 * kTileBytes;     // A hi, A lo, B hi, B lo
constexpr int kBarOff = kNST * kStageBytes;
constexpr int kSmemBytes = kBarOff + 8 * kNST + 16;

__device__ unsigned int tc_status_word;

__device__ __forceinline__ uint32_t smem_u32(const void* p) { return uint32_t(__cvta_generic_to_shared(p)); }

__device__ __forceinline__ uint32_t tf32_rna(float x) {
    uint32_t r;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
    return r;
}
// x = hi + lo, both representable in TF32
__device__ __forceinline__ void split3(float x, uint32_t& hi, uint32_t& lo) {
    hi = tf32_rna(x);
    lo = tf32_rna(x - __uint_as_float(hi));
}

// byte offset of element (row, k) of an operand tile in the K-major no-swizzle layout
__device__ __forceinline__ uint32_t toff(int row, int k) {
    return uint32_t((row >> 3) * kSBO + (k >> 2) * 128 + (row & 7) * 16 + (k & 3) * 4);
}

// Shared-memory matrix descriptor: start address, leading (K-direction) core-matrix stride 128 B,
// stride (8-row group) 528 B, fixed version bits 0b001 at 46, no swizzle.
__device__ __forceinline__ uint64_t sdesc(uint32_t addr) {
    return uint64_t((addr >> 4) & 0x3FFFu) | (uint64_t(128 >> 4) << 16) | (uint64_t(kSBO >> 4) << 32) | (1ull << 46);
}

// Instruction descriptor of kind::tf32: D fp32, A and B TF32, both K-major, M = 128, N = bn.
__device__ __forceinline__ uint32_t idesc(int bn) {
    return (1u << 4) | (2u << 7) | (2u << 10) | (uint32_t(bn >> 3) << 17) | (uint32_t(kBM >> 4) << 24);
}

__device__ __forceinline__ void mma_tf32(uint32_t d, uint64_t a, uint64_t b, uint32_t id, uint32_t accum) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %3, 0;\n"
        " tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %4, p;\n}\n" ::"r"(d),
        "l"(a), "l"(b), "r"(accum), "r"(id)
        : "memory");
}

__device__ __forceinline__ void mbar_init(uint32_t b) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(b) : "memory");
}
__device__ __forceinline__ bool mbar_test(uint32_t b, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}"
        : "=r"(ok)
        : "r"(b), "r"(parity)
        : "memory");
    return ok != 0;
}
__device__ __forceinline__ unsigned long long gtimer() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
// Bounded wait: false (and the status bit set) after about two seconds.
__device__ __noinline__ bool mbar_wait(uint32_t b, uint32_t parity) {
    if (mbar_test(b, parity)) return true;
    const unsigned long long t0 = gtimer();
    for (;;) {
        for (int i = 0; i < 64; ++i)
            if (mbar_test(b, parity)) return true;
        if (gtimer() - t0 > 2000000000ull) {
            atomicOr(&tc_status_word, 1u);
            return false;
        }
    }
}

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
          "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

}  // namespace

namespace {

// Loads of one 16-wide K chunk into registers: two 16-byte vectors of A and two of B per thread.
// Element (r, k) of the A tile and (n, k) of the B tile, as 4-vectors along the contiguous
// dimension; masked entries read as zero.
struct Chunk {
    float4 a[2], b[2];
};

// Product mode, A: row = idx >> 2 (128 rows), k = (idx & 3) * 4 (16 k), contiguous in k.
__device__ __forceinline__ float4 ld4(const float* p, bool ok) {
    return ok ? __ldg(reinterpret_cast<const float4*>(p)) : make_float4(0.f, 0.f, 0.f, 0.f);
}

__device__ __forceinline__ void store_k4(unsigned char* tile_hi, unsigned char* tile_lo, int row, int k, float4 v) {
    uint32_t h0, l0, h1, l1, h2, l2, h3, l3;
    split3(v.x, h0, l0);
    split3(v.y, h1, l1);
    split3(v.z, h2, l2);
    split3(v.w, h3, l3);
    const uint32_t o = toff(row, k);
    *reinterpret_cast<uint4*>(tile_hi + o) = make_uint4(h0, h1, h2, h3);
    *reinterpret_cast<uint4*>(tile_lo + o) = make_uint4(l0, l1, l2, l3);
}
// four consecutive rows (row .. row + 3) at one k
__device__ __forceinline__ void store_r4(unsigned char* tile_hi, unsigned char* tile_lo, int row, int k, float4 v) {
    const float e[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        uint32_t h, l;
        split3(e[i], h, l);
        const uint32_t o = toff(row + i, k);
        *reinterpret_cast<uint32_t*>(tile_hi + o) = h;
        *reinterpret_cast<uint32_t*>(tile_lo + o) = l;
    }
}

__global__ void __launch_bounds__(kThreads, 2) tc_gemm_kernel(TcJobs J) {
    extern __shared__ __align__(1024) unsigned char smem[];
    const int tid = threadIdx.x, warp = tid >> 5;
    const uint32_t sbase = smem_u32(smem);
    uint32_t* tslot = reinterpret_cast<uint32_t*>(smem + kBarOff + 8 * kNST);
    const int bn = J.bn;

    // ---- the tile: segment, rows [m0, min(m0 + 128, rend)), columns [n0, n0 + bn)
    int seg = 0;
    const int t = int(blockIdx.x);
    while (seg + 1 < J.nseg && t >= J.tile0[seg + 1]) ++seg;
    const long long m0 = J.row0[seg] + (long long)(t - J.tile0[seg]) * kBM;
    const long long rend = J.row0[seg] + J.rows[seg];
    const int n0 = int(blockIdx.y) * bn;
    const int K = J.K;

    if (tid == 0) {
        for (int i = 0; i < kNST; ++i) mbar_init(sbase + kBarOff + 8 * i);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tslot)),
                     "r"(J.tmem_cols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(tslot);

    const int nk = (K + kBK - 1) / kBK;
    const int kacc_chunks = J.kacc / kBK;  // K chunks per accumulator
    const float* Bs = J.B + (long long)seg * J.b_seg_stride;

    auto load = [&](int i, Chunk& c) {
        const int k0 = i * kBK;
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            const int idx = tid + kThreads * j;
            // A: 128 rows x 16 k, 4-vectors along k
            const int r = idx >> 2, kq = (idx & 3) * 4;
            const long long row = m0 + r;
            c.a[j] = ld4(J.A + row * J.lda + (k0 + kq), row < rend && k0 + kq < K);
            if (J.b_kcont) {  // B_s[k][n], k contiguous: 128 n x 16 k, 4-vectors along k
                const int n = idx >> 2;
                c.b[j] = ld4(Bs + (long long)(n0 + n) * J.sbn + (k0 + kq), n < bn && n0 + n < J.N && k0 + kq < K);
            } else {  // n contiguous: 16 k x 128 n, 4-vectors along n
                const int kk = idx >> 5, nq = (idx & 31) * 4;
                c.b[j] = ld4(Bs + (long long)(k0 + kk) * J.sbk + (n0 + nq), k0 + kk < K && nq < bn && n0 + nq < J.N);
            }
        }
    };
    auto store = [&](int s, const Chunk& c) {
        unsigned char* st = smem + s * kStageBytes;
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            const int idx = tid + kThreads * j;
            store_k4(st, st + kTileBytes, idx >> 2, (idx & 3) * 4, c.a[j]);
            if (J.b_kcont) store_k4(st + 2 * kTileBytes, st + 3 * kTileBytes, idx >> 2, (idx & 3) * 4, c.b[j]);
            else store_r4(st + 2 * kTileBytes, st + 3 * kTileBytes, (idx & 31) * 4, idx >> 5, c.b[j]);
        }
    };

    // A timed-out wait is combined over the block by the barrier itself (__syncthreads_or), so
    // every thread takes the same exit.
    bool dead = false;
    const uint32_t id = idesc(bn);
    Chunk cur, nxt;
    if (nk > 0) load(0, cur);
    for (int i = 0; i < nk; ++i) {
        if (i + 1 < nk) load(i + 1, nxt);
        const int s = i % kNST;
        const bool late = i >= kNST && !mbar_wait(sbase + kBarOff + 8 * s, uint32_t((i / kNST) - 1) & 1u);
        store(s, cur);
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        if (__syncthreads_or(late)) {
            dead = true;
            break;
        }
        if (tid == 0) {
            asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
            const uint32_t st = sbase + s * kStageBytes;
            const int acc = i / kacc_chunks;          // accumulator of this chunk
            const bool fresh = i % kacc_chunks == 0;  // its first chunk
            const uint32_t d = tmem + uint32_t(acc * bn);
#pragma unroll
            for (int ks = 0; ks < kBK / 8; ++ks) {
                const uint32_t ko = ks * 256;  // two 16-byte core-matrix columns per K = 8 step
                const uint64_t ah = sdesc(st + ko), al = sdesc(st + kTileBytes + ko);
                const uint64_t bh = sdesc(st + 2 * kTileBytes + ko), bl = sdesc(st + 3 * kTileBytes + ko);
                mma_tf32(d, al, bh, id, (fresh && ks == 0) ? 0u : 1u);
                mma_tf32(d, ah, bl, id, 1u);
                mma_tf32(d, ah, bh, id, 1u);
            }
            asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                             sbase + kBarOff + 8 * s)
                         : "memory");
        }
        cur = nxt;
    }
    bool late = false;
    if (nk > 0 && !dead) {
        const int l = nk - 1;
        late = !mbar_wait(sbase + kBarOff + 8 * (l % kNST), uint32_t(l / kNST) & 1u);
    }
    dead = __syncthreads_or(late || dead) != 0;
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");

    // ---- epilogue: warp w reads lanes 32 (w % 4) .. + 31 and columns (w / 4) bn/2 .. + bn/2 - 1
    // of every accumulator and adds them in accumulator order
    if (!dead) {
        const int nacc = nk > 0 ? (nk + kacc_chunks - 1) / kacc_chunks : 0;
        const int lane_row = (warp & 3) * 32 + (tid & 31);
        const int half = bn / 2;
        const int cbase = (warp >> 2) * half;
        const long long row = m0 + lane_row;
#pragma unroll 1
        for (int cc = 0; cc < half; cc += 16) {
            float v[16];
#pragma unroll
            for (int q = 0; q < 16; ++q) v[q] = 0.f;
#pragma unroll 1
            for (int a = 0; a < nacc; ++a) {
                uint32_t r[16];
                tmem_ld16(tmem + (uint32_t((warp & 3) * 32) << 16) + uint32_t(a * bn + cbase + cc), r);
#pragma unroll
                for (int q = 0; q < 16; ++q) v[q] += __uint_as_float(r[q]);
            }
            const int c0 = n0 + cbase + cc;
            if (row < rend) {
                float* out = J.C + row * J.ldc + c0;
                if (c0 + 16 <= J.N) {
#pragma unroll
                    for (int q = 0; q < 16; q += 4) *reinterpret_cast<float4*>(out + q) = make_float4(v[q], v[q + 1], v[q + 2], v[q + 3]);
                } else {
#pragma unroll
                    for (int q = 0; q < 16; ++q)
                        if (c0 + q < J.N) out[q] = v[q];
                }
            }
        }
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    if (warp == 0)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(J.tmem_cols) : "memory");
}

}  // namespace

// Tile shape of a product: N tiles of 128 columns (64 when N <= 64), K split over accumulators
// of at most kKacc K each (at most 8, so that accumulators x BN columns fit the tensor memory of
// two resident CTAs per SM: 256 columns each, or one CTA with 512).
namespace {
constexpr int kKacc = 256;
int pow2_cols(int c) {
    int p = 32;
    while (p < c) p <<= 1;
    return p;
}
}  // namespace

bool tc_gemm_configure(TcJobs& J) {
    J.bn = J.N <= 64 ? 64 : kBNmax;
    const int nk = (J.K + kBK - 1) / kBK;
    int nacc = (J.K + kKacc - 1) / kKacc;
    if (nacc < 1) nacc = 1;
    const int per = (nk + nacc - 1) / nacc;  // chunks per accumulator
    J.kacc = per * kBK;
    nacc = (nk + per - 1) / per;
    J.tmem_cols = pow2_cols(nacc * J.bn);
    return J.tmem_cols <= 512;
}

// Requirements of the tensor-core path: 16-byte aligned base pointers and row strides that keep
// every row 16-byte aligned (the loads are 4-vectors); widths that are multiples of 4; K small
// enough that its accumulators fit the tensor memory.
bool tc_gemm_supported(const TcJobs& J) {
    auto al = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
    if (!al(J.A) || !al(J.B) || !al(J.C) || J.nseg < 1 || J.nseg > kTcMaxSeg || J.N % 4 || J.N < 1) return false;
    if (J.K < 1 || J.K % 4 || J.lda % 4 || J.ldc % 4 || J.b_seg_stride % 4) return false;
    if (J.b_kcont ? (J.sbk != 1 || J.sbn % 4) : (J.sbn != 1 || J.sbk % 4)) return false;
    TcJobs T = J;
    return tc_gemm_configure(T);
}

cudaError_t launch_tc_gemm(TcJobs& J, cudaStream_t st) {
    static bool configured = false;  // the attribute is per function, not per call
    if (!configured) {
        cudaError_t e = cudaFuncSetAttribute(tc_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
        if (e != cudaSuccess) return e;
        configured = true;
    }
    if (!tc_gemm_configure(J)) return cudaErrorInvalidValue;
    long long t = 0;
    for (int s = 0; s < J.nseg; ++s) {
        J.tile0[s] = int(t);
        t += (J.rows[s] + kBM - 1) / kBM;
    }
    J.tile0[J.nseg] = int(t);
    if (t == 0) return cudaSuccess;
    if (t > 0x7FFFFFFF) return cudaErrorInvalidConfiguration;
    const int ntn = (J.N + J.bn - 1) / J.bn;
    tc_gemm_kernel<<<dim3(unsigned(t), unsigned(ntn), 1), kThreads, kSmemBytes, st>>>(J);
    return cudaGetLastError();
}

// Device status of the tensor-core kernels (bit 0: a bounded wait gave up); reset clears it.
cudaError_t tc_status(unsigned* word, bool reset) {
    cudaError_t e = cudaMemcpyFromSymbol(word, tc_status_word, sizeof(unsigned));
    if (e != cudaSuccess || !reset) return e;
    const unsigned z = 0;
    return cudaMemcpyToSymbol(tc_status_word, &z, sizeof(unsigned));
}

}  // namespace uvu
