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
// Persistent kernel, one CTA per SM looping over 128 x BN tiles of C (BN = 128, or 64 when N <= 64
// or K spans several ranges), with warp roles.  Eight producer warps load 16-wide K chunks of A
// and B from global memory (three chunks in flight per thread), split them and store the hi and
// lo parts into a ring of four shared-memory stages in the canonical K-major no-swizzle layout of
// the MMA (8-row x 16-byte core matrices); one thread of a ninth warp issues the MMAs (M = 128,
// N = BN, K = 8 per instruction) into one of two tensor-memory accumulators and commits each
// stage back to its producers; four epilogue warps read the finished accumulator with
// tcgen05.ld (one tile row per thread) and store it while the MMAs fill the other one.
// Measured on GB300: an accumulation in tensor memory loses more than a round-to-nearest fp32
// add (a 35,000-term reduction was off by 3e-3 where fp32 sums in registers stay near 1e-4), so
// long K is summed in ranges of at most 256, each accumulated afresh and added into fp32
// registers by the epilogue, and sums over tens of thousands of rows are left to compensated
// CUDA-core kernels.  Every mbarrier wait is bounded (about two seconds on the global timer); on
// expiry the role sets a shared flag and the tc_status_word bit, every role leaves its loop, and
// the CTA frees its tensor memory and returns.
//
//   C[row][n] = sum_k A[row][k] B_s[k][n] over the rows of each segment s (A row-major, K
//   contiguous; B_s = B + s * b_seg_stride, either n- or k-contiguous).
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>

#include "plan.h"
#include "tcgemm.h"

namespace uvu {
namespace {

constexpr int kBM = 128, kBNmax = 128, kBK = 16;
constexpr int kSBO = 528;                       // bytes between 8-row core-matrix groups (512 + 16)
constexpr int kTileBytes = 16 * kSBO;           // one 128-row x 16-k operand tile
constexpr int kStageBytes = 4 * kTileBytes;     // A hi, A lo, B hi, B lo
constexpr int kTcBTile = 2 * kTileBytes;        // a pre-split B chunk: hi tile, then lo tile

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


}  // namespace

namespace {

// Loads of one 16-wide K chunk of A into registers: two 16-byte vectors per thread (masked
// entries read as zero).
struct Chunk {
    float4 a[2];
};

__device__ __forceinline__ float4 ld4(const float* p, bool ok) {
    return ok ? __ldg(reinterpret_cast<const float4*>(p)) : make_float4(0.f, 0.f, 0.f, 0.f);
}

// four consecutive k of one row, as hi and lo TF32 parts, one 16-byte store each
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

// Warp roles of the persistent kernel (13 warps): 0-7 load and split the operand chunks into the
// stage ring; 8-11 drain the accumulators (warp w reads TMEM lanes 32 (w % 4) .. + 31, i.e. one
// row of the tile per thread); 12 issues the MMAs (one thread).
constexpr int kProdWarps = 8, kEpiWarp0 = 8, kMmaWarp = 12;
constexpr int kThreadsP = 13 * 32;
constexpr int kStages = 4;
constexpr int kStagesBytes = kStages * kStageBytes;
// barriers after the stages: full[kStages], empty[kStages], accfull[2], accempty[2], tmem slot
constexpr int kBarFull = kStagesBytes, kBarEmpty = kBarFull + 8 * kStages, kBarAccF = kBarEmpty + 8 * kStages,
              kBarAccE = kBarAccF + 16, kTslot = kBarAccE + 16;
// output staging of the epilogue warps: 32 rows x (BN + 4) floats each (the pad keeps the rows'
// 16-byte writes in distinct banks); rows leave as one bulk copy each
constexpr int kStgPitch = kBNmax + 4;
constexpr int kStage0 = (kTslot + 16 + 127) / 128 * 128;
constexpr int kSmemP = kStage0 + 4 * 32 * kStgPitch * 4;

__device__ __forceinline__ void mbar_init_n(uint32_t b, uint32_t n) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(b), "r"(n) : "memory");
}
__device__ __forceinline__ void mbar_arrive1(uint32_t b) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(b) : "memory");
}
__device__ __forceinline__ void tmem_ld16_nw(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
          "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
}
__device__ __forceinline__ void tmem_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void mbar_expect_tx_only(uint32_t b, uint32_t bytes) {
    asm volatile("mbarrier.expect_tx.shared::cta.b64 [%0], %1;" ::"r"(b), "r"(bytes) : "memory");
}
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
                 "l"(src), "r"(bytes), "r"(bar)
                 : "memory");
}
__device__ __forceinline__ void tc_commit(uint32_t b) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(b) : "memory");
}

__global__ void __maxnreg__(128) tc_gemm_kernel(TcJobs J) {  // 13 warps: 4 share one SM sub-partition's 16K registers
    extern __shared__ __align__(1024) unsigned char smem[];
    __shared__ int s_dead;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t sbase = smem_u32(smem);
    uint32_t* tslot = reinterpret_cast<uint32_t*>(smem + kTslot);
    const int bn = J.bn, K = J.K;
    const int nk = (K + kBK - 1) / kBK;   // K chunks per tile
    const int cpr = J.kacc / kBK;         // K chunks per accumulation range
    const int nr = (nk + cpr - 1) / cpr;  // ranges per tile
    const int ntn = (J.N + bn - 1) / bn;
    const int T = J.tile0[J.nseg] * ntn;  // tiles (< 2^31, checked by the launcher)
    const int my_tiles = T > int(blockIdx.x) ? (T - 1 - int(blockIdx.x)) / int(gridDim.x) + 1 : 0;

    if (tid == 0) {
        s_dead = 0;
        for (int i = 0; i < kStages; ++i) {
            mbar_init_n(sbase + kBarFull + 8 * i, kProdWarps);
            mbar_init_n(sbase + kBarEmpty + 8 * i, 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init_n(sbase + kBarAccF + 8 * i, 1);
            mbar_init_n(sbase + kBarAccE + 8 * i, 4);
        }
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
    volatile int* dead = &s_dead;
    // the shared flag read warp-uniformly (every lane of the warp takes the same branch)
    auto wdead = [&]() { return __any_sync(0xffffffffu, *dead != 0); };

    // tile number (within this CTA's sequence) -> segment, first row, row end, first column; tile
    // counts fit 32 bits (the launcher checks), and the callers advance tile by tile
    auto tile_of = [&](int lt, int& seg, long long& m0, long long& rend, int& n0) {
        const int t = int(blockIdx.x) + lt * int(gridDim.x);
        const int rt = t / ntn;
        n0 = (t - rt * ntn) * bn;
        seg = 0;
        while (seg + 1 < J.nseg && rt >= J.tile0[seg + 1]) ++seg;
        m0 = J.row0[seg] + (long long)(rt - J.tile0[seg]) * kBM;
        rend = J.row0[seg] + J.rows[seg];
    };

    if (warp < kProdWarps) {
        // ---------------------------------------------------------------- producers
        // Chunks in order (tile by tile, K chunks within a tile); the load cursor runs five chunks
        // ahead of the store cursor (a ring of six register buffers), both advanced incrementally.
        // Lane 0 of warp 0 also brings the chunk's pre-split B tile into the stage by one bulk
        // copy, counted on the stage's "full" barrier with the eight warps' arrivals.
        const int C = my_tiles * nk;  // chunks of this CTA
        const int ptid = tid;         // 0 .. 255
        int l_lt = 0, l_kc = 0, l_seg = 0, l_n0 = 0;
        long long l_m0 = 0, l_rend = 0;
        if (my_tiles > 0) tile_of(0, l_seg, l_m0, l_rend, l_n0);
        auto load_next = [&](Chunk& ch) {
            if (l_lt >= my_tiles) return;
            const int k0 = l_kc * kBK;
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                // a quarter-warp covers 8 rows at one k group: its 16-byte stores fill one core
                // matrix (conflict-free), and each row's 64 bytes are read by 4 lanes of the warp
                const int idx = ptid + 256 * j;
                const int r = ((idx >> 5) << 3) | (idx & 7), kq = ((idx >> 3) & 3) * 4;
                const long long row = l_m0 + r;
                ch.a[j] = ld4(J.A + row * J.lda + (k0 + kq), row < l_rend && k0 + kq < K);
            }
            if (++l_kc == nk) {
                l_kc = 0;
                if (++l_lt < my_tiles) tile_of(l_lt, l_seg, l_m0, l_rend, l_n0);
            }
        };
        // store cursor: the B tile of the chunk being stored
        int s_lt = 0, s_kc = 0, s_seg = 0, s_n0 = 0;
        long long s_m0 = 0, s_rend = 0;
        if (my_tiles > 0) tile_of(0, s_seg, s_m0, s_rend, s_n0);
        int s = 0;
        uint32_t ph = 0;  // use count of stage s, mod 2 (the parity its "empty" barrier completes)
        auto step = [&](int c, Chunk& cur, Chunk& fut) {
            if (c >= C || wdead()) return;
            load_next(fut);
            if (c >= kStages && !__all_sync(0xffffffffu, mbar_wait(sbase + kBarEmpty + 8 * s, ph ^ 1u))) {
                *dead = 1;
                return;
            }
            const uint32_t full = sbase + kBarFull + 8 * s;
            if (ptid == 0) {
                const size_t bt = ((size_t(s_seg) * ntn + s_n0 / bn) * nk + s_kc) * size_t(kTcBTile);
                mbar_expect_tx_only(full, kTcBTile);
                bulk_g2s(sbase + s * kStageBytes + 2 * kTileBytes, static_cast<const unsigned char*>(J.bpack) + bt,
                         kTcBTile, full);
            }
            unsigned char* st = smem + s * kStageBytes;
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                const int idx = ptid + 256 * j;
                const int r = ((idx >> 5) << 3) | (idx & 7), kq = ((idx >> 3) & 3) * 4;
                store_k4(st, st + kTileBytes, r, kq, cur.a[j]);
            }
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            __syncwarp();
            if (lane == 0) mbar_arrive1(full);
            if (++s == kStages) {
                s = 0;
                ph ^= 1u;
            }
            if (++s_kc == nk) {
                s_kc = 0;
                if (++s_lt < my_tiles) tile_of(s_lt, s_seg, s_m0, s_rend, s_n0);
            }
        };
        Chunk b0, b1, b2, b3, b4, b5;
        load_next(b0);
        load_next(b1);
        load_next(b2);
        load_next(b3);
        load_next(b4);
        for (int c = 0; c < C && !wdead(); c += 6) {
            step(c, b0, b5);
            step(c + 1, b1, b0);
            step(c + 2, b2, b1);
            step(c + 3, b3, b2);
            step(c + 4, b4, b3);
            step(c + 5, b5, b4);
        }
    } else if (warp == kMmaWarp) {
        // ---------------------------------------------------------------- MMA issue
        if (lane == 0) {
            const uint32_t id = idesc(bn);
            int s = 0, q = 0;
            uint32_t ph = 0;  // parity of the stage's current use
            for (int lt = 0; lt < my_tiles && !*dead; ++lt) {
                for (int r = 0; r < nr && !*dead; ++r, ++q) {
                    const int b = q & 1;
                    const int v = q >> 1;
                    if (v > 0 && !mbar_wait(sbase + kBarAccE + 8 * b, uint32_t(v - 1) & 1u)) {
                        *dead = 1;
                        break;
                    }
                    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
                    const uint32_t d = tmem + uint32_t(b * bn);
                    const int k1 = min(nk, (r + 1) * cpr);
                    for (int kc = r * cpr; kc < k1; ++kc) {
                        if (!mbar_wait(sbase + kBarFull + 8 * s, ph)) {
                            *dead = 1;
                            break;
                        }
                        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
                        const uint32_t st = sbase + s * kStageBytes;
#pragma unroll
                        for (int ks = 0; ks < kBK / 8; ++ks) {
                            const uint32_t ko = ks * 256;
                            const uint64_t ah = sdesc(st + ko), al = sdesc(st + kTileBytes + ko);
                            const uint64_t bh = sdesc(st + 2 * kTileBytes + ko), bl = sdesc(st + 3 * kTileBytes + ko);
                            mma_tf32(d, al, bh, id, (kc == r * cpr && ks == 0) ? 0u : 1u);
                            mma_tf32(d, ah, bl, id, 1u);
                            mma_tf32(d, ah, bh, id, 1u);
                        }
                        tc_commit(sbase + kBarEmpty + 8 * s);  // the stage is free once these MMAs are done
                        if (++s == kStages) {
                            s = 0;
                            ph ^= 1u;
                        }
                    }
                    if (*dead) break;
                    tc_commit(sbase + kBarAccF + 8 * b);  // the range's accumulator is complete
                }
            }
        }
        __syncwarp();
    } else {
        // ---------------------------------------------------------------- epilogue
        // Each thread holds one tile row: 32 columns per TMEM read round (two loads, one wait),
        // added to the running sums of earlier ranges when K spans several, then written into the
        // warp's staging rows; after the last range the warp stores its rows row by row.
        const int ew = warp - kEpiWarp0;  // 0..3 = TMEM lane quadrant
        const uint32_t tl = tmem + (uint32_t(ew * 32) << 16);
        float* stg = reinterpret_cast<float*>(smem + kStage0) + ew * 32 * kStgPitch;
        float* myrow = stg + lane * kStgPitch;
        int q = 0;
        for (int lt = 0; lt < my_tiles && !wdead(); ++lt) {
            int seg, n0;
            long long m0, rend;
            tile_of(lt, seg, m0, rend, n0);
            for (int r = 0; r < nr && !wdead(); ++r, ++q) {
                const int b = q & 1;
                const bool ok = __all_sync(0xffffffffu, mbar_wait(sbase + kBarAccF + 8 * b, uint32_t(q >> 1) & 1u));
                if (!ok) *dead = 1;
                asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
#pragma unroll 1
                for (int cc = 0; cc < bn; cc += 32) {
                    uint32_t v0[16], v1[16];
                    tmem_ld16_nw(tl + uint32_t(b * bn + cc), v0);
                    tmem_ld16_nw(tl + uint32_t(b * bn + cc + 16), v1);
                    tmem_wait();
                    float4* dst = reinterpret_cast<float4*>(myrow + cc);
#pragma unroll
                    for (int x = 0; x < 4; ++x) {
                        float4 a = make_float4(__uint_as_float(v0[4 * x]), __uint_as_float(v0[4 * x + 1]),
                                               __uint_as_float(v0[4 * x + 2]), __uint_as_float(v0[4 * x + 3]));
                        float4 c = make_float4(__uint_as_float(v1[4 * x]), __uint_as_float(v1[4 * x + 1]),
                                               __uint_as_float(v1[4 * x + 2]), __uint_as_float(v1[4 * x + 3]));
                        if (r > 0) {  // later ranges add onto the staged sums (fixed order)
                            const float4 pa = dst[x], pc = dst[4 + x];
                            a = make_float4(pa.x + a.x, pa.y + a.y, pa.z + a.z, pa.w + a.w);
                            c = make_float4(pc.x + c.x, pc.y + c.y, pc.z + c.z, pc.w + c.w);
                        }
                        dst[x] = a;
                        dst[4 + x] = c;
                    }
                }
                asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
                __syncwarp();
                if (lane == 0) mbar_arrive1(sbase + kBarAccE + 8 * b);  // the accumulator may be reused
                if (r == nr - 1 && ok) {
                    // the warp's 32 staged rows leave with coalesced 16-byte stores: one full row per
                    // instruction for BN = 128, two rows for BN = 64
                    __syncwarp();
                    const int w4 = min(bn, J.N - n0) / 4;  // 16-byte groups per row
                    const int lpr = bn / 4;                // lanes per row
                    const int sub = lane / lpr, g = lane - sub * lpr;
                    for (int i = sub; i < 32; i += 32 / lpr) {
                        const long long row = m0 + ew * 32 + i;
                        if (row < rend && g < w4)
                            *reinterpret_cast<float4*>(J.C + row * J.ldc + n0 + 4 * g) =
                                *reinterpret_cast<const float4*>(stg + i * kStgPitch + 4 * g);
                    }
                    __syncwarp();
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

namespace {
// B_s[k][n] (any strides) -> the pre-split tiles of J.bpack: one block per (segment, N tile,
// K chunk), zeros outside [0, K) x [0, N) and beyond BN columns.
__global__ void __launch_bounds__(256) tc_pack_b(TcJobs J, int ntn, int nk) {
    const int kc = blockIdx.x % nk, nt = (blockIdx.x / nk) % ntn, seg = blockIdx.x / (nk * ntn);
    unsigned char* t = static_cast<unsigned char*>(J.bpack) + size_t(blockIdx.x) * kTcBTile;
    const float* Bs = J.B + (long long)seg * J.b_seg_stride;
    const int n0 = nt * J.bn, k0 = kc * kBK;
    for (int e = threadIdx.x; e < 128 * kBK; e += 256) {
        const int n = J.b_kcont ? (e >> 4) : (e & 127), k = J.b_kcont ? (e & 15) : (e >> 7);
        float v = 0.f;
        if (n < J.bn && n0 + n < J.N && k0 + k < J.K) v = Bs[(long long)(k0 + k) * J.sbk + (long long)(n0 + n) * J.sbn];
        uint32_t h, l;
        split3(v, h, l);
        const uint32_t o = toff(n, k);
        *reinterpret_cast<uint32_t*>(t + o) = h;
        *reinterpret_cast<uint32_t*>(t + kTileBytes + o) = l;
    }
}
}  // namespace

// Tile shape of a product: N tiles of 128 columns (64 when N <= 64, or when K spans several
// ranges, whose sums then fit the registers), K summed in ranges of at most kKacc.
namespace {
constexpr int kKacc = 256;
}  // namespace

bool tc_gemm_configure(TcJobs& J) {
    const int nk = (J.K + kBK - 1) / kBK;
    const int nr = (J.K + kKacc - 1) / kKacc;  // ranges
    const int per = (nk + nr - 1) / nr;        // chunks per range
    J.kacc = per * kBK;
    J.bn = (J.N <= 64 || nr > 1) ? 64 : kBNmax;
    J.tmem_cols = 2 * J.bn;  // two accumulators: the MMAs fill one while the epilogue drains the other
    return true;
}

// Requirements of the tensor-core path: 16-byte aligned base pointers and row strides that keep
// every row 16-byte aligned (the loads are 4-vectors); widths that are multiples of 4; K small
// enough that its accumulators fit the tensor memory.
bool tc_gemm_supported(const TcJobs& J) {
    auto al = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
    if (!al(J.A) || !al(J.C) || !J.B || !J.bpack || !al(J.bpack) || J.nseg < 1 || J.nseg > kTcMaxSeg || J.N % 4 || J.N < 1)
        return false;
    if (J.K < 1 || J.K % 4 || J.lda % 4 || J.ldc % 4 || J.b_seg_stride % 4) return false;
    TcJobs T = J;
    return tc_gemm_configure(T) && tc_gemm_workspace(T) <= J.bpack_bytes;
}

size_t tc_gemm_workspace(const TcJobs& J) {
    TcJobs T = J;
    tc_gemm_configure(T);
    const size_t ntn = size_t((T.N + T.bn - 1) / T.bn), nk = size_t((T.K + kBK - 1) / kBK);
    return size_t(T.nseg) * ntn * nk * kTcBTile;
}

cudaError_t launch_tc_gemm(TcJobs& J, cudaStream_t st) {
    static int sms = 0;  // the attribute is per function, not per call; one resident CTA per SM
    if (!sms) {
        cudaError_t e = cudaFuncSetAttribute(tc_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemP);
        int dev = 0;
        if (e == cudaSuccess) e = cudaGetDevice(&dev);
        if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return e;
    }
    if (!tc_gemm_configure(J) || tc_gemm_workspace(J) > J.bpack_bytes) return cudaErrorInvalidValue;
    long long t = 0;
    for (int s = 0; s < J.nseg; ++s) {
        J.tile0[s] = int(t);
        t += (J.rows[s] + kBM - 1) / kBM;
    }
    J.tile0[J.nseg] = int(t);
    const long long tiles = t * ((J.N + J.bn - 1) / J.bn);
    if (tiles == 0) return cudaSuccess;
    if (tiles > 0x7FFFFFFF) return cudaErrorInvalidConfiguration;
    const int ntn = (J.N + J.bn - 1) / J.bn, nk = (J.K + kBK - 1) / kBK;
    tc_pack_b<<<unsigned(J.nseg * ntn * nk), 256, 0, st>>>(J, ntn, nk);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const unsigned grid = unsigned(std::min<long long>(tiles, sms));
    tc_gemm_kernel<<<grid, kThreadsP, kSmemP, st>>>(J);
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
