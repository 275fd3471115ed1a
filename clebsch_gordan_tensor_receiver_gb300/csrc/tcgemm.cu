// Dense fp32 products on the 5th-generation tensor cores (tcgen05) with fp32 accuracy.
//
// The dense contractions next to the convolution -- the channel mixing that reduces a factorised
// UVW convolution to the UVU one, and the last linear layer of the radial network (with its
// input gradient) -- are ordinary matrix products.  A single TF32 product keeps 11 significant
// bits, far outside the fp32 tolerance, so each operand is split as x = hi + lo (hi = x rounded to
// TF32, lo = x - hi rounded to TF32) and the product is accumulated as hi*hi + hi*lo + lo*hi
// ("3xTF32"; the dropped lo*lo term and the rounding of lo are about 2^-22 of each product; a
// split that truncated hi instead leaves a 13-bit lo whose truncation costs 2^-20 per product,
// which long reductions visibly accumulate).  Accumulation is fp32 in tensor memory.
//
// Persistent kernel, one CTA per SM looping over 128 x BN tiles of C (BN = 128, or 64 for narrow C
// or long K), with warp roles (an MMA costs about 60 ns up to N = 128 and 66 ns at N = 256 on
// GB300 when its operands change, so wide tiles pay):
//   warp 0      A producer: one TMA load per 32-wide K chunk of a 128-row tile (raw fp32, 128-byte
//               swizzled K-major rows) into a ring of A stages;
//   warp 1      B producer: B is pre-split once per call into hi and lo tiles in the MMA's layout
//               (tc_pack_b); one bulk copy per chunk into a ring of B stages, skipped when the
//               stage already holds that tile (a CTA keeps its N tile across row tiles, and a
//               short K fits the ring, so small B stays resident);
//   warp 2      MMA issue (one thread): M = 128, N = BN, K = 8 per instruction, three products per
//               K step, into one of two tensor-memory accumulators;
//   warps 4-7   epilogue: tcgen05.ld (one tile row per thread), fp32 sums of the K ranges in
//               registers, rows staged in shared memory and stored 128 bytes at a time;
//   warps 8-11  converters: thread = tile row; its 32 raw values of the chunk, split into hi and
//               lo, written into tensor memory (tcgen05.st) as the A operand of the MMAs.
// Measured on GB300: an accumulation in tensor memory loses more than a round-to-nearest fp32
// add (a 35,000-term reduction was off by 3e-3 where fp32 sums in registers stay near 1e-4), so
// long K is summed in ranges of at most 256, each accumulated afresh and added into fp32
// registers by the epilogue.  Every mbarrier wait is bounded (about two seconds on the global
// timer); on expiry the role sets a shared flag and the tc_status_word bit, every role leaves its
// loop, the producers wait (bounded) for the copies they issued, the MMA thread for its issued
// MMAs, and the CTA frees its tensor memory and returns.
//
//   C[row][n] = sum_k A[row][k] B_s[k][n] over the rows of each segment s (A row-major, K
//   contiguous; B_s = B + s * b_seg_stride, either n- or k-contiguous).
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <mutex>

#include "plan.h"
#include "tcgemm.h"

namespace uvu {
namespace {

constexpr int kBM = 128, kBNmax = 128, kBK = 32;
constexpr int kRawBytes = kBM * kBK * 4;  // one raw A chunk: 128 rows x 128 bytes
constexpr int kKacc = 256;                // longest K accumulated in tensor memory at once
constexpr int kThreadsP = 12 * 32;
constexpr int kStgPitch = 36;                      // floats per staged row (32 + 4 pad)
constexpr int kStgBytes = 4 * 32 * kStgPitch * 4;  // four epilogue warps x 32 rows
constexpr int kSmemMax = 232448;                   // 227 KB per CTA
constexpr int kBarBytes = 512;  // up to 41 barriers (raw 8, A 6, B 4 stages), 8 bytes each

__device__ unsigned int tc_status_word;

__device__ __forceinline__ uint32_t smem_u32(const void* p) { return uint32_t(__cvta_generic_to_shared(p)); }

__device__ __forceinline__ uint32_t tf32_rna(float x) {
    uint32_t r;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
    return r;
}

// Byte offset of element (row, k), k < 32, in a 128-byte-swizzled K-major tile: 8-row groups of
// 1024 bytes, 128 bytes per row, the 16-byte chunk index XORed with the row within the group
// (the layout a TMA load with 128-byte swizzle writes, and the MMA's SWIZZLE_128B operand form).
__device__ __forceinline__ uint32_t sw128(int row, int k) {
    return uint32_t((row >> 3) * 1024 + (row & 7) * 128 + ((((k >> 2) ^ row) & 7) << 4) + (k & 3) * 4);
}

// Shared-memory matrix descriptor, K-major with 128-byte swizzle: start address, leading offset
// unused (1), stride between 8-row groups 1024 bytes, fixed version bits 0b001 at 46, swizzle
// mode 2 (128 bytes) at 61.  Advancing K by 8 TF32 values adds 32 bytes to the start address.
__device__ __forceinline__ uint64_t sdesc(uint32_t addr) {
    return uint64_t((addr >> 4) & 0x3FFFu) | (uint64_t(1) << 16) | (uint64_t(1024 >> 4) << 32) | (1ull << 46) |
           (2ull << 61);
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
__device__ __forceinline__ void mbar_init_n(uint32_t b, uint32_t n) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(b), "r"(n) : "memory");
}
__device__ __forceinline__ void mbar_arrive1(uint32_t b) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(b) : "memory");
}
__device__ __forceinline__ void mbar_arrive_tx(uint32_t b, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(b), "r"(bytes) : "memory");
}
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
            dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
        : "memory");
}
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
                 "l"(src), "r"(bytes), "r"(bar)
                 : "memory");
}
__device__ __forceinline__ void tc_commit(uint32_t b) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(b) : "memory");
}
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
          "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]),
          "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
          "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
}
__device__ __forceinline__ void tmem_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// Shared-memory layout of one launch (offsets from the 1024-aligned base): nraw raw A stages (TMA
// destinations), nb B stages (hi, lo), the epilogue staging rows, the barriers.  Tensor memory:
// two accumulators of bn columns, then na A stages of 64 columns (hi in the first 32, lo in the
// next 32; lane = tile row, column = k).
struct Layout {
    int bn, nraw, nb;
    __host__ __device__ int b_bytes() const { return 2 * bn * 128; }
    __host__ __device__ int b0() const { return nraw * kRawBytes; }
    __host__ __device__ int stg0() const { return b0() + nb * b_bytes(); }
    __host__ __device__ int bar0() const { return stg0() + kStgBytes; }
    __host__ __device__ int total() const { return bar0() + kBarBytes + 1024; }  // + alignment slack
};

// Warp roles
constexpr int kWarpA = 0, kWarpB = 1, kWarpMma = 2, kEpi0 = 4, kConv0 = 8;

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
        "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
        "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]),
        "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]),
        "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
        : "memory");
}
// D (tensor memory) += A (tensor memory) B (shared memory descriptor)
__device__ __forceinline__ void mma_tf32_ta(uint32_t d, uint32_t a, uint64_t b, uint32_t id, uint32_t accum) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %3, 0;\n"
        " tcgen05.mma.cta_group::1.kind::tf32 [%0], [%1], %2, %4, p;\n}\n" ::"r"(d),
        "r"(a), "l"(b), "r"(accum), "r"(id)
        : "memory");
}

__global__ void __launch_bounds__(kThreadsP, 1) tc_gemm_kernel(const __grid_constant__ CUtensorMap tmA, TcJobs J) {
    extern __shared__ unsigned char smem_raw[];
    __shared__ int s_dead;
    __shared__ uint32_t s_tmem;
    unsigned char* smem =
        reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const Layout L{J.bn, J.nraw, J.nb};
    const uint32_t sbase = smem_u32(smem);
    const int bn = J.bn, K = J.K, NA = J.na;
    const int nk = (K + kBK - 1) / kBK;   // K chunks per tile
    const int cpr = J.kacc / kBK;         // K chunks per accumulation range
    const int nr = (nk + cpr - 1) / cpr;  // ranges per tile
    const int ntn = (J.N + bn - 1) / bn;
    const int nrt = J.tile0[J.nseg];      // row tiles
    const int T = nrt * ntn;              // tiles (< 2^31, checked by the launcher)
    const int my_tiles = T > int(blockIdx.x) ? (T - 1 - int(blockIdx.x)) / int(gridDim.x) + 1 : 0;
    const int C = my_tiles * nk;          // chunks of this CTA
    const int nbu = nk <= L.nb ? nk : L.nb;  // B stages in use: chunk kc keeps stage kc when K fits
    // barriers: raw_full[nraw], raw_empty[nraw], ta_full[na], ta_empty[na], b_full[nb], b_empty[nb],
    // acc_full[2], acc_empty[2], fin
    const uint32_t raw_full = sbase + L.bar0(), raw_empty = raw_full + 8 * L.nraw, ta_full = raw_empty + 8 * L.nraw,
                   ta_empty = ta_full + 8 * NA, b_full = ta_empty + 8 * NA, b_empty = b_full + 8 * L.nb,
                   acc_full = b_empty + 8 * L.nb, acc_empty = acc_full + 16, fin = acc_empty + 16;

    if (tid == 0) {
        s_dead = 0;
        for (int i = 0; i < L.nraw; ++i) {
            mbar_init_n(raw_full + 8 * i, 1);
            mbar_init_n(raw_empty + 8 * i, 4);
        }
        for (int i = 0; i < NA; ++i) {
            mbar_init_n(ta_full + 8 * i, 4);
            mbar_init_n(ta_empty + 8 * i, 1);
        }
        for (int i = 0; i < L.nb; ++i) {
            mbar_init_n(b_full + 8 * i, 1);
            mbar_init_n(b_empty + 8 * i, 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init_n(acc_full + 8 * i, 1);
            mbar_init_n(acc_empty + 8 * i, 4);
        }
        mbar_init_n(fin, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&s_tmem)),
                     "r"(J.tmem_cols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(&s_tmem);
    const uint32_t ta0 = tmem + uint32_t(2 * bn);  // first A stage column
    volatile int* dead = &s_dead;
    auto wdead = [&]() { return __any_sync(0xffffffffu, *dead != 0); };

    // tile number (within this CTA's sequence) -> segment, first row, row end, N tile.  With
    // J.nmajor the row tiles of one N tile are consecutive (a CTA keeps its N tile, and so its B,
    // over many row tiles); otherwise the N tiles of one row tile are.
    auto tile_of = [&](int lt, int& seg, long long& m0, long long& rend, int& nt) {
        const int t = int(blockIdx.x) + lt * int(gridDim.x);
        int rt;
        if (J.nmajor) {
            nt = t / nrt;
            rt = t - nt * nrt;
        } else {
            rt = t / ntn;
            nt = t - rt * ntn;
        }
        seg = 0;
        while (seg + 1 < J.nseg && rt >= J.tile0[seg + 1]) ++seg;
        m0 = J.row0[seg] + (long long)(rt - J.tile0[seg]) * kBM;
        rend = J.row0[seg] + J.rows[seg];
    };

    if (warp == kWarpA) {
        // ---------------------------------------------------------------- A producer (TMA)
        if (lane == 0) {
            int q = 0;
            for (int lt = 0; lt < my_tiles && !*dead; ++lt) {
                int seg, nt;
                long long m0, rend;
                tile_of(lt, seg, m0, rend, nt);
                for (int kc = 0; kc < nk; ++kc, ++q) {
                    const int s = q % L.nraw;
                    if (q >= L.nraw && !mbar_wait(raw_empty + 8 * s, uint32_t((q / L.nraw) - 1) & 1u)) {
                        *dead = 1;
                        break;
                    }
                    if (*dead) break;
                    mbar_arrive_tx(raw_full + 8 * s, kRawBytes);
                    tma_load_2d(sbase + s * kRawBytes, &tmA, kc * kBK, int(m0), raw_full + 8 * s);
                }
            }
            // copies still in flight land before the CTA can leave (only waits when a role gave up)
            if (*dead)
                for (int k = max(0, q - L.nraw); k < q; ++k)
                    mbar_wait(raw_full + 8 * (k % L.nraw), uint32_t(k / L.nraw) & 1u);
        }
    } else if (warp == kWarpB) {
        // ---------------------------------------------------------------- B producer (bulk copy)
        if (lane == 0) {
            const uint32_t bb = uint32_t(L.b_bytes());
            long long held[4] = {-1, -1, -1, -1};  // the tile each stage holds (-1: none)
            int q = 0, issued = 0;
            for (int lt = 0; lt < my_tiles && !*dead; ++lt) {
                int seg, nt;
                long long m0, rend;
                tile_of(lt, seg, m0, rend, nt);
                for (int kc = 0; kc < nk; ++kc, ++q) {
                    const int s = q % nbu;
                    if (q >= nbu && !mbar_wait(b_empty + 8 * s, uint32_t((q / nbu) - 1) & 1u)) {
                        *dead = 1;
                        break;
                    }
                    if (*dead) break;
                    const long long id = ((long long)seg * ntn + nt) * nk + kc;
                    if (held[s] == id) {
                        mbar_arrive1(b_full + 8 * s);  // already in place
                    } else {
                        held[s] = id;
                        mbar_arrive_tx(b_full + 8 * s, bb);
                        bulk_g2s(sbase + L.b0() + s * bb, static_cast<const unsigned char*>(J.bpack) + size_t(id) * bb, bb,
                                 b_full + 8 * s);
                        issued = q + 1;
                    }
                }
            }
            if (*dead)
                for (int k = max(0, issued - nbu); k < issued; ++k) mbar_wait(b_full + 8 * (k % nbu), uint32_t(k / nbu) & 1u);
        }
    } else if (warp >= kConv0) {
        // ---------------------------------------------------------------- converters
        // thread = tile row (its warp's TMEM lane quadrant); the row's 32 raw values are read from
        // the swizzled stage, split, and written as 32 hi and 32 lo columns of the A stage
        const int row = 32 * (warp & 3) + lane;
        const uint32_t tq = uint32_t(32 * (warp & 3)) << 16;
        const unsigned char* rbase = smem + (row >> 3) * 1024 + (row & 7) * 128;
        for (int q = 0; q < C && !wdead(); ++q) {
            const int r = q % L.nraw, a = q % NA;
            bool ok = mbar_wait(raw_full + 8 * r, uint32_t(q / L.nraw) & 1u);
            if (ok && q >= NA) ok = mbar_wait(ta_empty + 8 * a, uint32_t((q / NA) - 1) & 1u);
            if (!__all_sync(0xffffffffu, ok)) {
                *dead = 1;
                break;
            }
            asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
            uint32_t hi[32], lo[32];
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                const float4 v = *reinterpret_cast<const float4*>(rbase + r * kRawBytes + (((c ^ row) & 7) << 4));
                const float x[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const uint32_t h = tf32_rna(x[j]);
                    hi[4 * c + j] = h;
                    lo[4 * c + j] = tf32_rna(x[j] - __uint_as_float(h));
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive1(raw_empty + 8 * r);  // the raw stage has been read
            const uint32_t col = ta0 + uint32_t(a * 64);
            tmem_st32(tq + col, hi);
            tmem_st32(tq + col + 32, lo);
            asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
            asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
            __syncwarp();
            if (lane == 0) mbar_arrive1(ta_full + 8 * a);
        }
    } else if (warp == kWarpMma) {
        // ---------------------------------------------------------------- MMA issue
        if (lane == 0) {
            const uint32_t id = idesc(bn);
            int q = 0, qa = 0;
            for (int lt = 0; lt < my_tiles && !*dead; ++lt) {
                for (int rr = 0; rr < nr && !*dead; ++rr, ++qa) {
                    const int b = qa & 1, v = qa >> 1;
                    if (v > 0 && !mbar_wait(acc_empty + 8 * b, uint32_t(v - 1) & 1u)) {
                        *dead = 1;
                        break;
                    }
                    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
                    const uint32_t d = tmem + uint32_t(b * bn);
                    const int k1 = min(nk, (rr + 1) * cpr);
                    for (int kc = rr * cpr; kc < k1; ++kc, ++q) {
                        const int a = q % NA, sb = q % nbu;
                        if (!mbar_wait(ta_full + 8 * a, uint32_t(q / NA) & 1u) ||
                            !mbar_wait(b_full + 8 * sb, uint32_t(q / nbu) & 1u)) {
                            *dead = 1;
                            break;
                        }
                        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
                        const uint32_t ah = ta0 + uint32_t(a * 64), al = ah + 32;
                        const uint32_t bh = sbase + L.b0() + sb * L.b_bytes(), bl = bh + bn * 128;
#pragma unroll
                        for (int ks = 0; ks < kBK / 8; ++ks) {
                            const uint32_t ko = ks * 32;
                            mma_tf32_ta(d, al + ks * 8, sdesc(bh + ko), id, (kc == rr * cpr && ks == 0) ? 0u : 1u);
                            mma_tf32_ta(d, ah + ks * 8, sdesc(bl + ko), id, 1u);
                            mma_tf32_ta(d, ah + ks * 8, sdesc(bh + ko), id, 1u);
                        }
                        // the stages are free once these MMAs are done
                        tc_commit(ta_empty + 8 * a);
                        tc_commit(b_empty + 8 * sb);
                    }
                    if (*dead) break;
                    tc_commit(acc_full + 8 * b);  // the range's accumulator is complete
                }
            }
            // every issued MMA has finished before the tensor memory is released
            tc_commit(fin);
            mbar_wait(fin, 0);
        }
        __syncwarp();
    } else if (warp >= kEpi0 && warp < kEpi0 + 4) {
        // ---------------------------------------------------------------- epilogue
        const int ew = warp & 3;  // TMEM lane quadrant: this warp may read lanes 32 ew .. + 31
        const uint32_t tl = tmem + (uint32_t(ew * 32) << 16);
        float* stg = reinterpret_cast<float*>(smem + L.stg0()) + (warp - kEpi0) * 32 * kStgPitch;
        float sums[64];
        int qa = 0;
        // 32 columns of this warp's 32 rows, staged and stored 128 bytes per row segment
        auto store32 = [&](const float* v, long long m0, long long rend, int col) {
            float4* my = reinterpret_cast<float4*>(stg + lane * kStgPitch);
#pragma unroll
            for (int x = 0; x < 8; ++x) my[x] = make_float4(v[4 * x], v[4 * x + 1], v[4 * x + 2], v[4 * x + 3]);
            __syncwarp();
            const int c4 = lane & 7;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int row = 4 * i + (lane >> 3);
                const long long grow = m0 + ew * 32 + row;
                if (grow < rend && col + 4 * c4 < J.N)
                    *reinterpret_cast<float4*>(J.C + grow * J.ldc + col + 4 * c4) =
                        *reinterpret_cast<const float4*>(stg + row * kStgPitch + 4 * c4);
            }
            __syncwarp();
        };
        for (int lt = 0; lt < my_tiles && !wdead(); ++lt) {
            int seg, nt;
            long long m0, rend;
            tile_of(lt, seg, m0, rend, nt);
            const int n0 = nt * bn;
            for (int rr = 0; rr < nr && !wdead(); ++rr, ++qa) {
                const int b = qa & 1;
                const bool ok = __all_sync(0xffffffffu, mbar_wait(acc_full + 8 * b, uint32_t(qa >> 1) & 1u));
                if (!ok) {
                    *dead = 1;
                    break;
                }
                asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
                if (nr == 1) {
                    // one range: each 32-column block leaves as soon as it is read
                    for (int cc = 0; cc < bn; cc += 32) {
                        uint32_t v[32];
                        tmem_ld32(tl + uint32_t(b * bn + cc), v);
                        tmem_wait();
                        float f[32];
#pragma unroll
                        for (int x = 0; x < 32; ++x) f[x] = __uint_as_float(v[x]);
                        store32(f, m0, rend, n0 + cc);
                    }
                } else {
                    // several ranges (bn = 64): running fp32 sums in registers, in range order
#pragma unroll
                    for (int cc = 0; cc < 64; cc += 32) {
                        uint32_t v[32];
                        tmem_ld32(tl + uint32_t(b * bn + cc), v);
                        tmem_wait();
#pragma unroll
                        for (int x = 0; x < 32; ++x)
                            sums[cc + x] = rr == 0 ? __uint_as_float(v[x]) : sums[cc + x] + __uint_as_float(v[x]);
                    }
                }
                asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
                __syncwarp();
                if (lane == 0) mbar_arrive1(acc_empty + 8 * b);  // the accumulator may be reused
                if (nr > 1 && rr == nr - 1) {
                    store32(sums, m0, rend, n0);
                    store32(sums + 32, m0, rend, n0 + 32);
                }
            }
        }
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    if (warp == 0)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(J.tmem_cols) : "memory");
}

// B_s[k][n] (any strides) -> the pre-split tiles of J.bpack: one block per (segment, N tile,
// K chunk), hi tile then lo tile, each bn rows (n) x 32 k in the 128-byte-swizzled K-major layout;
// zeros outside [0, K) x [0, N).
// One tile (segment, N tile, K chunk) per blockIdx.x, its bn x 32 elements spread over
// gridDim.y blocks (a few elements per thread: the tiles are small and latency-bound).
__global__ void __launch_bounds__(256) tc_pack_b(TcJobs J, int ntn, int nk) {
    const int kc = blockIdx.x % nk, nt = (blockIdx.x / nk) % ntn, seg = blockIdx.x / (nk * ntn);
    const int bn = J.bn;
    unsigned char* t = static_cast<unsigned char*>(J.bpack) + size_t(blockIdx.x) * (2 * bn * 128);
    const float* Bs = J.B + (long long)seg * J.b_seg_stride;
    const int n0 = nt * bn, k0 = kc * kBK;
    for (int e = blockIdx.y * 256 + threadIdx.x; e < bn * kBK; e += 256 * gridDim.y) {
        const int n = J.b_kcont ? (e / kBK) : (e % bn), k = J.b_kcont ? (e % kBK) : (e / bn);
        float v = 0.f;
        if (n0 + n < J.N && k0 + k < J.K) v = Bs[(long long)(k0 + k) * J.sbk + (long long)(n0 + n) * J.sbn];
        const uint32_t h = tf32_rna(v);
        const uint32_t l = tf32_rna(v - __uint_as_float(h));
        const uint32_t o = sw128(n, k);
        *reinterpret_cast<uint32_t*>(t + o) = h;
        *reinterpret_cast<uint32_t*>(t + bn * 128 + o) = l;
    }
}

using EncodeTiled = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                 const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                 CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// The driver's tensor-map encoder, looked up once through the runtime (the library does not link
// the driver library).
EncodeTiled encoder() {
    static EncodeTiled fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiled>(p);
    });
    return fn;
}

}  // namespace

// Tile shape of a product: N tiles of 128 columns when N >= 128 and K is one range, else 64
// (whose several K-range sums then fit the registers); K summed in ranges of at most kKacc.
// Tensor memory (512 columns): the two accumulators, then as many 64-column A stages as fit.
// Shared memory: B stages enough to hold a short K, the rest raw A stages (up to 8).
bool tc_gemm_configure(TcJobs& J) {
    const int nk = (J.K + kBK - 1) / kBK;
    const int nr = (J.K + kKacc - 1) / kKacc;  // ranges
    const int per = (nk + nr - 1) / nr;        // chunks per range
    J.kacc = per * kBK;
    J.bn = (J.N >= 128 && nr == 1) ? kBNmax : 64;
    J.tmem_cols = 512;
    J.na = (512 - 2 * J.bn) / 64;
    J.nb = J.bn == kBNmax ? 3 : 4;
    const Layout none{J.bn, 0, J.nb};
    const int room = kSmemMax - 1024 /* static shared memory */ - none.total();
    J.nraw = std::min(8, room / kRawBytes);
    return J.nraw >= 2;
}

// Requirements of the tensor-core path: 16-byte aligned base pointers and row strides that keep
// every row 16-byte aligned (TMA and 16-byte stores); widths that are multiples of 4; room for
// the pre-split B tiles.
bool tc_gemm_supported(const TcJobs& J) {
    auto al = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
    if (!al(J.A) || !al(J.C) || !J.B || !J.bpack || !al(J.bpack) || J.nseg < 1 || J.nseg > kTcMaxSeg || J.N % 4 || J.N < 1)
        return false;
    if (J.K < 1 || J.K % 4 || J.lda % 4 || J.ldc % 4 || J.b_seg_stride % 4) return false;
    if (!encoder()) return false;
    TcJobs T = J;
    return tc_gemm_configure(T) && tc_gemm_workspace(T) <= J.bpack_bytes;
}

size_t tc_gemm_workspace(const TcJobs& J) {
    TcJobs T = J;
    tc_gemm_configure(T);
    const size_t ntn = size_t((T.N + T.bn - 1) / T.bn), nk = size_t((T.K + kBK - 1) / kBK);
    return size_t(T.nseg) * ntn * nk * size_t(2 * T.bn * 128);
}

cudaError_t launch_tc_gemm(TcJobs& J, cudaStream_t st) {
    if (!tc_gemm_configure(J) || tc_gemm_workspace(J) > J.bpack_bytes) return cudaErrorInvalidValue;
    const EncodeTiled enc = encoder();
    if (!enc) return cudaErrorNotSupported;
    const Layout L{J.bn, J.nraw, J.nb};
    static int sms = 0;  // one resident CTA per SM; the attribute is per function
    static int attr_bytes = 0;
    if (!sms) {
        int dev = 0;
        cudaError_t e = cudaGetDevice(&dev);
        if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return e;
    }
    if (L.total() > attr_bytes) {
        cudaError_t e = cudaFuncSetAttribute(tc_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, L.total());
        if (e != cudaSuccess) return e;
        attr_bytes = L.total();
    }
    long long t = 0, extent = 0;
    for (int s = 0; s < J.nseg; ++s) {
        J.tile0[s] = int(t);
        t += (J.rows[s] + kBM - 1) / kBM;
        extent = std::max(extent, J.row0[s] + J.rows[s]);
    }
    J.tile0[J.nseg] = int(t);
    const long long tiles = t * ((J.N + J.bn - 1) / J.bn);
    if (tiles == 0) return cudaSuccess;
    if (tiles > 0x7FFFFFFF || extent > 0x7FFFFFFF) return cudaErrorInvalidConfiguration;
    // A as a 2-D tensor [extent rows][K] (row pitch lda), boxes of 128 rows x 32 values (128 bytes,
    // the swizzle span); rows and K beyond the extent read as zeros
    CUtensorMap tm;
    const cuuint64_t dims[2] = {cuuint64_t(J.K), cuuint64_t(extent)};
    const cuuint64_t strides[1] = {cuuint64_t(J.lda) * 4u};
    const cuuint32_t box[2] = {uint32_t(kBK), uint32_t(kBM)};
    const cuuint32_t es[2] = {1u, 1u};
    if (enc(&tm, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float*>(J.A), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    const int ntn = (J.N + J.bn - 1) / J.bn, nk = (J.K + kBK - 1) / kBK;
    tc_pack_b<<<dim3(unsigned(J.nseg * ntn * nk), unsigned((J.bn * kBK + 1023) / 1024)), 256, 0, st>>>(J, ntn, nk);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const unsigned grid = unsigned(std::min<long long>(tiles, sms));
    // a CTA keeps one N tile in either order when the grid is a multiple of the N tiles (and then
    // the CTAs on one row tile run together, sharing its A through L2); otherwise N-major order
    J.nmajor = (grid % unsigned(ntn)) != 0 ? 1 : 0;
    tc_gemm_kernel<<<grid, kThreadsP, L.total(), st>>>(tm, J);
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
