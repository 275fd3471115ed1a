// Job tables of the tensor-core product kernel (tcgemm.cu); shared by its callers.
#pragma once

#include "plan.h"

namespace uvu {

struct TcJobs {
    int nseg;
    long long row0[kTcMaxSeg];
    long long rows[kTcMaxSeg];
    int tile0[kTcMaxSeg + 1];  // prefix of 128-row tiles over the segments (set by the launcher)
    int K;                   // reduction length (columns of A)
    int N;                   // columns of C
    int b_kcont;             // B[k][n] has k contiguous (else n contiguous)
    const float* A;
    long long lda;           // elements between rows of A
    const float* B;
    long long sbk, sbn;      // B strides for k and n
    long long b_seg_stride;  // offset of B_s
    float* C;
    long long ldc;           // elements between rows of C
    // B pre-split into its hi and lo TF32 parts in the MMA's shared-memory layout, one 32-k chunk
    // of one N tile per 2 x bn x 128 bytes: [segment][N tile][K chunk] (written by the launcher
    // into caller workspace of tc_gemm_workspace() bytes)
    void* bpack;
    size_t bpack_bytes;      // room at bpack (the launcher refuses less than tc_gemm_workspace())
    // set by the launcher
    int bn;                  // columns per tile
    int kacc;                // K per accumulator
    int tmem_cols;           // tensor-memory columns allocated per CTA
    int nraw, na, nb;        // stages of the raw A ring (shared memory), the A ring (tensor memory), the B ring
    int nmajor;              // tile order: the row tiles of one N tile consecutive (else the N tiles of a row tile)
};

}  // namespace uvu
