/*
 * CPU fp64 oracle of the channel-wise (UVU) CG tensor-product graph convolution.
 * TEST INFRASTRUCTURE ONLY: built and called by the test suite, the smoke check and the
 * CPU-baseline leg of the benchmark; never by the CUDA library.
 *
 * Definitions followed (the pages give the ownership scheme and the fused CG product +
 * convolution; the sums below are the operation itself, written out with no blocking,
 * fusion or reordering):
 *
 *   forward   ("Receiver-streaming convolutions for channel-wise UVU tensor products",
 *              opening post: a (receiver, channel) owner reduces over the receiver's edges)
 *     out[r,u,oo(p)+m3] = sum_{e in seg(r)} w[e,p,u]
 *                         sum_{m1,m2} C_p[m1,m2,m3] x[src(e),u,xo(p)+m1] Y[e,yo(p)+m2]
 *
 *   backward  (same post, backward paragraph: radial-weight, spherical-harmonic and node
 *              feature gradients; "An Efficient Sparse Kernel Generator for O(3)-Equivariant
 *              Deep Networks", abstract: gradient kernels of the CG tensor product)
 *     dw[e,p,u]        = sum_{m3} d_out[recv(e),u,oo+m3] sum_{m1,m2} C_p x[src(e),u,xo+m1] Y[e,yo+m2]
 *     dY[e,yo+m2]     += sum_u sum_{p} w[e,p,u] sum_{m1,m3} C_p x[src(e),u,xo+m1] d_out[recv(e),u,oo+m3]
 *     dx[s,u,xo+m1]   += sum_{e: src(e)=s} sum_p w[e,p,u] sum_{m2,m3} C_p Y[e,yo+m2] d_out[recv(e),u,oo+m3]
 *
 * Each path is described by 7 ints: l1, l2, l3, xo, yo, oo, cgo (offset of its dense
 * (2l1+1)(2l2+1)(2l3+1) CG block, row-major in m1, m2, m3, inside `cg`).  The CG loops are dense
 * (zeros included) so that the code reads as the formula.  Every output element is owned by one
 * OpenMP iteration (receiver, edge or sender), so results do not depend on the thread count.
 */
#include <stdint.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define PL1(p) paths[7 * (p) + 0]
#define PL2(p) paths[7 * (p) + 1]
#define PL3(p) paths[7 * (p) + 2]
#define PXO(p) paths[7 * (p) + 3]
#define PYO(p) paths[7 * (p) + 4]
#define POO(p) paths[7 * (p) + 5]
#define PCG(p) paths[7 * (p) + 6]

static void set_threads(int n) {
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

int oracle_max_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Forward over a list of receivers: seg(r) = [offsets[r], offsets[r+1]) indexes src, Y and w. */
void oracle_fwd(int64_t n_recv, const int64_t *offsets, const int32_t *src, int U, int P,
                const int *paths, const double *cg, int Dx, int Dy, int Do, const double *x,
                const double *Y, const double *w, double *out, int nthreads) {
    set_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 4)
    for (int64_t r = 0; r < n_recv; ++r) {
        double *o = out + r * (int64_t)U * Do;
        memset(o, 0, sizeof(double) * (size_t)U * Do);
        for (int64_t e = offsets[r]; e < offsets[r + 1]; ++e) {
            const int64_t s = src[e];
            for (int u = 0; u < U; ++u) {
                const double *xs = x + (s * U + u) * Dx;
                const double *ye = Y + e * Dy;
                double *ou = o + (int64_t)u * Do;
                for (int p = 0; p < P; ++p) {
                    const int d1 = 2 * PL1(p) + 1, d2 = 2 * PL2(p) + 1, d3 = 2 * PL3(p) + 1;
                    const double *c = cg + PCG(p);
                    const double wp = w[(e * P + p) * U + u];
                    for (int m1 = 0; m1 < d1; ++m1)
                        for (int m2 = 0; m2 < d2; ++m2)
                            for (int m3 = 0; m3 < d3; ++m3)
                                ou[POO(p) + m3] += wp * c[(m1 * d2 + m2) * d3 + m3] *
                                                   xs[PXO(p) + m1] * ye[PYO(p) + m2];
                }
            }
        }
    }
}

/* dw and dY for a list of edges; edge k reads Y[k], w[k], x[src[k]], d_out[recv[k]]. */
void oracle_bwd_edges(int64_t n_edges, const int32_t *recv, const int32_t *src, int U, int P,
                      const int *paths, const double *cg, int Dx, int Dy, int Do,
                      const double *x, const double *Y, const double *w, const double *d_out,
                      double *dY, double *dw, int nthreads) {
    set_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 64)
    for (int64_t e = 0; e < n_edges; ++e) {
        const int64_t s = src[e], r = recv[e];
        const double *ye = Y + e * Dy;
        double *dye = dY ? dY + e * Dy : 0;
        if (dye) memset(dye, 0, sizeof(double) * (size_t)Dy);
        for (int p = 0; p < P; ++p) {
            const int d1 = 2 * PL1(p) + 1, d2 = 2 * PL2(p) + 1, d3 = 2 * PL3(p) + 1;
            const double *c = cg + PCG(p);
            for (int u = 0; u < U; ++u) {
                const double *xs = x + (s * U + u) * Dx;
                const double *g = d_out + (r * U + u) * Do;
                const double wp = w[(e * P + p) * U + u];
                double acc_w = 0.0;
                for (int m1 = 0; m1 < d1; ++m1)
                    for (int m2 = 0; m2 < d2; ++m2)
                        for (int m3 = 0; m3 < d3; ++m3) {
                            const double cv = c[(m1 * d2 + m2) * d3 + m3];
                            acc_w += g[POO(p) + m3] * cv * xs[PXO(p) + m1] * ye[PYO(p) + m2];
                            if (dye)
                                dye[PYO(p) + m2] += wp * cv * xs[PXO(p) + m1] * g[POO(p) + m3];
                        }
                if (dw) dw[(e * P + p) * U + u] = acc_w;
            }
        }
    }
}

/* dx for a list of senders: entries k in [soff[s], soff[s+1]) name edge eids[k] (indexing Y
 * and w) and its receiver krecv[k] (indexing d_out). */
void oracle_bwd_dx(int64_t n_send, const int64_t *soff, const int32_t *eids, const int32_t *krecv,
                   int U, int P, const int *paths, const double *cg, int Dx, int Dy, int Do,
                   const double *Y, const double *w, const double *d_out, double *dx,
                   int nthreads) {
    set_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 16)
    for (int64_t s = 0; s < n_send; ++s) {
        double *o = dx + s * (int64_t)U * Dx;
        memset(o, 0, sizeof(double) * (size_t)U * Dx);
        for (int64_t k = soff[s]; k < soff[s + 1]; ++k) {
            const int64_t e = eids[k], r = krecv[k];
            const double *ye = Y + e * Dy;
            for (int u = 0; u < U; ++u) {
                const double *g = d_out + (r * U + u) * Do;
                double *ou = o + (int64_t)u * Dx;
                for (int p = 0; p < P; ++p) {
                    const int d1 = 2 * PL1(p) + 1, d2 = 2 * PL2(p) + 1, d3 = 2 * PL3(p) + 1;
                    const double *c = cg + PCG(p);
                    const double wp = w[(e * P + p) * U + u];
                    for (int m1 = 0; m1 < d1; ++m1)
                        for (int m2 = 0; m2 < d2; ++m2)
                            for (int m3 = 0; m3 < d3; ++m3)
                                ou[PXO(p) + m1] += wp * c[(m1 * d2 + m2) * d3 + m3] *
                                                   ye[PYO(p) + m2] * g[POO(p) + m3];
                }
            }
        }
    }
}
