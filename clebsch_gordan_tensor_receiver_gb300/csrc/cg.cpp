// Real Clebsch-Gordan tensors for the planner.
//
// Derivation (deliberately a different route from a closed-form sum): the coupled multiplet
// |l3, M> inside |l1> (x) |l2> is built from its highest-weight state, fixed by J+ |l3,l3> = 0,
// and then lowered with J- = J1- + J2-.  That gives the complex (Condon-Shortley) coefficients
// <l1 m1 l2 m2 | l3 M>.  They are then expressed in the real basis of each l (rows m = -l..l):
//     m > 0 : (|-m> + (-1)^m |m>) / sqrt(2),   m = 0 : |0>,   m < 0 : i (|m> - (-1)^m |-m>) / sqrt(2)
// as C[m1,m2,m3] = sum Q1[m1,a] Q2[m2,b] conj(Q3[m3,c]) <l1 a l2 b | l3 c>, which is purely real
// (l1+l2+l3 even) or purely imaginary (odd); the non-zero part is kept and the tensor is signed
// so that its first non-zero entry in row-major (m1, m2, m3) order is positive.
// "An Efficient Sparse Kernel Generator for O(3)-Equivariant Deep Networks" (abstract) contracts
// two dense vectors with this structured sparse tensor; the phase and normalisation conventions
// are the plainest ones (unitary per output component, no extra path factor).
#include <cmath>
#include <complex>
#include <stdexcept>
#include <vector>

#include "plan.h"

namespace uvu {
namespace {

// The recursion runs in long double (80- or 128-bit depending on the host) so that the
// lowering chain adds no visible rounding before the final conversion to double.
using R = long double;
R raise_coef(int j, int m) { return std::sqrt(R(j * (j + 1) - m * (m + 1))); }
R lower_coef(int j, int m) { return std::sqrt(R(j * (j + 1) - m * (m - 1))); }

// cg[(m1+l1)][(m2+l2)][(M+l3)] complex-basis coefficients.
std::vector<R> complex_cg(int l1, int l2, int l3) {
    const int d1 = 2 * l1 + 1, d2 = 2 * l2 + 1, d3 = 2 * l3 + 1;
    std::vector<R> out(size_t(d1) * d2 * d3, 0.0L);
    auto at = [&](int m1, int m2, int M) -> R& {
        return out[(size_t(m1 + l1) * d2 + (m2 + l2)) * d3 + (M + l3)];
    };
    // highest weight: coefficients c(m1) on |m1>|l3 - m1>
    const int lo = std::max(-l1, l3 - l2), hi = std::min(l1, l3 + l2);
    std::vector<R> c(d1, 0.0L);
    c[lo + l1] = 1.0L;
    for (int k = lo + 1; k <= hi; ++k)
        c[k + l1] = -c[k - 1 + l1] * raise_coef(l1, k - 1) / raise_coef(l2, l3 - k);
    R nrm = 0.0L;
    for (int k = lo; k <= hi; ++k) nrm += c[k + l1] * c[k + l1];
    nrm = std::sqrt(nrm);
    const R sgn = c[hi + l1] >= 0 ? 1.0L : -1.0L;  // <l1 l1 l2 (l3-l1)|l3 l3> > 0
    // hi == l1 whenever the triangle rule holds, so the sign convention applies to m1 = l1
    for (int k = lo; k <= hi; ++k) at(k, l3 - k, l3) = sgn * c[k + l1] / nrm;
    // lower: |M-1> = (J1- + J2-)|M> / lower_coef(l3, M)
    for (int M = l3; M > -l3; --M) {
        const R b = lower_coef(l3, M);
        for (int m1 = -l1; m1 <= l1; ++m1) {
            const int m2 = M - 1 - m1;
            if (m2 < -l2 || m2 > l2) continue;
            R v = 0.0L;
            if (m1 + 1 <= l1) v += at(m1 + 1, m2, M) * lower_coef(l1, m1 + 1);
            if (m2 + 1 <= l2) v += at(m1, m2 + 1, M) * lower_coef(l2, m2 + 1);
            at(m1, m2, M - 1) = v / b;
        }
    }
    return out;
}

// Row m (index m+l) of the real-from-complex change of basis, as (column m', coefficient) pairs.
struct QRow {
    int n = 0;
    int col[2];
    std::complex<R> v[2];
};

QRow qrow(int l, int m) {
    const R h = 1.0L / std::sqrt(R(2));
    const R par = (m % 2 == 0) ? 1.0L : -1.0L;  // (-1)^m
    QRow q;
    if (m > 0) {
        q.n = 2;
        q.col[0] = -m; q.v[0] = h;
        q.col[1] = m;  q.v[1] = par * h;
    } else if (m == 0) {
        q.n = 1;
        q.col[0] = 0; q.v[0] = 1.0L;
    } else {
        q.n = 2;
        q.col[0] = m;  q.v[0] = std::complex<R>(0.0L, h);
        q.col[1] = -m; q.v[1] = std::complex<R>(0.0L, -par * h);
    }
    (void)l;
    return q;
}

}  // namespace

std::vector<double> real_cg_dense(int l1, int l2, int l3) {
    if (l3 < std::abs(l1 - l2) || l3 > l1 + l2) throw std::invalid_argument("triangle rule");
    const int d1 = 2 * l1 + 1, d2 = 2 * l2 + 1, d3 = 2 * l3 + 1;
    const std::vector<R> cc = complex_cg(l1, l2, l3);
    auto ccat = [&](int a, int b, int c) { return cc[(size_t(a + l1) * d2 + (b + l2)) * d3 + (c + l3)]; };
    std::vector<std::complex<R>> t(size_t(d1) * d2 * d3);
    for (int m1 = -l1; m1 <= l1; ++m1) {
        const QRow q1 = qrow(l1, m1);
        for (int m2 = -l2; m2 <= l2; ++m2) {
            const QRow q2 = qrow(l2, m2);
            for (int m3 = -l3; m3 <= l3; ++m3) {
                const QRow q3 = qrow(l3, m3);
                std::complex<R> s = 0.0L;
                for (int i = 0; i < q1.n; ++i)
                    for (int j = 0; j < q2.n; ++j)
                        for (int k = 0; k < q3.n; ++k) {
                            const int a = q1.col[i], b = q2.col[j], c = q3.col[k];
                            if (a + b != c) continue;
                            s += q1.v[i] * q2.v[j] * std::conj(q3.v[k]) * ccat(a, b, c);
                        }
                t[(size_t(m1 + l1) * d2 + (m2 + l2)) * d3 + (m3 + l3)] = s;
            }
        }
    }
    const bool even = ((l1 + l2 + l3) % 2) == 0;
    std::vector<double> out(t.size());
    double off_part = 0.0;
    for (size_t i = 0; i < t.size(); ++i) {
        out[i] = double(even ? t[i].real() : t[i].imag());
        off_part = std::max(off_part, double(std::abs(even ? t[i].imag() : t[i].real())));
        if (std::abs(out[i]) < 1e-15) out[i] = 0.0;
    }
    if (off_part > 1e-12) throw std::runtime_error("real CG is not purely real or imaginary");
    for (size_t i = 0; i < out.size(); ++i) {
        if (std::abs(out[i]) > 1e-9) {
            if (out[i] < 0)
                for (double& v : out) v = -v;
            break;
        }
    }
    return out;
}

}  // namespace uvu
