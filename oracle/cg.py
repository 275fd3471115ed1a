"""Real Clebsch-Gordan coefficients for the oracle (test infrastructure only).

Steps, in the order the real coupling tensor is built:

1. ``complex_cg(l1, m1, l2, m2, l3, m3)``: the textbook Racah closed-form sum for
   <l1 m1 l2 m2 | l3 m3> with the Condon-Shortley phase.  The sum and the factorial prefactor
   are evaluated in exact rational arithmetic (``fractions.Fraction``); only the final square
   root is rounded, so each coefficient is correct to one fp64 rounding.
2. ``real_basis(l)``: the unitary matrix Q_l whose row m (m = -l..l) expresses the real harmonic
   of order m in the complex ones Y_l^{m'} (Condon-Shortley):
       m > 0 : (Y^{-m} + (-1)^m Y^{m}) / sqrt(2)
       m = 0 : Y^0
       m < 0 : i (Y^{m} - (-1)^m Y^{-m}) / sqrt(2)
   With this choice l = 1 is proportional to (y, z, x).
3. ``real_cg(l1, l2, l3)``: C[m1,m2,m3] = sum_{a,b,c} Q1[m1,a] Q2[m2,b] conj(Q3[m3,c]) <l1 a l2 b|l3 c>.
   The result is purely real when l1+l2+l3 is even and purely imaginary when odd; the non-zero
   part is kept.  Then the canonical sign: the first entry (row-major in m1, m2, m3) whose
   magnitude exceeds 1e-9 is made positive.

Normalisation: unitary, sum_{m1,m2} C[m1,m2,m3] C[m1,m2,m3'] = delta(m3,m3'), with no extra
path factor.  The pages ("An Efficient Sparse Kernel Generator for O(3)-Equivariant Deep
Networks", abstract: the CG tensor product contracts two dense vectors with a structured sparse
tensor; its code samples name a real/complex basis change and a Wigner 3j routine) fix neither
the phase nor the normalisation, so this is the plainest reading.
"""

from __future__ import annotations

from fractions import Fraction
from functools import lru_cache
from math import factorial, sqrt

import numpy as np


def _f(n: int) -> int:
    return factorial(n)


@lru_cache(maxsize=None)
def complex_cg(l1: int, m1: int, l2: int, m2: int, l3: int, m3: int) -> float:
    """<l1 m1 l2 m2 | l3 m3>, Racah's closed form, Condon-Shortley phase."""
    if m1 + m2 != m3:
        return 0.0
    if not (abs(l1 - l2) <= l3 <= l1 + l2):
        return 0.0
    if abs(m1) > l1 or abs(m2) > l2 or abs(m3) > l3:
        return 0.0
    pref = Fraction(
        (2 * l3 + 1) * _f(l3 + l1 - l2) * _f(l3 - l1 + l2) * _f(l1 + l2 - l3),
        _f(l1 + l2 + l3 + 1),
    ) * (
        _f(l3 + m3) * _f(l3 - m3) * _f(l1 - m1) * _f(l1 + m1) * _f(l2 - m2) * _f(l2 + m2)
    )
    s = Fraction(0)
    for k in range(0, l1 + l2 + l3 + 2):
        args = (
            k,
            l1 + l2 - l3 - k,
            l1 - m1 - k,
            l2 + m2 - k,
            l3 - l2 + m1 + k,
            l3 - l1 - m2 + k,
        )
        if min(args) < 0:
            continue
        den = 1
        for a in args:
            den *= _f(a)
        s += Fraction((-1) ** k, den)
    if s == 0:
        return 0.0
    # value = sqrt(pref) * s, computed as sign(s) * sqrt(pref * s^2) with one rounding of the
    # exact rational before the root.
    v2 = pref * s * s
    return (1.0 if s > 0 else -1.0) * sqrt(float(v2))


def real_basis(l: int) -> np.ndarray:
    """Q_l, (2l+1) x (2l+1) complex unitary; row index m+l, column index m'+l."""
    d = 2 * l + 1
    q = np.zeros((d, d), dtype=np.complex128)
    r2 = 1.0 / sqrt(2.0)
    for m in range(-l, l + 1):
        row = m + l
        if m > 0:
            q[row, -m + l] += r2
            q[row, m + l] += ((-1) ** m) * r2
        elif m == 0:
            q[row, l] = 1.0
        else:
            q[row, m + l] += 1j * r2
            q[row, -m + l] += -1j * ((-1) ** m) * r2
    return q


def complex_cg_tensor(l1: int, l2: int, l3: int) -> np.ndarray:
    t = np.zeros((2 * l1 + 1, 2 * l2 + 1, 2 * l3 + 1))
    for a in range(-l1, l1 + 1):
        for b in range(-l2, l2 + 1):
            c = a + b
            if -l3 <= c <= l3:
                t[a + l1, b + l2, c + l3] = complex_cg(l1, a, l2, b, l3, c)
    return t


@lru_cache(maxsize=None)
def _real_cg_cached(l1: int, l2: int, l3: int) -> np.ndarray:
    cc = complex_cg_tensor(l1, l2, l3)
    q1, q2, q3 = real_basis(l1), real_basis(l2), real_basis(l3)
    cr = np.einsum("ia,jb,kc,abc->ijk", q1, q2, np.conj(q3), cc)
    if (l1 + l2 + l3) % 2 == 0:
        keep, drop = cr.real, cr.imag
    else:
        keep, drop = cr.imag, cr.real
    if np.max(np.abs(drop)) > 1e-12:
        raise AssertionError(f"real CG ({l1},{l2},{l3}) is not purely real/imaginary")
    c = np.array(keep, dtype=np.float64)
    c[np.abs(c) < 1e-15] = 0.0
    flat = c.reshape(-1)
    nz = np.nonzero(np.abs(flat) > 1e-9)[0]
    if nz.size and flat[nz[0]] < 0:
        c = -c
    c.setflags(write=False)
    return c


def real_cg(l1: int, l2: int, l3: int) -> np.ndarray:
    """Real coupling tensor C[m1, m2, m3] (indices 0..2l), canonical sign, unitary."""
    if not (abs(l1 - l2) <= l3 <= l1 + l2):
        raise ValueError(f"({l1},{l2},{l3}) violates the triangle rule")
    return _real_cg_cached(l1, l2, l3).copy()
