"""Real spherical harmonics for the oracle (test infrastructure only).

Component normalisation: sum_m Y_{l,m}(r)^2 = 2l+1 for every unit vector r, so Y_0 = 1 and
Y_1 = sqrt(3) (y, z, x).  The real basis is the one of ``oracle.cg.real_basis`` (Condon-Shortley
complex harmonics, m > 0 -> cos(m phi), m < 0 -> sin(|m| phi)); the intertwining pins in the
tests tie this SH basis to the CG basis.

Evaluation uses the associated-Legendre three-term recursion on P_l^m(z) / (1 - z^2)^{m/2}
(a polynomial in z) times Re / Im of (x + i y)^m, so no angle is ever formed:

    Pb[m][m]   = (2m-1)!!
    Pb[m+1][m] = (2m+1) z Pb[m][m]
    Pb[l][m]   = ((2l-1) z Pb[l-1][m] - (l+m-1) Pb[l-2][m]) / (l-m)

    Y_{l,0}  = sqrt(2l+1) Pb[l][0]
    Y_{l,+m} = sqrt(2 (2l+1) (l-m)!/(l+m)!) Pb[l][m] Re (x+iy)^m
    Y_{l,-m} = sqrt(2 (2l+1) (l-m)!/(l+m)!) Pb[l][m] Im (x+iy)^m

The layout is Y[..., l*l + l + m] for l = 0..lmax, m = -l..l.  The pages ask for "real spherical
harmonics, component-normalised" of unit edge vectors and fix nothing else.
"""

from __future__ import annotations

from math import factorial, sqrt

import numpy as np


def real_sh(vectors: np.ndarray, lmax: int) -> np.ndarray:
    """Component-normalised real SH of unit vectors, shape (n, (lmax+1)^2), fp64."""
    v = np.asarray(vectors, dtype=np.float64)
    x, y, z = v[:, 0], v[:, 1], v[:, 2]
    n = v.shape[0]
    out = np.zeros((n, (lmax + 1) ** 2), dtype=np.float64)
    # Pb[l][m] as arrays over the n points
    pb = [[None] * (lmax + 1) for _ in range(lmax + 1)]
    for m in range(lmax + 1):
        dfact = 1.0
        for k in range(1, 2 * m, 2):
            dfact *= k
        pb[m][m] = np.full(n, dfact)
        if m + 1 <= lmax:
            pb[m + 1][m] = (2 * m + 1) * z * pb[m][m]
        for l in range(m + 2, lmax + 1):
            pb[l][m] = ((2 * l - 1) * z * pb[l - 1][m] - (l + m - 1) * pb[l - 2][m]) / (l - m)
    # (x + i y)^m
    xy = [np.ones(n, dtype=np.complex128)]
    for m in range(1, lmax + 1):
        xy.append(xy[-1] * (x + 1j * y))
    for l in range(lmax + 1):
        base = l * l + l
        out[:, base] = sqrt(2 * l + 1) * pb[l][0]
        for m in range(1, l + 1):
            c = sqrt(2.0 * (2 * l + 1) * factorial(l - m) / factorial(l + m))
            out[:, base + m] = c * pb[l][m] * xy[m].real
            out[:, base - m] = c * pb[l][m] * xy[m].imag
    return out
