"""Real Wigner-D matrices for the equivariance pins (test infrastructure only).

D^l(R) is defined by Y_l(R r) = D^l(R) Y_l(r) for every unit vector r, with Y_l the oracle's
real SH.  It is obtained by a least-squares fit over many sample directions, which needs no
Euler-angle convention; the fit residual is returned so a test can check that the relation holds
exactly (to rounding).
"""

from __future__ import annotations

import numpy as np

from .sh import real_sh


def random_rotation(rng: np.random.Generator) -> np.ndarray:
    q = rng.standard_normal(4)
    q /= np.linalg.norm(q)
    a, b, c, d = q
    return np.array([
        [a * a + b * b - c * c - d * d, 2 * (b * c - a * d), 2 * (b * d + a * c)],
        [2 * (b * c + a * d), a * a - b * b + c * c - d * d, 2 * (c * d - a * b)],
        [2 * (b * d - a * c), 2 * (c * d + a * b), a * a - b * b - c * c + d * d],
    ])


def wigner_d(l: int, R: np.ndarray, n_samples: int = 200, seed: int = 7):
    """(D^l(R), max residual of Y_l(R r) - D Y_l(r) over the samples)."""
    rng = np.random.default_rng(seed)
    v = rng.standard_normal((n_samples, 3))
    v /= np.linalg.norm(v, axis=1, keepdims=True)
    sl = slice(l * l, (l + 1) * (l + 1))
    A = real_sh(v, l)[:, sl]
    B = real_sh(v @ R.T, l)[:, sl]
    # rows: B_i = D A_i  ->  A D^T = B
    DT, *_ = np.linalg.lstsq(A, B, rcond=None)
    D = DT.T
    return D, float(np.max(np.abs(A @ D.T - B)))
