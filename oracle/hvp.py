"""Double backward (Hessian-vector product) of the UVU convolution, fp64 (test infrastructure only).

"Receiver-streaming convolutions for channel-wise UVU tensor products" (opening post, results
table: HVP column; the standard HVP ran out of memory on the largest case) and "An Efficient
Sparse Kernel Generator for O(3)-Equivariant Deep Networks" (abstract: higher partial derivatives
for interatomic forces) both treat the derivative of the VJP.  With T(g, x, Y, w) = <g, F(x, Y, w)>
the VJP is (dx, dY, dw) = (dT/dx, dT/dY, dT/dw).  Given cotangents (ax, aY, aw) of the VJP
outputs, the scalar

    L2 = <ax, dx> + <aY, dY> + <aw, dw>

equals T(g, ax, Y, w) + T(g, x, aY, w) + T(g, x, Y, aw) because T is linear in each argument
separately.  Its gradients are therefore forward and VJP evaluations with one argument
substituted:

    dL2/dg = F(ax, Y, w) + F(x, aY, w) + F(x, Y, aw)
    dL2/dx = dx(Y <- aY) + dx(w <- aw)
    dL2/dY = dY(x <- ax) + dY(w <- aw)
    dL2/dw = dw(x <- ax) + dw(Y <- aY)

This module evaluates exactly that with the oracle's own forward and VJP loops.  It is pinned in
tests/test_oracle_hvp.py by finite differences of the VJP, which do not use the identity.
"""

from __future__ import annotations

import numpy as np

from . import conv


def hvp(lay, recv_offsets, src, x, Y, w, g, ax, aY, aw, n_nodes):
    """(dL2/dg, dL2/dx, dL2/dY, dL2/dw) for cotangents ax, aY, aw (None = zero)."""
    x, Y, w, g = (np.asarray(a, dtype=np.float64) for a in (x, Y, w, g))
    ax = np.zeros_like(x) if ax is None else np.asarray(ax, dtype=np.float64)
    aY = np.zeros_like(Y) if aY is None else np.asarray(aY, dtype=np.float64)
    aw = np.zeros_like(w) if aw is None else np.asarray(aw, dtype=np.float64)
    gg = (conv.fwd(lay, recv_offsets, src, ax, Y, w) + conv.fwd(lay, recv_offsets, src, x, aY, w)
          + conv.fwd(lay, recv_offsets, src, x, Y, aw))
    gx = (conv.bwd_dx(lay, recv_offsets, src, aY, w, g, n_nodes)
          + conv.bwd_dx(lay, recv_offsets, src, Y, aw, g, n_nodes))
    dY_ax, dw_ax = conv.bwd_edges(lay, recv_offsets, src, ax, Y, w, g)
    dY_aw, _ = conv.bwd_edges(lay, recv_offsets, src, x, Y, aw, g)
    _, dw_aY = conv.bwd_edges(lay, recv_offsets, src, x, aY, w, g)
    return gg, gx, dY_ax + dY_aw, dw_ax + dw_aY
