"""Batched (non-convolution) channel-wise CG tensor product, fp64 (test infrastructure only).

"An Efficient Sparse Kernel Generator for O(3)-Equivariant Deep Networks" (abstract) describes
the CG tensor product on its own, before its fusion with a graph convolution: two dense feature
vectors contracted with a structured sparse tensor, repeated over a batch.  In the channel-wise
(UVU) form of "Receiver-streaming convolutions for channel-wise UVU tensor products" (opening
post), with one sample b in place of one edge and no aggregation over a graph:

    z[b,u,ooff(p)+m3] = w[b,p,u] * sum_{m1,m2} C^p[m1,m2,m3] x[b,u,xoff(p)+m1] y[b,yoff(p)+m2]

Reading taken where the pages are silent: the weights are either per sample, w [B][P][U] (as
the per-edge weights of the convolution), or shared by the whole batch, w [P][U] (the layer's
own weights); x [B][U][D_x], y [B][D_Y] and z [B][U][D_out] follow the convolution's layouts.
For shared weights dw is the sum over the batch of the per-sample gradients.

Each function is the definition written out per path with ``numpy.einsum`` on the dense real CG
block of ``oracle.cg``; nothing is fused or reordered beyond the sum itself.
"""

from __future__ import annotations

import numpy as np

from . import cg as _cg


def _blocks(lay, p):
    d1, d2, d3 = 2 * p.l1 + 1, 2 * p.l2 + 1, 2 * p.l3 + 1
    return (slice(p.xoff, p.xoff + d1), slice(p.yoff, p.yoff + d2), slice(p.ooff, p.ooff + d3))


def _wp(w, i, shared):
    """Weights of path i as [B or 1][U]."""
    return w[i][None, :] if shared else w[:, i, :]


def fwd(lay, x, y, w, shared=False):
    """z [B][U][D_out]."""
    x, y, w = (np.asarray(a, dtype=np.float64) for a in (x, y, w))
    B, U = x.shape[0], lay.mul
    z = np.zeros((B, U, lay.dim_out))
    for i, p in enumerate(lay.paths):
        C = _cg.real_cg(p.l1, p.l2, p.l3)
        sx, sy, so = _blocks(lay, p)
        t = np.einsum("bui,bj,ijk->buk", x[:, :, sx], y[:, sy], C)
        z[:, :, so] = _wp(w, i, shared)[:, :, None] * t
    return z


def vjp(lay, x, y, w, g, shared=False):
    """(dx [B][U][D_x], dy [B][D_Y], dw [B][P][U] or [P][U] when shared) for the cotangent g of z."""
    x, y, w, g = (np.asarray(a, dtype=np.float64) for a in (x, y, w, g))
    B, U = x.shape[0], lay.mul
    dx, dy = np.zeros_like(x), np.zeros_like(y)
    dw = np.zeros((B, len(lay.paths), U))
    for i, p in enumerate(lay.paths):
        C = _cg.real_cg(p.l1, p.l2, p.l3)
        sx, sy, so = _blocks(lay, p)
        xs, ys, gs = x[:, :, sx], y[:, sy], g[:, :, so]
        wp = _wp(w, i, shared)
        dx[:, :, sx] += np.einsum("bu,bj,ijk,buk->bui", np.broadcast_to(wp, (B, U)), ys, C, gs)
        dy[:, sy] += np.einsum("bu,bui,ijk,buk->bj", np.broadcast_to(wp, (B, U)), xs, C, gs)
        dw[:, i, :] = np.einsum("bui,bj,ijk,buk->bu", xs, ys, C, gs)
    return dx, dy, (dw.sum(axis=0) if shared else dw)
