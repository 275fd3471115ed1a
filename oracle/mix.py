"""Channel mixing that reduces a factorised UVW convolution to the UVU one, fp64 (test
infrastructure only).

"Receiver-streaming convolutions for channel-wise UVU tensor products" (replies) says the
streaming kernel serves UVU convolutions "including UVW cases that can be reduced to UVU", and
does not say which.  Reading taken: a UVW path (second operand of multiplicity 1, as the edge
harmonics are) whose per-edge weights factor into per-edge channel weights and a channel mixing
shared by all edges,

    W_e[p,u,w] = w[e,p,u] * M[p,u,w],

so that, the mixing being linear and the same on every edge, it commutes with the sum over a
receiver's edges:

    out_uvw[r,w,ooff(p)+m3] = sum_u M[p,u,w] * out_uvu[r,u,ooff(p)+m3].

``fwd`` and ``vjp`` are that per-path contraction and its gradients, each one ``numpy.einsum``
call (a matrix product over the channel index, left to numpy's contraction routine);
``uvw_conv_brute`` is the UVW convolution with the factorised weights summed
edge by edge (no reduction), which pins the reading.
"""

from __future__ import annotations

import numpy as np

from . import cg as _cg


def _so(p):
    return slice(p.ooff, p.ooff + 2 * p.l3 + 1)


def fwd(lay, inp, M):
    """inp [N][U][D_out], M [P][U][W] -> out [N][W][D_out]."""
    inp, M = np.asarray(inp, dtype=np.float64), np.asarray(M, dtype=np.float64)
    out = np.zeros((inp.shape[0], M.shape[2], lay.dim_out))
    for i, p in enumerate(lay.paths):
        out[:, :, _so(p)] = np.einsum("nuk,uw->nwk", inp[:, :, _so(p)], M[i], optimize=True)
    return out


def vjp(lay, inp, M, g):
    """(d_inp [N][U][D_out], dM [P][U][W]) for the cotangent g [N][W][D_out] of fwd."""
    inp, M, g = (np.asarray(a, dtype=np.float64) for a in (inp, M, g))
    d_inp, dM = np.zeros_like(inp), np.zeros_like(M)
    for i, p in enumerate(lay.paths):
        d_inp[:, :, _so(p)] = np.einsum("nwk,uw->nuk", g[:, :, _so(p)], M[i], optimize=True)
        dM[i] = np.einsum("nuk,nwk->uw", inp[:, :, _so(p)], g[:, :, _so(p)], optimize=True)
    return d_inp, dM


def uvw_conv_brute(lay, recv, src, x, Y, w, M, n_nodes):
    """The UVW convolution with weights W_e[p,u,w] = w[e,p,u] M[p,u,w], one edge at a time:
    out[r,w,ooff+m3] = sum_{e: recv(e)=r} sum_u W_e[p,u,w] sum_{m1,m2} C x[src(e),u,m1] Y[e,m2]."""
    x, Y, w, M = (np.asarray(a, dtype=np.float64) for a in (x, Y, w, M))
    out = np.zeros((n_nodes, M.shape[2], lay.dim_out))
    for i, p in enumerate(lay.paths):
        C = _cg.real_cg(p.l1, p.l2, p.l3)
        sx = slice(p.xoff, p.xoff + 2 * p.l1 + 1)
        sy = slice(p.yoff, p.yoff + 2 * p.l2 + 1)
        for e in range(len(src)):
            t = np.einsum("ui,j,ijk->uk", x[src[e], :, sx], Y[e, sy], C)   # [U][d3]
            We = w[e, i, :, None] * M[i]                                  # [U][W]
            out[recv[e], :, _so(p)] += np.einsum("uw,uk->wk", We, t)
    return out
