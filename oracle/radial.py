"""Radial weights computed from edge lengths, and the convolution that uses them, fp64 (test
infrastructure only).

"Receiver-streaming convolutions for channel-wise UVU tensor products" (replies) notes that the
convolution's radial weights are materialised by a separate network before the kernel runs, and
names fusing that network into the convolution as a further step; the page does not give the
network.  Reading taken: the radial network of MACE-style potentials, an edge length r expanded
in n_basis spherical Bessel functions of order zero with a polynomial cutoff envelope, followed by
a fully connected network with SiLU activations and no biases:

    b_n(r) = sqrt(2 / r_cut) * sin(n pi r / r_cut) / r * f(r / r_cut),   n = 1 .. n_basis
    f(s)   = 1 - (p+1)(p+2)/2 s^p + p(p+2) s^(p+1) - p(p+1)/2 s^(p+2)  for s < 1, else 0
    a_0 = b,   a_i = silu(a_(i-1) W_i)  (i = 1 .. L),   h = a_L
    w[e, p, u] = sum_k h[e, k] W_last[k, p, u]

with silu(v) = v / (1 + exp(-v)).  The envelope is the polynomial that equals 1 at s = 0 and
whose value and first two derivatives vanish at s = 1, so an edge at or beyond the cutoff gets
zero weights.  Any scaling of the layers (1/sqrt(fan-in) and the like) is folded into the weight
matrices, which are inputs.

``hidden`` computes h, ``weights`` the per-edge weights from h, and ``conv_fwd`` the
convolution of the oracle's ``conv.fwd`` with those weights: the result the fused kernel must
reproduce without materialising w.  ``hidden_vjp`` and ``weights_vjp`` are the reverse pass: the
gradients of <dh, h> with respect to the edge lengths (forces) and the layers, and of <dw, w>
with respect to h and W_last.
"""

from __future__ import annotations

import numpy as np

from . import conv as _conv


def envelope(s, p: int):
    """Polynomial cutoff f(s) of order p: 1 at s = 0; f, f', f'' = 0 at s = 1; 0 for s >= 1."""
    s = np.asarray(s, dtype=np.float64)
    f = 1.0 - (p + 1) * (p + 2) / 2.0 * s**p + p * (p + 2) * s ** (p + 1) - p * (p + 1) / 2.0 * s ** (p + 2)
    return np.where(s < 1.0, f, 0.0)


def bessel_basis(r, r_cut: float, n_basis: int):
    """b[e, n-1] = sqrt(2/r_cut) sin(n pi r_e / r_cut) / r_e for n = 1 .. n_basis (no envelope)."""
    r = np.asarray(r, dtype=np.float64)[:, None]
    n = np.arange(1, n_basis + 1, dtype=np.float64)[None, :]
    return np.sqrt(2.0 / r_cut) * np.sin(n * np.pi * r / r_cut) / r


def silu(v):
    v = np.asarray(v, dtype=np.float64)
    return v / (1.0 + np.exp(-v))


def hidden(r, r_cut: float, p_env: int, layers):
    """h [E][H_L]: the enveloped basis through the SiLU layers W_1 .. W_L ([H_(i-1)][H_i] each)."""
    n_basis = np.asarray(layers[0]).shape[0]
    a = bessel_basis(r, r_cut, n_basis) * envelope(np.asarray(r, dtype=np.float64) / r_cut, p_env)[:, None]
    for W in layers:
        a = silu(a @ np.asarray(W, dtype=np.float64))
    return a


def weights(h, w_last):
    """w [E][P][U] = h [E][H] contracted with W_last [H][P][U]."""
    return np.einsum("ek,kpu->epu", np.asarray(h, dtype=np.float64), np.asarray(w_last, dtype=np.float64), optimize=True)


def conv_fwd(lay, recv_offsets, src, x, Y, h, w_last, receivers=None, nthreads=None):
    """The convolution with radial weights w = weights(h, W_last): out [N][U][D_out], or the rows
    of ``receivers`` (then only their edges' weights are formed)."""
    off = np.asarray(recv_offsets, dtype=np.int64)
    if receivers is None:
        receivers = np.arange(off.size - 1)
    receivers = np.asarray(receivers, dtype=np.int64)
    segs = [np.arange(off[r], off[r + 1]) for r in receivers]
    eidx = np.concatenate(segs) if segs else np.zeros(0, np.int64)
    loff = np.zeros(receivers.size + 1, dtype=np.int64)
    np.cumsum([sg.size for sg in segs], out=loff[1:])
    w = weights(np.asarray(h)[eidx], w_last)
    return _conv.fwd(lay, loff, np.asarray(src)[eidx], x, np.asarray(Y)[eidx], w, nthreads=nthreads)


# ----------------------------------------------------------------------------------- gradients
#
# The reverse pass of the same network, for training the radial layers and for forces (the edge
# lengths' gradient).  Each step is the chain rule through the forward definition above:
#   d/dr b_n(r)      = sqrt(2/r_cut) (n pi / r_cut cos(n pi r / r_cut) / r - sin(n pi r / r_cut) / r^2)
#   d/dr f(r/r_cut)  = f'(s) / r_cut,  f'(s) = -p(p+1)(p+2)/2 s^(p-1) + p(p+1)(p+2) s^p - p(p+1)(p+2)/2 s^(p+1)
#                      for s < 1 (0 beyond)
#   silu'(v)         = sigma(v) (1 + v (1 - sigma(v))),  sigma(v) = 1 / (1 + exp(-v))


def envelope_deriv(s, p: int):
    """f'(s) of the polynomial cutoff (0 for s >= 1)."""
    s = np.asarray(s, dtype=np.float64)
    c = p * (p + 1) * (p + 2) / 2.0
    d = -c * s ** (p - 1) + 2.0 * c * s**p - c * s ** (p + 1)
    return np.where(s < 1.0, d, 0.0)


def bessel_basis_deriv(r, r_cut: float, n_basis: int):
    """d b[e, n-1] / d r_e."""
    r = np.asarray(r, dtype=np.float64)[:, None]
    n = np.arange(1, n_basis + 1, dtype=np.float64)[None, :]
    k = n * np.pi / r_cut
    return np.sqrt(2.0 / r_cut) * (k * np.cos(k * r) / r - np.sin(k * r) / r**2)


def silu_deriv(v):
    v = np.asarray(v, dtype=np.float64)
    sg = 1.0 / (1.0 + np.exp(-v))
    return sg * (1.0 + v * (1.0 - sg))


def hidden_vjp(r, r_cut: float, p_env: int, layers, dh):
    """Gradients of <dh, hidden(r)>: (dr [E], [dW_1 .. dW_L] shaped as the layers)."""
    r = np.asarray(r, dtype=np.float64)
    n_basis = np.asarray(layers[0]).shape[0]
    b = bessel_basis(r, r_cut, n_basis)
    f = envelope(r / r_cut, p_env)
    acts, pre = [b * f[:, None]], []
    for W in layers:
        z = acts[-1] @ np.asarray(W, dtype=np.float64)
        pre.append(z)
        acts.append(silu(z))
    g = np.asarray(dh, dtype=np.float64)
    dWs = [None] * len(layers)
    for i in range(len(layers) - 1, -1, -1):
        dz = g * silu_deriv(pre[i])
        dWs[i] = acts[i].T @ dz
        g = dz @ np.asarray(layers[i], dtype=np.float64).T
    # g = d/d a_0, a_0 = b(r) f(r / r_cut)
    da0_dr = bessel_basis_deriv(r, r_cut, n_basis) * f[:, None] + b * (envelope_deriv(r / r_cut, p_env) / r_cut)[:, None]
    dr = (g * da0_dr).sum(axis=1)
    return dr, dWs


def weights_vjp(h, w_last, dw):
    """Gradients of <dw, weights(h, W_last)>: (dh [E][H], dW_last [H][P][U])."""
    h = np.asarray(h, dtype=np.float64)
    w_last = np.asarray(w_last, dtype=np.float64)
    dw = np.asarray(dw, dtype=np.float64)
    dh = np.einsum("epu,kpu->ek", dw, w_last, optimize=True)
    dwl = np.einsum("ek,epu->kpu", h, dw, optimize=True)
    return dh, dwl
