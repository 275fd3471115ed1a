"""Property tests of the oracle convolution with hypothesis: random irreps (l <= 3), random small
graphs (including receivers and senders without edges), random values.  For every draw:
- the adjoint (Euler) identities <d_out, out> = <dx, x> = <dY, Y> = <dw, w>, which hold because out
  is linear in each of x, Y, w separately;
- linearity of out in w (out(a w1 + b w2) = a out(w1) + b out(w2));
- a receiver's output depends only on its own edges (permuting the other receivers' edges leaves
  it unchanged)."""
import numpy as np
import pytest

hyp = pytest.importorskip("hypothesis")
from hypothesis import given, settings, strategies as st  # noqa: E402

from oracle import conv, graph, paths, sh  # noqa: E402


@st.composite
def problems(draw):
    lx = sorted(draw(st.sets(st.integers(0, 2), min_size=1, max_size=3)))
    ly = sorted(draw(st.sets(st.integers(0, 3), min_size=1, max_size=3)))
    lo = draw(st.integers(0, 3))
    U = draw(st.integers(1, 3))
    par = lambda l: "e" if l % 2 == 0 else "o"
    irx = "+".join(f"{U}x{l}{par(l)}" for l in lx)
    irs = "+".join(f"1x{l}{par(l)}" for l in ly)
    lay = paths.layout(irx, irs, lo)
    if not lay.paths:
        return None
    N = draw(st.integers(1, 5))
    deg = draw(st.lists(st.integers(0, 3), min_size=N, max_size=N))
    seed = draw(st.integers(0, 2 ** 31 - 1))
    rng = np.random.default_rng(seed)
    recv = np.repeat(np.arange(N, dtype=np.int32), deg)
    src = np.concatenate([np.sort(rng.integers(0, N, size=d)) for d in deg]).astype(np.int32) if recv.size else np.zeros(0, np.int32)
    Y = rng.standard_normal((src.size, lay.dim_y))
    x = rng.standard_normal((N, U, lay.dim_x))
    w = rng.standard_normal((src.size, len(lay.paths), U))
    g = rng.standard_normal((N, U, lay.dim_out))
    return lay, recv, src, x, Y, w, g, N, rng


@settings(max_examples=40, deadline=None)
@given(problems())
def test_adjoint_identities_and_linearity(prob):
    if prob is None:
        return
    lay, recv, src, x, Y, w, g, N, rng = prob
    off = graph.recv_offsets(recv, N)
    out = conv.fwd(lay, off, src, x, Y, w)
    dY, dw = conv.bwd_edges(lay, off, src, x, Y, w, g)
    dx = conv.bwd_dx(lay, off, src, Y, w, g, N)
    ref = float((g * out).sum())
    scale = 1.0 + abs(ref) + float(np.abs(g).sum() * np.abs(out).max(initial=0.0))
    for v in ((dx * x).sum(), (dY * Y).sum(), (dw * w).sum()):
        assert abs(float(v) - ref) <= 1e-10 * scale
    w2 = rng.standard_normal(w.shape)
    lin = conv.fwd(lay, off, src, x, Y, 2.0 * w - 3.0 * w2)
    np.testing.assert_allclose(lin, 2.0 * out - 3.0 * conv.fwd(lay, off, src, x, Y, w2), atol=1e-10 * scale)


@settings(max_examples=25, deadline=None)
@given(problems())
def test_receivers_depend_only_on_their_edges(prob):
    if prob is None:
        return
    lay, recv, src, x, Y, w, g, N, rng = prob
    off = graph.recv_offsets(recv, N)
    out = conv.fwd(lay, off, src, x, Y, w)
    # scramble the values on every edge outside receiver 0's segment
    Y2, w2 = Y.copy(), w.copy()
    e0, e1 = off[0], off[1]
    other = np.r_[0:e0, e1:src.size]
    Y2[other] = rng.standard_normal(Y2[other].shape)
    w2[other] = rng.standard_normal(w2[other].shape)
    out2 = conv.fwd(lay, off, src, x, Y2, w2)
    np.testing.assert_array_equal(out2[0], out[0])
