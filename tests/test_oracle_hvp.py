"""Pin of the oracle's double backward: central finite differences of the VJP.

The VJP (dx, dY, dw) is linear in each of x, Y, w and g separately, so a central difference of
L2 = <ax, dx> + <aY, dY> + <aw, dw> along any coordinate is exact up to rounding for any step.
This checks the substitution identity used by oracle.hvp without relying on it."""
import numpy as np
import pytest

from oracle import conv, graph, hvp, paths, sh
from clebsch_gordan_tensor_receiver_gb300 import workloads


def _problem(irx, irs, lo, N, seed):
    rng = np.random.default_rng(seed)
    lay = paths.layout(irx, irs, lo)
    recv, src = workloads.random_degree_graph(N, rng.integers(0, 4, size=N), rng)
    off = graph.recv_offsets(recv, N)
    lsh = int(irs.split("+")[-1].split("x")[1][:-1])
    Y = sh.real_sh(workloads.unit_vectors(src.size, rng), lsh)
    x = rng.standard_normal((N, lay.mul, lay.dim_x))
    w = rng.standard_normal((src.size, len(lay.paths), lay.mul))
    g = rng.standard_normal((N, lay.mul, lay.dim_out))
    ax, aY, aw = (rng.standard_normal(a.shape) for a in (x, Y, w))
    return lay, off, src, x, Y, w, g, ax, aY, aw


@pytest.mark.parametrize("irx,irs,lo", [("2x0e+2x1o", "1x0e+1x1o+1x2e", 2),
                                        ("2x1o+2x2e", "1x0e+1x1o+1x2e+1x3o", 3)])
def test_hvp_matches_finite_differences_of_the_vjp(irx, irs, lo):
    N = 5
    lay, off, src, x, Y, w, g, ax, aY, aw = _problem(irx, irs, lo, N, 21)

    def L2(x_, Y_, w_, g_):
        dY, dw = conv.bwd_edges(lay, off, src, x_, Y_, w_, g_)
        dx = conv.bwd_dx(lay, off, src, Y_, w_, g_, N)
        return float((ax * dx).sum() + (aY * dY).sum() + (aw * dw).sum())

    gg, gx, gY, gw = hvp.hvp(lay, off, src, x, Y, w, g, ax, aY, aw, N)
    h = 0.5
    for name, arr, grad in (("g", g, gg), ("x", x, gx), ("Y", Y, gY), ("w", w, gw)):
        fd = np.zeros_like(arr)
        it = np.nditer(arr, flags=["multi_index"])
        for _ in it:
            i = it.multi_index
            args = {"x": x, "Y": Y, "w": w, "g": g}
            a = arr.copy(); a[i] += h
            args[name] = a
            fp = L2(args["x"], args["Y"], args["w"], args["g"])
            a = arr.copy(); a[i] -= h
            args[name] = a
            fm = L2(args["x"], args["Y"], args["w"], args["g"])
            fd[i] = (fp - fm) / (2 * h)
        np.testing.assert_allclose(grad, fd, atol=1e-10, err_msg=name)


def test_hvp_none_cotangents_are_zero():
    N = 4
    lay, off, src, x, Y, w, g, ax, aY, aw = _problem("2x0e+2x1o", "1x0e+1x1o", 1, N, 3)
    full = hvp.hvp(lay, off, src, x, Y, w, g, ax, None, None, N)
    zeros = hvp.hvp(lay, off, src, x, Y, w, g, ax, np.zeros_like(Y), np.zeros_like(w), N)
    for a, b in zip(full, zeros):
        assert np.array_equal(a, b)
