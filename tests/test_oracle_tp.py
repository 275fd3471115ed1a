"""Pins of the batched tensor-product oracle (oracle.tp).

- closed forms for l <= 1 written with numpy dot / cross products (the textbook real-basis forms
  of the l=1 x l=1 coupling, components ordered (y, z, x)) and the identity paths;
- central finite differences of the forward for the VJP (exact up to rounding: the product is
  linear in each of x, y, w), for per-sample and shared weights;
- the convolution oracle on a graph where every receiver has exactly one edge from itself;
- equivariance under random rotations (Wigner-D fitted from SH samples).
"""
import numpy as np
import pytest

from oracle import conv, graph, paths, sh, tp, wigner

S2, S3, S6 = np.sqrt(2.0), np.sqrt(3.0), np.sqrt(6.0)


def _xyz(v):  # (y, z, x) -> (x, y, z)
    return np.stack([v[..., 2], v[..., 0], v[..., 1]], axis=-1)


def _yzx(v):  # (x, y, z) -> (y, z, x)
    return np.stack([v[..., 1], v[..., 2], v[..., 0]], axis=-1)


def test_l1_closed_forms_per_sample():
    rng = np.random.default_rng(0)
    lay = paths.layout("3x1o", "1x1o", 2)
    assert [(p.l1, p.l2, p.l3) for p in lay.paths] == [(1, 1, 0), (1, 1, 1), (1, 1, 2)]
    B, U = 5, 3
    x, y = rng.standard_normal((B, U, 3)), rng.standard_normal((B, 3))
    w = rng.standard_normal((B, 3, U))
    z = tp.fwd(lay, x, y, w)
    a, b = _xyz(x), _xyz(y)[:, None, :]
    ax_, ay_, az_ = a[..., 0], a[..., 1], a[..., 2]
    bx, by, bz = b[..., 0], b[..., 1], b[..., 2]
    dot = (a * b).sum(-1) / S3
    cross = _yzx(np.cross(a, np.broadcast_to(b, a.shape))) / S2
    sym = np.stack([-(ay_ * bx + ax_ * by) / S2, -(ay_ * bz + az_ * by) / S2,
                    (ax_ * bx + ay_ * by - 2 * az_ * bz) / S6, -(az_ * bx + ax_ * bz) / S2,
                    (ay_ * by - ax_ * bx) / S2], axis=-1)
    np.testing.assert_allclose(z[:, :, 0], w[:, 0, :] * dot, atol=1e-14)
    np.testing.assert_allclose(z[:, :, 1:4], w[:, 1, :, None] * cross, atol=1e-14)
    np.testing.assert_allclose(z[:, :, 4:9], w[:, 2, :, None] * sym, atol=1e-14)


def test_identity_paths_shared_weights():
    rng = np.random.default_rng(1)
    lay = paths.layout("2x0e", "1x0e+1x1o+1x2e", 2)
    B = 4
    x, y, w = rng.standard_normal((B, 2, 1)), rng.standard_normal((B, 9)), rng.standard_normal((3, 2))
    z = tp.fwd(lay, x, y, w, shared=True)
    for i, sl in enumerate((slice(0, 1), slice(1, 4), slice(4, 9))):
        np.testing.assert_allclose(z[:, :, sl], w[i][None, :, None] * x[:, :, :1] * y[:, None, sl], atol=1e-14)


@pytest.mark.parametrize("shared", [False, True])
def test_vjp_matches_central_differences(shared):
    rng = np.random.default_rng(2)
    lay = paths.layout("2x0e+2x1o", "1x0e+1x1o+1x2e", 2)
    B, U, P = 3, 2, len(lay.paths)
    x, y = rng.standard_normal((B, U, lay.dim_x)), rng.standard_normal((B, lay.dim_y))
    w = rng.standard_normal((P, U) if shared else (B, P, U))
    g = rng.standard_normal((B, U, lay.dim_out))
    dx, dy, dw = tp.vjp(lay, x, y, w, g, shared)
    h = 0.5
    for name, arr, grad in (("x", x, dx), ("y", y, dy), ("w", w, dw)):
        fd = np.zeros_like(arr)
        for i in np.ndindex(arr.shape):
            args = {"x": x, "y": y, "w": w}
            a = arr.copy(); a[i] += h; args[name] = a
            fp = (tp.fwd(lay, args["x"], args["y"], args["w"], shared) * g).sum()
            a = arr.copy(); a[i] -= h; args[name] = a
            fm = (tp.fwd(lay, args["x"], args["y"], args["w"], shared) * g).sum()
            fd[i] = (fp - fm) / (2 * h)
        np.testing.assert_allclose(grad, fd, atol=1e-11, err_msg=name)


def test_equals_the_convolution_on_a_self_loop_graph():
    rng = np.random.default_rng(3)
    lay = paths.layout("4x0e+4x1o+4x2e", "1x0e+1x1o+1x2e+1x3o", 3)
    B, U, P = 6, 4, len(lay.paths)
    x = rng.standard_normal((B, U, lay.dim_x))
    y = sh.real_sh(rng.standard_normal((B, 3)), 3)
    w, g = rng.standard_normal((B, P, U)), rng.standard_normal((B, U, lay.dim_out))
    recv = np.arange(B, dtype=np.int32)
    off = graph.recv_offsets(recv, B)
    np.testing.assert_allclose(tp.fwd(lay, x, y, w), conv.fwd(lay, off, recv, x, y, w), atol=1e-13)
    dx, dy, dw = tp.vjp(lay, x, y, w, g)
    dY_c, dw_c = conv.bwd_edges(lay, off, recv, x, y, w, g)
    np.testing.assert_allclose(dy, dY_c, atol=1e-13)
    np.testing.assert_allclose(dw, dw_c, atol=1e-13)
    np.testing.assert_allclose(dx, conv.bwd_dx(lay, off, recv, y, w, g, B), atol=1e-13)


def test_rotation_equivariance():
    rng = np.random.default_rng(4)
    lay = paths.layout("3x0e+3x1o+3x2e", "1x0e+1x1o+1x2e", 2)
    B, U, P = 4, 3, len(lay.paths)
    R = wigner.random_rotation(rng)
    D = {l: wigner.wigner_d(l, R)[0] for l in range(3)}
    x, y = rng.standard_normal((B, U, lay.dim_x)), rng.standard_normal((B, lay.dim_y))
    w = rng.standard_normal((P, U))
    xr, yr = x.copy(), y.copy()
    for l, o in ((0, 0), (1, 1), (2, 4)):
        xr[:, :, o:o + 2 * l + 1] = x[:, :, o:o + 2 * l + 1] @ D[l].T
        yr[:, o:o + 2 * l + 1] = y[:, o:o + 2 * l + 1] @ D[l].T
    z, zr = tp.fwd(lay, x, y, w, True), tp.fwd(lay, xr, yr, w, True)
    for p in lay.paths:
        so = slice(p.ooff, p.ooff + 2 * p.l3 + 1)
        np.testing.assert_allclose(zr[:, :, so], z[:, :, so] @ D[p.l3].T, atol=1e-10)
