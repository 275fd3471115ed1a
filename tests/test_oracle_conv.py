"""Pins of the oracle convolution and its VJP.

* closed forms: on graphs whose features are l <= 1, every path output is a dot, cross or
  symmetric-traceless product of the sender's vector feature with the edge direction, written
  here with numpy's dot/cross (not with CG tables);
* a special case that is a library routine: the (0,0,0) path is a weighted sparse matrix
  product, checked against scipy.sparse;
* finite differences: the output is linear in each of x, Y and w separately, so central
  differences are exact up to rounding;
* adjoint (Euler) identities: <d_out, out> = <dx, x> = <dY, Y> = <dw, w>;
* rotation equivariance of out, dx, dY and invariance of dw, and the parity under inversion;
* sampling, thread-count independence and empty segments."""
import numpy as np
import pytest
import scipy.sparse as sp

from conftest import golden_rows, signed_sqrt  # noqa: F401
from oracle import conv, graph, paths, sh, wigner
from clebsch_gordan_tensor_receiver_gb300 import workloads


def small_problem(irx, irs, lmax_out, N=7, degrees=None, seed=0, U=None):
    rng = np.random.default_rng(seed)
    lay = paths.layout(irx, irs, lmax_out)
    if degrees is None:
        degrees = rng.integers(0, 5, size=N)
    recv, src = workloads.random_degree_graph(N, degrees, rng)
    off = graph.recv_offsets(recv, N)
    E = src.size
    vec = workloads.unit_vectors(E, rng)
    lsh = int(irs.split("+")[-1].split("x")[1][:-1])
    Y = sh.real_sh(vec, lsh)
    x = rng.standard_normal((N, lay.mul, lay.dim_x))
    w = rng.standard_normal((E, len(lay.paths), lay.mul))
    g = rng.standard_normal((N, lay.mul, lay.dim_out))
    return lay, off, src, vec, Y, x, w, g


def to_cart(s):  # (y, z, x) storage -> (x, y, z)
    return s[..., [2, 0, 1]]


def to_store(c):  # (x, y, z) -> (y, z, x)
    return c[..., [1, 2, 0]]


def test_closed_forms_l_le_1():
    lay, off, src, vec, Y, x, w, g = small_problem("2x0e+2x1o", "1x0e+1x1o", 2, N=6, seed=1)
    keys = [(p.l1, p.l2, p.l3) for p in lay.paths]
    assert keys == [(0, 0, 0), (0, 1, 1), (1, 0, 1), (1, 1, 0), (1, 1, 1), (1, 1, 2)]
    out = conv.fwd(lay, off, src, x, Y, w)
    recv = graph.recv_of_edges(off)
    want = np.zeros_like(out)
    s3 = np.sqrt(3.0)
    for e in range(src.size):
        r, s = recv[e], src[e]
        r_hat = vec[e]  # Y_1 = sqrt(3) r_hat (storage order)
        for u in range(lay.mul):
            x0, a = x[s, u, 0], to_cart(x[s, u, 1:4])
            wp = w[e, :, u]
            col = []
            col.append([wp[0] * x0 * Y[e, 0]])
            col.append(wp[1] * x0 * s3 * to_store(r_hat))
            col.append(wp[2] * Y[e, 0] * to_store(a))
            col.append([wp[3] * s3 * a.dot(r_hat) / np.sqrt(3.0)])
            col.append(wp[4] * s3 * to_store(np.cross(a, r_hat)) / np.sqrt(2.0))
            b = s3 * r_hat
            ax, ay, az = a
            bx, by, bz = b
            t = np.array([-(ay * bx + ax * by) / np.sqrt(2), -(ay * bz + az * by) / np.sqrt(2),
                          (ax * bx + ay * by - 2 * az * bz) / np.sqrt(6),
                          -(az * bx + ax * bz) / np.sqrt(2), (ay * by - ax * bx) / np.sqrt(2)])
            col.append(wp[5] * t)
            want[r, u] += np.concatenate([np.atleast_1d(c) for c in col])
    np.testing.assert_allclose(out, want, atol=1e-13)


def test_scalar_path_is_sparse_matmul():
    lay, off, src, vec, Y, x, w, g = small_problem("3x0e", "1x0e", 0, N=9, seed=2)
    Y = np.random.default_rng(9).standard_normal(Y.shape)  # any per-edge scalar
    out = conv.fwd(lay, off, src, x, Y, w)
    for u in range(3):
        A = sp.csr_matrix((w[:, 0, u] * Y[:, 0], src, off), shape=(9, 9))
        np.testing.assert_allclose(out[:, u, 0], A @ x[:, u, 0], atol=1e-13)


def _all_grads(lay, off, src, Y, x, w, g, N):
    dY, dw = conv.bwd_edges(lay, off, src, x, Y, w, g)
    dx = conv.bwd_dx(lay, off, src, Y, w, g, N)
    return dx, dY, dw


@pytest.mark.parametrize("irx,irs,lo", [("2x0e+2x1o", "1x0e+1x1o+1x2e", 2),
                                        ("2x0e+2x1o+2x2e", "1x0e+1x1o+1x2e+1x3o", 3),
                                        ("1x1o+1x2e", "1x0e+1x1o+1x2e+1x3o", 4)])
def test_vjp_finite_differences(irx, irs, lo):
    N = 5
    lay, off, src, vec, Y, x, w, g = small_problem(irx, irs, lo, N=N, seed=3)
    dx, dY, dw = _all_grads(lay, off, src, Y, x, w, g, N)

    def f(xx, YY, ww):
        return float((conv.fwd(lay, off, src, xx, YY, ww) * g).sum())

    h = 0.5  # linear in each argument: any step is exact up to rounding
    for arr, grad, name in ((x, dx, "x"), (Y, dY, "Y"), (w, dw, "w")):
        fd = np.zeros_like(arr)
        it = np.nditer(arr, flags=["multi_index"])
        for _ in it:
            i = it.multi_index
            a = arr.copy(); a[i] += h
            b = arr.copy(); b[i] -= h
            args = {"x": x, "Y": Y, "w": w}
            args[name] = a
            fp = f(args["x"], args["Y"], args["w"])
            args[name] = b
            fm = f(args["x"], args["Y"], args["w"])
            fd[i] = (fp - fm) / (2 * h)
        np.testing.assert_allclose(grad, fd, atol=1e-10, err_msg=name)


def test_adjoint_identities():
    N = 40
    lay, off, src, vec, Y, x, w, g = small_problem("4x0e+4x1o+4x2e", "1x0e+1x1o+1x2e+1x3o", 3,
                                                   N=N, seed=4,
                                                   degrees=np.full(40, 6))
    out = conv.fwd(lay, off, src, x, Y, w)
    dx, dY, dw = _all_grads(lay, off, src, Y, x, w, g, N)
    s = float((out * g).sum())
    for a, b in ((dx, x), (dY, Y), (dw, w)):
        assert float((a * b).sum()) == pytest.approx(s, rel=1e-12)


def _rotate_blocks(arr, ls, D):
    out = arr.copy()
    o = 0
    for l in ls:
        d = 2 * l + 1
        out[..., o:o + d] = arr[..., o:o + d] @ D[l].T
        o += d
    return out


def test_equivariance():
    N = 12
    lay, off, src, vec, Y, x, w, g = small_problem("3x0e+3x1o+3x2e", "1x0e+1x1o+1x2e+1x3o", 3,
                                                   N=N, seed=5)
    rng = np.random.default_rng(6)
    R = wigner.random_rotation(rng)
    D = {l: wigner.wigner_d(l, R)[0] for l in range(4)}
    xl = [0, 1, 2]
    ol = [p.l3 for p in lay.paths]
    Yr = sh.real_sh(vec @ R.T, 3)
    xr = _rotate_blocks(x, xl, D)
    out = conv.fwd(lay, off, src, x, Y, w)
    outr = conv.fwd(lay, off, src, xr, Yr, w)
    np.testing.assert_allclose(outr, _rotate_blocks(out, ol, D), atol=1e-11)
    gr = _rotate_blocks(g, ol, D)
    dx, dY, dw = _all_grads(lay, off, src, Y, x, w, g, N)
    dxr, dYr, dwr = _all_grads(lay, off, src, Yr, xr, w, gr, N)
    np.testing.assert_allclose(dxr, _rotate_blocks(dx, xl, D), atol=1e-11)
    np.testing.assert_allclose(dYr, _rotate_blocks(dY, [0, 1, 2, 3], D), atol=1e-11)
    np.testing.assert_allclose(dwr, dw, atol=1e-11)


def test_inversion_parity():
    N = 8
    lay, off, src, vec, Y, x, w, g = small_problem("2x0e+2x1o+2x2e", "1x0e+1x1o+1x2e+1x3o", 3,
                                                   N=N, seed=7)
    px = np.concatenate([[1.0], [-1.0] * 3, [1.0] * 5])
    Yi = sh.real_sh(-vec, 3)
    out = conv.fwd(lay, off, src, x, Y, w)
    outi = conv.fwd(lay, off, src, x * px, Yi, w)
    sign = np.concatenate([[p.parity] * (2 * p.l3 + 1) for p in lay.paths])
    np.testing.assert_allclose(outi, out * sign, atol=1e-12)


def test_sampling_and_threads_and_empty_segments():
    N = 30
    degrees = np.random.default_rng(8).integers(0, 6, size=N)
    degrees[[0, 5, 29]] = 0
    lay, off, src, vec, Y, x, w, g = small_problem("3x0e+3x1o", "1x0e+1x1o+1x2e", 2, N=N,
                                                   degrees=degrees, seed=8)
    full = conv.fwd(lay, off, src, x, Y, w, nthreads=1)
    assert np.array_equal(full, conv.fwd(lay, off, src, x, Y, w, nthreads=3))
    assert np.all(full[[0, 5, 29]] == 0)
    pick = np.array([29, 3, 3, 17])
    assert np.array_equal(conv.fwd(lay, off, src, x, Y, w, receivers=pick), full[pick])
    dY, dw = conv.bwd_edges(lay, off, src, x, Y, w, g, nthreads=1)
    dY3, dw3 = conv.bwd_edges(lay, off, src, x, Y, w, g, nthreads=3)
    assert np.array_equal(dY, dY3) and np.array_equal(dw, dw3)
    ep = np.array([src.size - 1, 0, 4])
    dYs, dws = conv.bwd_edges(lay, off, src, x, Y, w, g, edges=ep)
    assert np.array_equal(dYs, dY[ep]) and np.array_equal(dws, dw[ep])
    dx = conv.bwd_dx(lay, off, src, Y, w, g, N, nthreads=1)
    assert np.array_equal(dx, conv.bwd_dx(lay, off, src, Y, w, g, N, nthreads=3))
    sp_ = np.array([7, 0, 29])
    assert np.array_equal(conv.bwd_dx(lay, off, src, Y, w, g, N, senders=sp_), dx[sp_])
    never_sent = np.setdiff1d(np.arange(N), src)
    assert np.all(dx[never_sent] == 0)


def test_no_edges():
    lay = paths.layout("2x0e+2x1o", "1x0e+1x1o", 1)
    N = 4
    off = np.zeros(N + 1, np.int32)
    src = np.zeros(0, np.int32)
    x = np.ones((N, 2, 4))
    out = conv.fwd(lay, off, src, x, np.zeros((0, 4)), np.zeros((0, len(lay.paths), 2)))
    assert out.shape == (N, 2, lay.dim_out) and np.all(out == 0)
    dx = conv.bwd_dx(lay, off, src, np.zeros((0, 4)), np.zeros((0, len(lay.paths), 2)),
                     np.ones((N, 2, lay.dim_out)), N)
    assert np.all(dx == 0)
