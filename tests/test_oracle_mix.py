"""Pins of the channel-mixing oracle (oracle.mix) and of the UVW-to-UVU reduction it serves:
the UVU convolution followed by the mixing equals the UVW convolution with the factorised
weights summed edge by edge; an identity mixing returns its input; the VJP matches central
finite differences (exact for a bilinear map); the mixing commutes with rotations."""
import numpy as np
import pytest

from clebsch_gordan_tensor_receiver_gb300 import workloads
from oracle import conv, graph, mix, paths, sh, wigner


def _conv_problem(seed, U=3, W=4):
    rng = np.random.default_rng(seed)
    lay = paths.layout(f"{U}x0e+{U}x1o+{U}x2e", "1x0e+1x1o+1x2e", 2)
    N = 6
    recv, src = workloads.random_degree_graph(N, rng.integers(0, 4, size=N), rng)
    Y = sh.real_sh(rng.standard_normal((src.size, 3)), 2)
    x = rng.standard_normal((N, U, lay.dim_x))
    w = rng.standard_normal((src.size, len(lay.paths), U))
    M = rng.standard_normal((len(lay.paths), U, W))
    return lay, recv, src, x, Y, w, M, N


def test_uvu_then_mixing_equals_the_factorised_uvw_convolution():
    lay, recv, src, x, Y, w, M, N = _conv_problem(0)
    off = graph.recv_offsets(recv, N)
    uvu = conv.fwd(lay, off, src, x, Y, w)
    np.testing.assert_allclose(mix.fwd(lay, uvu, M), mix.uvw_conv_brute(lay, recv, src, x, Y, w, M, N), atol=1e-12)


def test_identity_mixing():
    rng = np.random.default_rng(1)
    lay = paths.layout("5x0e+5x1o", "1x0e+1x1o", 1)
    inp = rng.standard_normal((7, 5, lay.dim_out))
    M = np.broadcast_to(np.eye(5), (len(lay.paths), 5, 5))
    np.testing.assert_array_equal(mix.fwd(lay, inp, M), inp)


def test_vjp_matches_central_differences():
    rng = np.random.default_rng(2)
    lay = paths.layout("2x0e+2x1o", "1x0e+1x1o", 1)
    P = len(lay.paths)
    inp, M = rng.standard_normal((3, 2, lay.dim_out)), rng.standard_normal((P, 2, 3))
    g = rng.standard_normal((3, 3, lay.dim_out))
    d_inp, dM = mix.vjp(lay, inp, M, g)
    h = 0.5
    for name, arr, grad in (("inp", inp, d_inp), ("M", M, dM)):
        fd = np.zeros_like(arr)
        for i in np.ndindex(arr.shape):
            a, b = arr.copy(), arr.copy()
            a[i] += h
            b[i] -= h
            fa = mix.fwd(lay, a, M) if name == "inp" else mix.fwd(lay, inp, a)
            fb = mix.fwd(lay, b, M) if name == "inp" else mix.fwd(lay, inp, b)
            fd[i] = ((fa - fb) * g).sum() / (2 * h)
        np.testing.assert_allclose(grad, fd, atol=1e-11, err_msg=name)


def test_mixing_commutes_with_rotations():
    rng = np.random.default_rng(3)
    lay = paths.layout("3x0e+3x1o+3x2e", "1x0e+1x1o+1x2e", 2)
    R = wigner.random_rotation(rng)
    inp, M = rng.standard_normal((4, 3, lay.dim_out)), rng.standard_normal((len(lay.paths), 3, 2))
    rot = inp.copy()
    for p in lay.paths:
        so = slice(p.ooff, p.ooff + 2 * p.l3 + 1)
        rot[:, :, so] = inp[:, :, so] @ wigner.wigner_d(p.l3, R)[0].T
    a, b = mix.fwd(lay, rot, M), mix.fwd(lay, inp, M)
    for p in lay.paths:
        so = slice(p.ooff, p.ooff + 2 * p.l3 + 1)
        np.testing.assert_allclose(a[:, :, so], b[:, :, so] @ wigner.wigner_d(p.l3, R)[0].T, atol=1e-10)
