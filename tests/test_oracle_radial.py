"""Pins of the radial-weight oracle (oracle.radial).

- the Bessel basis is orthonormal on [0, r_cut] with weight r^2 (numerical quadrature), matches
  hand-derived values at r = r_cut / 2 and its limit at r -> 0 (tests/golden);
- the envelope is the unique degree-(p+2) polynomial with f(0) = 1 and f, f', f'' = 0 at the
  cutoff (checked on a fitted polynomial), is monotone, vanishes beyond the cutoff and matches
  exact rationals;
- SiLU matches scipy's logistic function times its argument;
- the network matches torch.nn layers (Linear without bias, SiLU) in float64;
- the per-edge weights match a brute-force triple loop;
- the convolution with radial weights equals the convolution with the weights materialised, is
  unchanged by extra edges at or beyond the cutoff, and is linear in the last layer.
"""
import numpy as np
import pytest
import scipy.integrate
import scipy.special

from conftest import golden_rows
from clebsch_gordan_tensor_receiver_gb300 import workloads
from oracle import conv, graph, paths, radial, sh


def test_golden_closed_forms():
    for row in golden_rows("radial_closed_forms.txt"):
        kind, vals = row[0], [float(v) for v in row[1:]]
        if kind == "bessel":
            rc, r, n, want = vals
            got = radial.bessel_basis([r], rc, int(n))[0, int(n) - 1]
        elif kind == "bessel_limit":
            rc, r, n, want = vals
            got = radial.bessel_basis([r], rc, int(n))[0, int(n) - 1]
        elif kind == "envelope":
            p, s, want = vals
            got = float(radial.envelope(s, int(p)))
        else:
            v, want = vals
            got = float(radial.silu(v))
        assert got == pytest.approx(want, rel=1e-12, abs=1e-15), row


@pytest.mark.parametrize("rc", [1.0, 5.0])
def test_bessel_orthonormal_with_r2_weight(rc):
    nb = 6
    G = np.zeros((nb, nb))
    for a in range(nb):
        for b in range(nb):
            f = lambda r: radial.bessel_basis([r], rc, nb)[0, a] * radial.bessel_basis([r], rc, nb)[0, b] * r * r
            G[a, b] = scipy.integrate.quad(f, 1e-12, rc, limit=200, epsabs=1e-13)[0]
    np.testing.assert_allclose(G, np.eye(nb), atol=1e-9)


@pytest.mark.parametrize("p", [3, 5, 6])
def test_envelope_is_the_smooth_cutoff_polynomial(p):
    s = np.linspace(0.0, 0.999, 400)
    f = radial.envelope(s, p)
    c = np.polynomial.polynomial.Polynomial.fit(s, f, p + 2).convert()
    np.testing.assert_allclose(c(s), f, atol=1e-11)           # a polynomial of degree p + 2
    assert c(0.0) == pytest.approx(1.0, abs=1e-10)
    for k in range(3):                                          # value, slope and curvature vanish at 1
        assert c.deriv(k)(1.0) == pytest.approx(0.0, abs=1e-7), k
    assert np.all(np.diff(f) <= 1e-15) and np.all(f >= -1e-15) and np.all(f <= 1.0)
    np.testing.assert_array_equal(radial.envelope(np.array([1.0, 1.2, 3.0]), p), 0.0)


def test_silu_is_logistic_times_argument():
    v = np.linspace(-40, 40, 801)
    np.testing.assert_allclose(radial.silu(v), v * scipy.special.expit(v), rtol=1e-14, atol=1e-300)


def test_network_matches_torch_layers():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(0)
    widths = [8, 16, 12, 20]
    Ws = [rng.standard_normal((widths[i], widths[i + 1])) / np.sqrt(widths[i]) for i in range(3)]
    r = rng.uniform(0.3, 6.0, size=50)  # some beyond the 5.0 cutoff
    h = radial.hidden(r, 5.0, 5, Ws)
    layers = []
    for W in Ws:
        lin = torch.nn.Linear(W.shape[0], W.shape[1], bias=False).double()
        with torch.no_grad():
            lin.weight.copy_(torch.from_numpy(W.T))
        layers += [lin, torch.nn.SiLU()]
    net = torch.nn.Sequential(*layers)
    b = radial.bessel_basis(r, 5.0, 8) * radial.envelope(r / 5.0, 5)[:, None]
    with torch.no_grad():
        want = net(torch.from_numpy(b)).numpy()
    np.testing.assert_allclose(h, want, rtol=1e-13, atol=1e-15)
    assert np.all(h[r >= 5.0] == 0.0)


def test_weights_brute_force():
    rng = np.random.default_rng(1)
    h, Wl = rng.standard_normal((4, 5)), rng.standard_normal((5, 3, 2))
    w = radial.weights(h, Wl)
    for e in range(4):
        for p in range(3):
            for u in range(2):
                assert w[e, p, u] == pytest.approx(sum(h[e, k] * Wl[k, p, u] for k in range(5)), rel=1e-14)


def _problem(seed, N=9, dmax=5, U=3, H=8):
    rng = np.random.default_rng(seed)
    lay = paths.layout(f"{U}x0e+{U}x1o+{U}x2e", "1x0e+1x1o+1x2e", 2)
    recv, src = workloads.random_degree_graph(N, rng.integers(0, dmax + 1, size=N), rng)
    Y = sh.real_sh(rng.standard_normal((src.size, 3)), 2)
    x = rng.standard_normal((N, U, lay.dim_x))
    r = rng.uniform(0.5, 4.9, size=src.size)
    Ws = [rng.standard_normal((6, H)) / np.sqrt(6), rng.standard_normal((H, H)) / np.sqrt(H)]
    Wl = rng.standard_normal((H, len(lay.paths), U)) / np.sqrt(H)
    return lay, recv, src, x, Y, r, Ws, Wl, N


def test_conv_with_radial_weights_equals_materialised_weights():
    lay, recv, src, x, Y, r, Ws, Wl, N = _problem(2)
    off = graph.recv_offsets(recv, N)
    h = radial.hidden(r, 5.0, 5, Ws)
    want = conv.fwd(lay, off, src, x, Y, radial.weights(h, Wl))
    np.testing.assert_allclose(radial.conv_fwd(lay, off, src, x, Y, h, Wl), want, atol=1e-13)
    rs = np.array([0, 3, N - 1])
    np.testing.assert_allclose(radial.conv_fwd(lay, off, src, x, Y, h, Wl, receivers=rs), want[rs], atol=1e-13)


def test_edges_at_or_beyond_the_cutoff_contribute_nothing():
    lay, recv, src, x, Y, r, Ws, Wl, N = _problem(3)
    rng = np.random.default_rng(30)
    k = 7
    recv2 = np.concatenate([recv, rng.integers(0, N, size=k)]).astype(np.int32)
    src2 = np.concatenate([src, rng.integers(0, N, size=k)]).astype(np.int32)
    r2 = np.concatenate([r, [5.0] + list(rng.uniform(5.0, 9.0, size=k - 1))])
    Y2 = np.concatenate([Y, sh.real_sh(rng.standard_normal((k, 3)), 2)])
    order = np.argsort(recv2, kind="stable")
    off = graph.recv_offsets(recv, N)
    off2 = graph.recv_offsets(recv2[order], N)
    a = radial.conv_fwd(lay, off, src, x, Y, radial.hidden(r, 5.0, 5, Ws), Wl)
    b = radial.conv_fwd(lay, off2, src2[order], x, Y2[order], radial.hidden(r2[order], 5.0, 5, Ws), Wl)
    np.testing.assert_allclose(b, a, atol=1e-13)


def test_linear_in_the_last_layer():
    lay, recv, src, x, Y, r, Ws, Wl, N = _problem(4)
    off = graph.recv_offsets(recv, N)
    h = radial.hidden(r, 5.0, 5, Ws)
    W2 = np.random.default_rng(40).standard_normal(Wl.shape)
    lhs = radial.conv_fwd(lay, off, src, x, Y, h, Wl + 2.0 * W2)
    rhs = radial.conv_fwd(lay, off, src, x, Y, h, Wl) + 2.0 * radial.conv_fwd(lay, off, src, x, Y, h, W2)
    np.testing.assert_allclose(lhs, rhs, atol=1e-12)


# --------------------------------------------------------------------------- gradient pins
# The reverse pass (radial.hidden_vjp, radial.weights_vjp) is pinned by central finite
# differences of the forward definition (independent of the chain rule written out in the
# oracle), by closed-form derivative values, and by the adjoint identity of a bilinear map.

def _net(seed, widths=(8, 16, 12, 8)):
    rng = np.random.default_rng(seed)
    layers = [rng.standard_normal((widths[i], widths[i + 1])) / np.sqrt(widths[i]) for i in range(len(widths) - 1)]
    return rng, layers


def _fd(f, x, eps):
    g = np.zeros_like(x)
    it = np.nditer(x, flags=["multi_index"])
    for _ in it:
        i = it.multi_index
        xp, xm = x.copy(), x.copy()
        xp[i] += eps
        xm[i] -= eps
        g[i] = (f(xp) - f(xm)) / (2 * eps)
    return g


def test_envelope_and_basis_derivatives():
    s = np.linspace(0.05, 0.95, 19)
    for p in (3, 5, 6):
        fd = (radial.envelope(s + 1e-7, p) - radial.envelope(s - 1e-7, p)) / 2e-7
        np.testing.assert_allclose(radial.envelope_deriv(s, p), fd, atol=1e-7)
        # value and slope vanish at the cutoff, the slope at 0 too (p > 1); zero beyond
        assert abs(radial.envelope_deriv(np.array([1.0 - 1e-12]), p)[0]) < 1e-8
        assert radial.envelope_deriv(np.array([0.0]), p)[0] == 0.0
        assert radial.envelope_deriv(np.array([1.3]), p)[0] == 0.0
    r = np.linspace(0.3, 4.9, 23)
    fd = (radial.bessel_basis(r + 1e-7, 5.0, 8) - radial.bessel_basis(r - 1e-7, 5.0, 8)) / 2e-7
    np.testing.assert_allclose(radial.bessel_basis_deriv(r, 5.0, 8), fd, atol=1e-6)
    v = np.linspace(-6, 6, 25)
    np.testing.assert_allclose(radial.silu_deriv(v), (radial.silu(v + 1e-7) - radial.silu(v - 1e-7)) / 2e-7, atol=1e-7)
    # closed forms: silu'(0) = 1/2, d/dr b_n at r -> 0 tends to 0 (b_n is even in r about 0)
    assert radial.silu_deriv(np.array([0.0]))[0] == 0.5
    assert abs(radial.bessel_basis_deriv(np.array([1e-4]), 5.0, 3)).max() < 1e-3


def test_hidden_vjp_matches_finite_differences():
    rng, layers = _net(1)
    E = 6
    r = np.concatenate([rng.uniform(0.8, 4.9, size=E - 2), [4.999, 6.0]])  # one just inside, one beyond
    dh = rng.standard_normal((E, 8))
    dr, dWs = radial.hidden_vjp(r, 5.0, 5, layers, dh)

    def L(rr, ls):
        return float((dh * radial.hidden(rr, 5.0, 5, ls)).sum())

    np.testing.assert_allclose(dr, _fd(lambda rr: L(rr, layers), r, 1e-6), atol=1e-8)
    assert dr[-1] == 0.0  # beyond the cutoff: h = 0 around it
    for i in range(len(layers)):
        def Li(Wi, i=i):
            ls = list(layers)
            ls[i] = Wi
            return L(r, ls)
        np.testing.assert_allclose(dWs[i], _fd(Li, layers[i].copy(), 1e-6), atol=1e-8)


def test_weights_vjp_adjoint_and_finite_differences():
    rng = np.random.default_rng(9)
    E, H, P, U = 7, 5, 3, 4
    h = rng.standard_normal((E, H))
    Wl = rng.standard_normal((H, P, U))
    dw = rng.standard_normal((E, P, U))
    dh, dWl = radial.weights_vjp(h, Wl, dw)
    # w is bilinear in (h, W_last): <dw, w> = <dh, h> = <dW_last, W_last>
    s = float((dw * radial.weights(h, Wl)).sum())
    assert abs(float((dh * h).sum()) - s) < 1e-12 * max(1.0, abs(s))
    assert abs(float((dWl * Wl).sum()) - s) < 1e-12 * max(1.0, abs(s))
    np.testing.assert_allclose(dh, _fd(lambda hh: float((dw * radial.weights(hh, Wl)).sum()), h.copy(), 1e-6), atol=1e-8)
    np.testing.assert_allclose(dWl, _fd(lambda ww: float((dw * radial.weights(h, ww)).sum()), Wl.copy(), 1e-6), atol=1e-8)
    # brute force of one entry of each
    assert abs(dh[2, 3] - sum(dw[2, p, u] * Wl[3, p, u] for p in range(P) for u in range(U))) < 1e-12
    assert abs(dWl[1, 2, 0] - sum(h[e, 1] * dw[e, 2, 0] for e in range(E))) < 1e-12
