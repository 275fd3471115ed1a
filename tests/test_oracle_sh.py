"""Pins of the oracle's real spherical harmonics: closed forms at the axes, the component
normalisation, exact orthogonality by quadrature, parity, rotation covariance, and agreement
with the input generator's independent Cartesian polynomials."""
import numpy as np
import pytest

from conftest import golden_rows, signed_sqrt
from oracle import sh, wigner
from clebsch_gordan_tensor_receiver_gb300 import workloads


def test_axis_values():
    rows = golden_rows("sh_axis_values.txt")
    vecs = {}
    for vx, vy, vz, idx, s, n, d in rows:
        key = (int(vx), int(vy), int(vz))
        vecs.setdefault(key, np.zeros(16))[int(idx)] = signed_sqrt(s, n, d)
    for key, want in vecs.items():
        got = sh.real_sh(np.array([key], dtype=float), 3)[0]
        np.testing.assert_allclose(got, want, atol=1e-14)


def test_l_le_1_closed_form():
    rng = np.random.default_rng(1)
    v = workloads.unit_vectors(50, rng)
    y = sh.real_sh(v, 1)
    np.testing.assert_allclose(y[:, 0], 1.0, atol=1e-15)
    np.testing.assert_allclose(y[:, 1:4], np.sqrt(3) * v[:, [1, 2, 0]], atol=1e-15)


@pytest.mark.parametrize("lmax", [3, 6])
def test_component_normalisation(lmax):
    v = workloads.unit_vectors(200, np.random.default_rng(2))
    y = sh.real_sh(v, lmax)
    for l in range(lmax + 1):
        np.testing.assert_allclose((y[:, l * l:(l + 1) ** 2] ** 2).sum(1), 2 * l + 1, atol=1e-12)


def test_orthogonality_by_exact_quadrature():
    # Gauss-Legendre in cos(theta) x uniform phi integrates these polynomials exactly
    lmax = 5
    zs, wz = np.polynomial.legendre.leggauss(12)
    phis = np.arange(24) * (2 * np.pi / 24)
    Z, PH = np.meshgrid(zs, phis, indexing="ij")
    W = np.repeat(wz, phis.size) * (2 * np.pi / phis.size)
    s = np.sqrt(1 - Z ** 2)
    v = np.stack([s * np.cos(PH), s * np.sin(PH), Z], -1).reshape(-1, 3)
    y = sh.real_sh(v, lmax)
    gram = (y * W[:, None]).T @ y / (4 * np.pi)
    np.testing.assert_allclose(gram, np.eye((lmax + 1) ** 2), atol=1e-13)


def test_parity():
    v = workloads.unit_vectors(100, np.random.default_rng(3))
    a, b = sh.real_sh(v, 5), sh.real_sh(-v, 5)
    for l in range(6):
        sl = slice(l * l, (l + 1) ** 2)
        np.testing.assert_allclose(b[:, sl], (-1) ** l * a[:, sl], atol=1e-13)


def test_rotation_covariance():
    rng = np.random.default_rng(4)
    R = wigner.random_rotation(rng)
    for l in range(6):
        D, resid = wigner.wigner_d(l, R, n_samples=300)
        assert resid < 1e-12  # Y_l(R r) is exactly linear in Y_l(r)
        np.testing.assert_allclose(D @ D.T, np.eye(2 * l + 1), atol=1e-12)


def test_input_generator_matches_oracle():
    v = workloads.unit_vectors(1000, np.random.default_rng(5))
    np.testing.assert_allclose(workloads.sh_inputs(v, 3), sh.real_sh(v, 3), atol=1e-13)
