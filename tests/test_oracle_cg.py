"""Pins of the oracle's Clebsch-Gordan construction against facts fixed by the mathematics:
textbook complex CG values, closed forms in the real basis for l <= 1, orthogonality,
completeness and intertwining with Wigner-D matrices fitted from the spherical harmonics."""
import itertools

import numpy as np
import pytest

from conftest import golden_rows, signed_sqrt
from oracle import cg, wigner

LMAX = 4


def test_complex_cg_textbook_table():
    for j1, m1, j2, m2, J, M, s, n, d in golden_rows("complex_cg_table.txt"):
        got = cg.complex_cg(int(j1), int(m1), int(j2), int(m2), int(J), int(M))
        assert got == pytest.approx(signed_sqrt(s, n, d), abs=1e-15)


@pytest.mark.parametrize("l", range(0, 6))
def test_complex_cg_singlet_closed_form(l):
    # <l m l -m | 0 0> = (-1)^(l-m) / sqrt(2l+1)
    for m in range(-l, l + 1):
        want = (-1) ** (l - m) / np.sqrt(2 * l + 1)
        assert cg.complex_cg(l, m, l, -m, 0, 0) == pytest.approx(want, abs=1e-15)


def test_complex_cg_stretched_and_exchange_symmetry():
    for l1, l2 in itertools.product(range(5), repeat=2):
        assert cg.complex_cg(l1, l1, l2, l2, l1 + l2, l1 + l2) == pytest.approx(1.0, abs=1e-15)
        for l3 in range(abs(l1 - l2), l1 + l2 + 1):
            for m1 in range(-l1, l1 + 1):
                for m2 in range(-l2, l2 + 1):
                    a = cg.complex_cg(l1, m1, l2, m2, l3, m1 + m2)
                    b = cg.complex_cg(l2, m2, l1, m1, l3, m1 + m2)
                    assert a == pytest.approx((-1) ** (l1 + l2 - l3) * b, abs=1e-14)


def test_real_basis_unitary():
    for l in range(6):
        q = cg.real_basis(l)
        assert np.allclose(q @ q.conj().T, np.eye(2 * l + 1), atol=1e-15)


def test_real_cg_closed_forms_l_le_1():
    want = {}
    for l1, l2, l3, i1, i2, i3, s, n, d in golden_rows("real_cg_l_le_1.txt"):
        key = (int(l1), int(l2), int(l3))
        want.setdefault(key, np.zeros((2 * key[0] + 1, 2 * key[1] + 1, 2 * key[2] + 1)))
        want[key][int(i1), int(i2), int(i3)] = signed_sqrt(s, n, d)
    assert len(want) == 6
    for key, t in want.items():
        np.testing.assert_allclose(cg.real_cg(*key), t, atol=1e-15, rtol=0)


@pytest.mark.parametrize("l", range(LMAX + 1))
def test_real_cg_identity_paths(l):
    eye = np.eye(2 * l + 1)
    np.testing.assert_allclose(cg.real_cg(0, l, l)[0], eye, atol=1e-15)
    np.testing.assert_allclose(cg.real_cg(l, 0, l)[:, 0, :], eye, atol=1e-15)


def _triples(lmax):
    for l1, l2 in itertools.product(range(lmax + 1), repeat=2):
        for l3 in range(abs(l1 - l2), l1 + l2 + 1):
            yield l1, l2, l3


def test_real_cg_orthogonality():
    # sum_{m1,m2} C^{l3}[m1,m2,m3] C^{l3'}[m1,m2,m3'] = delta(l3,l3') delta(m3,m3')
    for l1, l2 in itertools.product(range(LMAX + 1), repeat=2):
        ls = list(range(abs(l1 - l2), l1 + l2 + 1))
        for a in ls:
            for b in ls:
                g = np.einsum("ijk,ijl->kl", cg.real_cg(l1, l2, a), cg.real_cg(l1, l2, b))
                want = np.eye(2 * a + 1) if a == b else np.zeros((2 * a + 1, 2 * b + 1))
                np.testing.assert_allclose(g, want, atol=1e-14)


def test_real_cg_completeness():
    # sum_{l3,m3} C[m1,m2,m3] C[m1',m2',m3] = delta delta
    for l1, l2 in itertools.product(range(LMAX + 1), repeat=2):
        d = (2 * l1 + 1) * (2 * l2 + 1)
        acc = np.zeros((d, d))
        for l3 in range(abs(l1 - l2), l1 + l2 + 1):
            c = cg.real_cg(l1, l2, l3).reshape(d, -1)
            acc += c @ c.T
        np.testing.assert_allclose(acc, np.eye(d), atol=1e-14)


def test_real_cg_canonical_sign():
    for t in _triples(LMAX):
        flat = cg.real_cg(*t).reshape(-1)
        first = flat[np.nonzero(np.abs(flat) > 1e-9)[0][0]]
        assert first > 0


def test_real_cg_intertwines_rotations():
    # C(D1 a, D2 b) = D3 C(a, b) for random rotations, D fitted from the oracle's SH
    rng = np.random.default_rng(11)
    for _ in range(3):
        R = wigner.random_rotation(rng)
        D = {}
        for l in range(2 * LMAX + 1):
            D[l], resid = wigner.wigner_d(l, R, n_samples=400)
            assert resid < 1e-12
            np.testing.assert_allclose(D[l] @ D[l].T, np.eye(2 * l + 1), atol=1e-12)
        for l1, l2, l3 in _triples(LMAX):
            C = cg.real_cg(l1, l2, l3)
            lhs = np.einsum("ijk,ia,jb->abk", C, D[l1], D[l2])
            rhs = np.einsum("kc,abc->abk", D[l3], C)
            np.testing.assert_allclose(lhs, rhs, atol=1e-12)


def test_planted_mistakes_are_caught():
    # a transposed operand or a dropped sign must break the pins above
    C = cg.real_cg(1, 1, 1)
    assert not np.allclose(C, np.transpose(C, (1, 0, 2)))
    C2 = cg.real_cg(1, 2, 2)
    assert not np.allclose(np.einsum("ijk,ijl->kl", C2, -np.abs(C2)), np.eye(5))
