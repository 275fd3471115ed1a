"""The seeded input generators: determinism, shapes and the workload recipes (degree, graph
structure, value scales)."""
import numpy as np
import pytest

from clebsch_gordan_tensor_receiver_gb300 import workloads


def test_tiny_recipe_and_determinism():
    a = workloads.make_workload(0)
    b = workloads.make_workload(0)
    assert np.array_equal(a.src, b.src) and np.array_equal(a.x, b.x) and np.array_equal(a.Y, b.Y)
    assert a.n_edges == 800 and a.x.shape == (100, 16, 4) and a.Y.shape == (800, 9)
    assert a.x.dtype == np.float32 and a.Y.dtype == np.float32
    assert np.all(np.diff(a.recv) >= 0)
    for r in range(100):
        s = a.src[a.recv == r]
        assert s.size == 8 and np.all(np.diff(s) > 0) and not np.any(s == r)
    w = workloads.make_weights(a.spec, a.n_edges, 9)
    assert w.shape == (800, 9, 16)
    assert np.std(w) == pytest.approx(1 / np.sqrt(8), rel=0.05)
    g = workloads.make_cotangent(a.spec, 100, 29)
    assert g.shape == (100, 16, 29)


def test_periodic_graph_small():
    rng = np.random.default_rng(1)
    recv, src, vec, box = workloads.periodic_graph(3000, 0.056, 5.0, rng)
    assert np.all(np.diff(recv) >= 0)
    deg = np.bincount(recv, minlength=3000)
    assert deg.mean() == pytest.approx(0.056 * 4 / 3 * np.pi * 125, rel=0.05)
    pairs = set(zip(recv.tolist(), src.tolist()))
    assert all((s, r) in pairs for r, s in list(pairs)[:500])  # symmetric neighbour list
    assert not np.any(recv == src)
    np.testing.assert_allclose(np.linalg.norm(vec, axis=1), 1.0, atol=1e-12)


def test_unit_vector_sh_normalisation():
    v = workloads.unit_vectors(100, np.random.default_rng(2))
    Y = workloads.sh_inputs(v, 3)
    for l in range(4):
        np.testing.assert_allclose((Y[:, l * l:(l + 1) ** 2] ** 2).sum(1), 2 * l + 1, atol=1e-12)


def test_radial_inputs_recipe():
    """Edge lengths of the fused-radial-weight inputs: density proportional to r^2 on
    [0.75, 5) (a Kolmogorov-Smirnov test against that law's CDF), seeded and reproducible;
    layer shapes [H_(i-1)][H_i] with variance 1/H_(i-1); the last layer [H][P][U]."""
    import scipy.stats
    from clebsch_gordan_tensor_receiver_gb300 import workloads
    spec = workloads.SPECS[1]
    r, layers, wl = workloads.radial_inputs(spec, 20000, 13)
    r2, layers2, wl2 = workloads.radial_inputs(spec, 20000, 13)
    assert np.array_equal(r, r2) and np.array_equal(wl, wl2) and all(np.array_equal(a, b) for a, b in zip(layers, layers2))
    assert r.dtype == np.float32 and r.min() >= 0.75 and r.max() < 5.0
    a3, c3 = 0.75 ** 3, 5.0 ** 3
    cdf = lambda t: np.clip((np.asarray(t, dtype=np.float64) ** 3 - a3) / (c3 - a3), 0.0, 1.0)
    assert scipy.stats.kstest(r.astype(np.float64), cdf).pvalue > 1e-3
    assert [W.shape for W in layers] == [(8, 64), (64, 64), (64, 64)] and wl.shape == (64, 13, 128)
    assert abs(layers[1].astype(np.float64).var() * 64 - 1.0) < 0.1
    assert abs(wl.astype(np.float64).var() * 64 * 56 - 1.0) < 0.05


def test_reduced_node_count():
    """A workload generated at fewer nodes than its recipe's default reports that count, and its
    graph and inputs stay inside it (the reduced sizes used for small profiling runs)."""
    from clebsch_gordan_tensor_receiver_gb300 import workloads
    wl = workloads.make_workload(1, 300)
    assert wl.n_nodes == 300 and wl.x.shape[0] == 300
    assert wl.recv.max() < 300 and wl.src.max() < 300 and wl.n_edges == 300 * 56
