"""Pins of the oracle's receiver CSR and transposed CSR: a hand-worked example and the defining
properties (offsets monotone, offsets[N] == E, every edge exactly once, ascending edge ids
within each sender, receivers consistent)."""
import numpy as np

from conftest import golden_rows
from oracle import graph
from clebsch_gordan_tensor_receiver_gb300 import workloads


def _fixture():
    return {r[0]: np.array([int(v) for v in r[1:]], dtype=np.int32)
            for r in golden_rows("csr_small.txt")}


def test_hand_worked_example():
    f = _fixture()
    off = graph.recv_offsets(f["recv"], 5)
    assert np.array_equal(off, f["recv_offsets"])
    so, se, sr = graph.transpose(off, f["src"], 5)
    assert np.array_equal(so, f["send_offsets"])
    assert np.array_equal(se, f["send_eids"])
    assert np.array_equal(sr, f["send_recv"])


def test_properties_random_graph():
    rng = np.random.default_rng(0)
    N = 200
    deg = rng.integers(0, 9, size=N)
    recv, src = workloads.random_degree_graph(N, deg, rng)
    off = graph.recv_offsets(recv, N)
    assert off[0] == 0 and off[-1] == src.size and np.all(np.diff(off) >= 0)
    assert np.array_equal(graph.recv_of_edges(off), recv)
    so, se, sr = graph.transpose(off, src, N)
    assert so[-1] == src.size and np.all(np.diff(so) >= 0)
    assert np.array_equal(np.sort(se), np.arange(src.size))
    for s in range(N):
        seg = se[so[s]:so[s + 1]]
        assert np.all(src[seg] == s) and np.all(np.diff(seg) > 0)
    assert np.array_equal(sr, recv[se])


def test_empty_graph():
    off = graph.recv_offsets(np.zeros(0, np.int32), 3)
    assert np.array_equal(off, [0, 0, 0, 0])
    so, se, sr = graph.transpose(off, np.zeros(0, np.int32), 3)
    assert np.array_equal(so, [0, 0, 0, 0]) and se.size == 0 and sr.size == 0
