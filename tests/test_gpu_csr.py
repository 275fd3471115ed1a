"""GPU graph preparation: the receiver CSR and the transposed CSR are bit-exact against the
oracle's counting/stable-sort construction on the workload graphs and on edge cases."""
import numpy as np
import pytest
import torch

from clebsch_gordan_tensor_receiver_gb300 import uvu, workloads
from oracle import graph

pytestmark = pytest.mark.gpu


def _check(N, recv, src):
    G = uvu.Graph(N, torch.from_numpy(recv).cuda(), torch.from_numpy(src).cuda())
    off = graph.recv_offsets(recv, N)
    so, se, sr = graph.transpose(off, src, N)
    E = src.size
    assert np.array_equal(G.recv_offsets.cpu().numpy(), off)
    assert np.array_equal(G.send_offsets.cpu().numpy(), so)
    assert np.array_equal(G.send_eids[:E].cpu().numpy(), se)
    assert np.array_equal(G.send_recv[:E].cpu().numpy(), sr)


@pytest.mark.parametrize("key", [0, 1, 4])
def test_workload_graphs(key):
    wl = workloads.make_workload(key)
    _check(wl.n_nodes, wl.recv, wl.src)


def test_edge_cases():
    rng = np.random.default_rng(3)
    _check(5, np.zeros(0, np.int32), np.zeros(0, np.int32))           # no edges
    _check(1, np.zeros(3, np.int32), np.zeros(3, np.int32))            # one node, self edges
    deg = rng.integers(0, 4, size=300)
    deg[:10] = 0
    deg[-10:] = 0
    recv, src = workloads.random_degree_graph(300, deg, rng)
    _check(300, recv, src)                                             # empty rows at both ends
    N = 4000
    recv = np.repeat(np.arange(N), 3).astype(np.int32)
    src = np.full(recv.size, 17, np.int32)
    src[::7] = 3
    _check(N, recv, src)                                               # two hub senders
