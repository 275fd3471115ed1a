"""GPU graph preparation: the receiver CSR and the transposed CSR are bit-exact against the
oracle's counting/stable-sort construction on the workload graphs and on edge cases."""
import ctypes

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


def test_hub_senders_and_the_sort_threshold():
    # sender segments of 64 edges (rank counting), 65 (the in-place sort), a non-power-of-two hub
    # of 100,003 edges and a power-of-two one of 4,096: every order ascending by edge id
    rng = np.random.default_rng(11)
    N = 2000
    counts = {5: 64, 6: 65, 7: 100_003, 8: 4_096, 9: 1}
    src = np.concatenate([np.full(c, s, np.int32) for s, c in counts.items()] +
                         [rng.integers(10, N, size=30_000).astype(np.int32)])
    rng.shuffle(src)
    recv = np.sort(rng.integers(0, N, size=src.size)).astype(np.int32)
    _check(N, recv, src)


def test_broken_recv_is_reported_not_written_outside():
    # a receiver id past the last node: the offsets stay inside recv_offsets and the CSR fails
    # validation (offsets[N] != E)
    N = 5
    recv = torch.tensor([0, 0, 7], dtype=torch.int32, device="cuda")
    guard = torch.full((N + 1 + 64,), -3, dtype=torch.int32, device="cuda")
    off = guard[:N + 1]
    st = torch.cuda.current_stream()
    uvu.uvu_csr_from_sorted_recv(N, 3, ctypes.c_void_p(recv.data_ptr()), ctypes.c_void_p(off.data_ptr()),
                                 ctypes.c_void_p(st.cuda_stream))
    torch.cuda.synchronize()
    assert torch.equal(guard[N + 1:].cpu(), torch.full((64,), -3, dtype=torch.int32))
    src = torch.zeros(3, dtype=torch.int32, device="cuda")
    ws = torch.zeros(2, dtype=torch.int64, device="cuda")
    bad = ctypes.c_int64()
    uvu.uvu_graph_validate(N, 3, ctypes.c_void_p(off.data_ptr()), ctypes.c_void_p(src.data_ptr()),
                           ctypes.c_void_p(ws.data_ptr()), ctypes.byref(bad), ctypes.c_void_p(st.cuda_stream))
    assert bad.value > 0
