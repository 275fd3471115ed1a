"""uvu_csr_transpose_noalloc: the sender-CSR build for callers that cannot allocate device memory
themselves (for instance a plugin whose host runtime owns the whole device memory pool and only
hands it input and output buffers, or a latency-critical path that must not take an allocator
lock or risk an out-of-memory failure mid-run).  Its scratch is a fixed array inside the library.

Checked here through the C ABI: on two calls in a row, with different graphs so that the second
call starts from the scratch the first one left behind, its results equal bit for bit the
oracle's stable counting sort and those of uvu_csr_transpose with a caller-provided workspace; a
graph without edges gives empty sender rows; a graph whose scratch need is exactly the built-in
16 MiB is served, and one needing more is refused before any work is enqueued."""
import ctypes

import numpy as np
import pytest
import torch

from clebsch_gordan_tensor_receiver_gb300 import uvu, workloads
from oracle import graph

pytestmark = pytest.mark.gpu

V = ctypes.c_void_p


def _p(t):
    return V(t.data_ptr())


def _stream():
    return V(torch.cuda.current_stream().cuda_stream)


def _prepared(N, recv, src):
    recv_d = torch.from_numpy(recv).cuda()
    src_d = torch.from_numpy(src).cuda()
    off = torch.empty(N + 1, dtype=torch.int32, device="cuda")
    uvu.uvu_csr_from_sorted_recv(N, src.size, _p(recv_d), _p(off), _stream())
    return off, src_d


def _outputs(N, E):
    return [torch.full((n,), -7, dtype=torch.int32, device="cuda") for n in (N + 1, max(E, 1), max(E, 1))]


def _with_workspace(N, off, src_d):
    E = src_d.numel()
    so, se, sr = _outputs(N, E)
    nb = ctypes.c_size_t()
    uvu.uvu_csr_transpose_workspace(N, E, ctypes.byref(nb))
    ws = torch.empty(nb.value, dtype=torch.uint8, device="cuda")
    uvu.uvu_csr_transpose(N, E, _p(off), _p(src_d), _p(so), _p(se), _p(sr), _p(ws), nb.value, _stream())
    return so, se[:E], sr[:E]


def _without_allocation(N, off, src_d):
    E = src_d.numel()
    so, se, sr = _outputs(N, E)
    uvu.uvu_csr_transpose_noalloc(N, E, _p(off), _p(src_d), _p(so), _p(se), _p(sr), _stream())
    return so, se[:E], sr[:E]


def _check_against_oracle(N, recv, src, got):
    off = graph.recv_offsets(recv, N)
    want = graph.transpose(off, src, N)
    for name, a, b in zip(("send_offsets", "send_eids", "send_recv"), got, want):
        assert np.array_equal(a.cpu().numpy(), b), name


def test_two_calls_in_a_row_match_the_oracle_and_the_workspace_version():
    medium = workloads.make_workload(1)  # 5,000 receivers x 56 senders
    rng = np.random.default_rng(77)
    deg = rng.integers(0, 10, size=700)
    deg[:5] = 0
    recv2, src2 = workloads.random_degree_graph(700, deg, rng)
    for N, recv, src in ((medium.n_nodes, medium.recv, medium.src), (700, recv2, src2)):
        off, src_d = _prepared(N, recv, src)
        want = _with_workspace(N, off, src_d)
        got = _without_allocation(N, off, src_d)
        torch.cuda.synchronize()
        for name, a, b in zip(("send_offsets", "send_eids", "send_recv"), got, want):
            assert torch.equal(a, b), name
        _check_against_oracle(N, recv, src, got)


def test_graph_without_edges():
    N = 9
    recv = np.zeros(0, np.int32)
    src = np.zeros(0, np.int32)
    off, src_d = _prepared(N, recv, src)
    so, se, sr = _without_allocation(N, off, src_d)
    torch.cuda.synchronize()
    assert torch.equal(so.cpu(), torch.zeros(N + 1, dtype=torch.int32))


def test_graph_at_the_scratch_limit():
    # 4(N+1) and 4E rounded up to 256 bytes sum to exactly 16 MiB: the largest graph served
    N, E = 194_303, 4_000_000
    nb = ctypes.c_size_t()
    uvu.uvu_csr_transpose_workspace(N, E, ctypes.byref(nb))
    assert nb.value == 16 << 20
    rng = np.random.default_rng(5)
    recv = np.sort(rng.integers(0, N, size=E)).astype(np.int32)
    src = rng.integers(0, N, size=E).astype(np.int32)
    off, src_d = _prepared(N, recv, src)
    got = _without_allocation(N, off, src_d)
    torch.cuda.synchronize()
    _check_against_oracle(N, recv, src, got)


def test_graph_beyond_the_builtin_scratch_is_refused():
    dummy = V(256)  # never dereferenced: the size check comes first
    for N, E in ((1000, 5_000_000), (194_304, 4_000_000)):  # the second is 256 bytes over
        nb = ctypes.c_size_t()
        uvu.uvu_csr_transpose_workspace(N, E, ctypes.byref(nb))
        assert nb.value > 16 << 20
        st = uvu.lib.uvu_csr_transpose_noalloc(N, E, dummy, dummy, dummy, dummy, dummy, None)
        assert st == 2  # UVU_ERR_UNSUPPORTED
        assert "scratch" in uvu.uvu_last_error_message()
