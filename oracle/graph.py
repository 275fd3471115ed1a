"""Receiver CSR and transposed (sender) CSR for the oracle (test infrastructure only).

"Receiver-streaming convolutions for channel-wise UVU tensor products" (opening post, benchmark
paragraph) runs on prepared, receiver-sorted edge lists: edges grouped by their receiver, i.e. a
CSR over receivers.  The transposed CSR groups the same edges by sender; within one sender the
edge ids are kept in ascending order (a stable sort), which makes the index build unique and
therefore checkable bit for bit.
"""

from __future__ import annotations

import numpy as np


def recv_offsets(recv: np.ndarray, n_nodes: int) -> np.ndarray:
    """offsets[r] = number of edges whose receiver is < r (recv must be non-decreasing)."""
    recv = np.asarray(recv, dtype=np.int64)
    if recv.size and np.any(np.diff(recv) < 0):
        raise ValueError("recv must be sorted")
    counts = np.bincount(recv, minlength=n_nodes) if recv.size else np.zeros(n_nodes, np.int64)
    off = np.zeros(n_nodes + 1, dtype=np.int64)
    np.cumsum(counts, out=off[1:])
    return off.astype(np.int32)


def recv_of_edges(offsets: np.ndarray) -> np.ndarray:
    """Expand a receiver CSR back to one receiver id per edge."""
    offsets = np.asarray(offsets, dtype=np.int64)
    return np.repeat(np.arange(offsets.size - 1), np.diff(offsets)).astype(np.int32)


def transpose(offsets: np.ndarray, src: np.ndarray, n_nodes: int):
    """(send_offsets[N+1], send_eids[E], send_recv[E]); edge ids ascending within each sender."""
    src = np.asarray(src, dtype=np.int64)
    recv = recv_of_edges(offsets)
    eids = np.argsort(src, kind="stable")
    counts = np.bincount(src, minlength=n_nodes) if src.size else np.zeros(n_nodes, np.int64)
    soff = np.zeros(n_nodes + 1, dtype=np.int64)
    np.cumsum(counts, out=soff[1:])
    return soff.astype(np.int32), eids.astype(np.int32), recv[eids].astype(np.int32)
