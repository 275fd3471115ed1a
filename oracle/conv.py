"""Python side of the fp64 oracle convolution (test infrastructure only).

Builds ``conv.c`` with gcc (OpenMP, no fast-math, no machine-specific flags) into
``oracle/_build/`` and calls it through ctypes.  Inputs of any float dtype are upcast exactly to
fp64 before the call.  Every entry point can restrict the work to a list of owners (receivers,
edges or senders), which is how full-size workloads are checked on sampled outputs: each sampled
output element is still computed from its complete definition.
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

from . import cg as _cg
from . import graph as _graph
from .paths import Layout

_HERE = os.path.dirname(os.path.abspath(__file__))
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle_conv.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile conv.c -> _build/liboracle_conv.so (skipped when up to date)."""
    srcp = os.path.join(_HERE, "conv.c")
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(srcp)):
        return _LIB_PATH
    os.makedirs(_BUILD, exist_ok=True)
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared", srcp, "-o", tmp]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P = ctypes.c_void_p
            i64, i32 = ctypes.c_int64, ctypes.c_int
            lib.oracle_fwd.argtypes = [i64, P, P, i32, i32, P, P, i32, i32, i32, P, P, P, P, i32]
            lib.oracle_bwd_edges.argtypes = [i64, P, P, i32, i32, P, P, i32, i32, i32,
                                             P, P, P, P, P, P, i32]
            lib.oracle_bwd_dx.argtypes = [i64, P, P, P, i32, i32, P, P, i32, i32, i32,
                                          P, P, P, P, i32]
            lib.oracle_max_threads.restype = ctypes.c_int
            _lib = lib
    return _lib


def default_threads() -> int:
    return len(os.sched_getaffinity(0))


def pack_paths(lay: Layout):
    """(paths int32[P*7], dense CG blocks fp64) in path order."""
    rows, blocks, off = [], [], 0
    for p in lay.paths:
        c = _cg.real_cg(p.l1, p.l2, p.l3)
        rows.append([p.l1, p.l2, p.l3, p.xoff, p.yoff, p.ooff, off])
        blocks.append(c.reshape(-1))
        off += c.size
    tab = np.ascontiguousarray(np.array(rows, dtype=np.int32).reshape(-1))
    cgv = np.ascontiguousarray(np.concatenate(blocks) if blocks else np.zeros(0))
    return tab, cgv


def _f64(a):
    return np.ascontiguousarray(a, dtype=np.float64)


def _ptr(a):
    return a.ctypes.data_as(ctypes.c_void_p)


def fwd(lay: Layout, recv_offsets, src, x, Y, w, receivers=None, nthreads=None):
    """out[len(receivers)][U][D_out] (all receivers when ``receivers`` is None)."""
    lib = _load()
    off = np.asarray(recv_offsets, dtype=np.int64)
    src = np.asarray(src, dtype=np.int32)
    if receivers is None:
        receivers = np.arange(off.size - 1)
    receivers = np.asarray(receivers, dtype=np.int64)
    # gather the sampled receivers' segments into one compact edge list
    segs = [np.arange(off[r], off[r + 1]) for r in receivers]
    eidx = np.concatenate(segs) if segs else np.zeros(0, np.int64)
    loff = np.zeros(receivers.size + 1, dtype=np.int64)
    np.cumsum([s.size for s in segs], out=loff[1:])
    tab, cgv = pack_paths(lay)
    P, U = len(lay.paths), lay.mul
    xs = _f64(x)
    Ys = _f64(np.asarray(Y)[eidx])
    ws = _f64(np.asarray(w)[eidx])
    ss = np.ascontiguousarray(src[eidx])
    out = np.zeros((receivers.size, U, lay.dim_out))
    lib.oracle_fwd(receivers.size, _ptr(loff), _ptr(ss), U, P, _ptr(tab), _ptr(cgv),
                   lay.dim_x, lay.dim_y, lay.dim_out, _ptr(xs), _ptr(Ys), _ptr(ws), _ptr(out),
                   nthreads or default_threads())
    return out


def bwd_edges(lay: Layout, recv_offsets, src, x, Y, w, d_out, edges=None, nthreads=None):
    """(dY[len(edges)][D_Y], dw[len(edges)][P][U]) for the listed edges (all when None)."""
    lib = _load()
    recv = _graph.recv_of_edges(recv_offsets)
    src = np.asarray(src, dtype=np.int32)
    if edges is None:
        edges = np.arange(src.size)
    edges = np.asarray(edges, dtype=np.int64)
    tab, cgv = pack_paths(lay)
    P, U = len(lay.paths), lay.mul
    rr = np.ascontiguousarray(recv[edges])
    ss = np.ascontiguousarray(src[edges])
    xs, gs = _f64(x), _f64(d_out)
    Ys = _f64(np.asarray(Y)[edges])
    ws = _f64(np.asarray(w)[edges])
    dY = np.zeros((edges.size, lay.dim_y))
    dw = np.zeros((edges.size, P, U))
    lib.oracle_bwd_edges(edges.size, _ptr(rr), _ptr(ss), U, P, _ptr(tab), _ptr(cgv),
                         lay.dim_x, lay.dim_y, lay.dim_out, _ptr(xs), _ptr(Ys), _ptr(ws),
                         _ptr(gs), _ptr(dY), _ptr(dw), nthreads or default_threads())
    return dY, dw


def bwd_dx(lay: Layout, recv_offsets, src, Y, w, d_out, n_nodes, senders=None, nthreads=None):
    """dx[len(senders)][U][D_x] (all nodes when None), through the oracle's own transposed CSR."""
    lib = _load()
    soff, eids, srecv = _graph.transpose(recv_offsets, src, n_nodes)
    soff = soff.astype(np.int64)
    if senders is None:
        senders = np.arange(n_nodes)
    senders = np.asarray(senders, dtype=np.int64)
    segs = [np.arange(soff[s], soff[s + 1]) for s in senders]
    kidx = np.concatenate(segs) if segs else np.zeros(0, np.int64)
    loff = np.zeros(senders.size + 1, dtype=np.int64)
    np.cumsum([s.size for s in segs], out=loff[1:])
    le = eids[kidx].astype(np.int64)
    tab, cgv = pack_paths(lay)
    P, U = len(lay.paths), lay.mul
    Ys = _f64(np.asarray(Y)[le])
    ws = _f64(np.asarray(w)[le])
    gs = _f64(d_out)
    keids = np.arange(le.size, dtype=np.int32)  # compact edge ids
    krecv = np.ascontiguousarray(srecv[kidx].astype(np.int32))
    dx = np.zeros((senders.size, U, lay.dim_x))
    lib.oracle_bwd_dx(senders.size, _ptr(loff), _ptr(keids), _ptr(krecv), U, P, _ptr(tab),
                      _ptr(cgv), lay.dim_x, lay.dim_y, lay.dim_out, _ptr(Ys), _ptr(ws), _ptr(gs),
                      _ptr(dx), nthreads or default_threads())
    return dx
