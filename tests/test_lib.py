"""The C-ABI library: it loads without a GPU, exports every symbol that include/uvu.h declares,
and rejects bad arguments on the host with clear statuses (no compute call is made here)."""
import ctypes
import os
import re
import shutil
import subprocess
import sys

import pytest

from conftest import ROOT
from clebsch_gordan_tensor_receiver_gb300 import uvu


def header_symbols():
    txt = open(os.path.join(ROOT, "include", "uvu.h")).read()
    txt = re.sub(r"/\*.*?\*/", "", txt, flags=re.S)
    return sorted(set(re.findall(r"\b(uvu_[a-z_0-9]+)\s*\(", txt)))


def test_exports_every_declared_symbol():
    syms = header_symbols()
    assert len(syms) >= 15
    assert sorted(uvu.EXPORTS) == syms
    for s in syms:
        assert hasattr(uvu.lib, s), s


def test_links_no_driver_library():
    # The library must load on a host without a GPU driver: it links the CUDA runtime statically
    # and names no driver library among its dynamic dependencies.
    maps = open("/proc/self/maps").read()
    assert uvu.LIB_PATH in maps
    readelf = shutil.which("readelf")
    if readelf:
        dyn = subprocess.run([readelf, "-d", uvu.LIB_PATH], capture_output=True, text=True, check=True).stdout
        needed = re.findall(r"\(NEEDED\)\s+Shared library: \[([^\]]+)\]", dyn)
        assert needed, dyn
        assert not [n for n in needed if n.startswith("libcuda.") or n.startswith("libcudart.")], needed
    # and loading it in a fresh process (without torch, which maps the driver on GPU hosts) maps
    # no driver library
    code = ("import ctypes, sys; ctypes.CDLL(sys.argv[1]); "
            "print(any('libcuda.so' in l for l in open('/proc/self/maps')))")
    r = subprocess.run([sys.executable, "-c", code, uvu.LIB_PATH], capture_output=True, text=True, check=True)
    assert r.stdout.strip() == "False", r.stdout


def test_status_strings():
    assert uvu.uvu_status_string(0) == "UVU_OK"
    assert uvu.uvu_status_string(1) == "UVU_ERR_INVALID_ARGUMENT"
    assert uvu.uvu_status_string(99) == "UVU_ERR_UNKNOWN"


@pytest.mark.parametrize("ix,isx,lo,status", [
    ("128x0e+128x1o", "1x0e+1x1o", 1, 0),
    ("128x0e+64x1o", "1x0e+1x1o", 1, 1),     # not channel-wise
    ("128x0e+128x1q", "1x0e", 1, 1),         # bad parity letter
    ("128x0e+", "1x0e", 1, 1),               # dangling '+'
    ("", "1x0e", 1, 1),                      # empty
    ("8x0e", "2x1o", 1, 1),                  # SH multiplicity != 1
    ("8x5e", "1x0e", 5, 2),                  # l > 4
    ("8x0e", "1x0e", -1, 1),                 # lmax_out < 0
    ("8x0e+8x0e", "1x0e", 1, 1),             # repeated l
    ("8x2e", "1x0e", 1, 2),                  # no path with l3 <= 1
])
def test_plan_create_statuses(ix, isx, lo, status):
    h = ctypes.c_void_p()
    st = uvu.lib.uvu_plan_create(ix.encode(), isx.encode(), lo, uvu.UVU_F32, ctypes.byref(h))
    assert st == status, uvu.uvu_last_error_message()
    if st == 0:
        assert h.value
        assert uvu.lib.uvu_plan_destroy(h) == 0
    else:
        assert not h.value
        assert uvu.uvu_last_error_message()


def test_host_argument_errors_before_any_launch():
    p = uvu.Plan("16x0e+16x1o", "1x0e+1x1o", 1)
    L = uvu.lib
    V = ctypes.c_void_p
    bad = V(0x1001)  # misaligned: rejected before anything reaches the device
    assert L.uvu_conv_fwd(None, 4, 4, None, None, None, None, None, None, None) == 1
    assert L.uvu_conv_fwd(p.handle, -1, 4, None, None, None, None, None, None, None) == 1
    assert L.uvu_conv_fwd(p.handle, 4, -2, None, None, None, None, None, None, None) == 1
    assert L.uvu_conv_fwd(p.handle, 4, 4, None, None, None, None, None, None, None) == 1
    assert L.uvu_conv_fwd(p.handle, 4, 4, bad, bad, bad, bad, bad, bad, None) == 1
    assert "aligned" in uvu.uvu_last_error_message()
    assert L.uvu_conv_bwd(p.handle, 4, 4, *[None] * 12, 7, None, 0, None) == 1  # bad dx_mode
    assert L.uvu_conv_bwd_dx(p.handle, 4, 4, None, None, None, None, None, None, None, None) == 1
    assert L.uvu_conv_bwd_edge(p.handle, 4, 4, None, None, None, None, None, None, bad, None,
                               None, None, None) == 1
    assert L.uvu_conv_bwd_dx_reduce(p.handle, 4, 4, None, None, None, None, None) == 1
    nbw = ctypes.c_size_t()
    assert L.uvu_conv_bwd_workspace(p.handle, 10, 20, uvu.UVU_DX_STAGED, ctypes.byref(nbw)) == 0
    assert nbw.value == 20 * 16 * 4 * 4
    assert L.uvu_conv_bwd_workspace(p.handle, 10, 20, uvu.UVU_DX_SENDER, ctypes.byref(nbw)) == 0
    assert nbw.value == 0
    nb = ctypes.c_size_t()
    assert L.uvu_csr_transpose_workspace(10, 20, ctypes.byref(nb)) == 0 and nb.value >= 120
    assert L.uvu_csr_transpose(10, 20, None, None, None, None, None, None, 0, None) == 1
    assert L.uvu_csr_transpose_workspace(-1, 20, ctypes.byref(nb)) == 1
    # zero nodes is a no-op that succeeds without touching the device
    assert L.uvu_conv_fwd(p.handle, 0, 0, None, None, None, None, None, None, None) == 0


def test_missing_library_fails_loudly(tmp_path, monkeypatch):
    import importlib
    import sys
    monkeypatch.setattr(uvu, "LIB_PATH", str(tmp_path / "nope.so"))
    with pytest.raises(ImportError):
        uvu._load()
    assert "clebsch_gordan_tensor_receiver_gb300.uvu" in sys.modules
    importlib.invalidate_caches()


def test_batched_tensor_product_host_checks():
    """Argument checks of the batched tensor product that run before any device work: plans with
    U < 32 are refused, negative batches are refused, and the shared-dw workspace size."""
    import pytest
    from clebsch_gordan_tensor_receiver_gb300 import uvu
    small = uvu.Plan("16x0e+16x1o", "1x0e+1x1o+1x2e", 2)
    with pytest.raises(uvu.UVUError) as ei:
        small.tp_workspace_bytes(10, True)
    assert ei.value.status == 2  # UVU_ERR_UNSUPPORTED
    p = uvu.Plan("128x0e+128x1o", "1x0e+1x1o+1x2e+1x3o", 3)
    i = p.info
    assert p.tp_workspace_bytes(10, False) == 0
    assert p.tp_workspace_bytes(10, True) == 10 * i.n_paths * i.mul * 8  # fp64 partial rows
    assert p.tp_workspace_bytes(10 ** 6, True) == 2048 * i.n_paths * i.mul * 8
    with pytest.raises(uvu.UVUError):
        p.tp_workspace_bytes(-1, True)


def test_forward_data_movement_model():
    """uvu_conv_fwd_model: the byte counts of the two forwards and the choice between them.
    MACE-medium (D_x = 4, D_out = 55) gathers little x per edge but has wide out rows, so the
    receiver-stationary forward moves less; an invariant readout of wide x (D_x = 25, D_out = 1)
    is the opposite."""
    from clebsch_gordan_tensor_receiver_gb300 import uvu
    N, E = 5000, 280000
    p = uvu.Plan("128x0e+128x1o", "1x0e+1x1o+1x2e+1x3o", 3)
    choice, br, bs = p.fwd_model(N, E)
    U, P, Dx, Dy, Do, s = 128, 13, 4, 16, 55, 4
    wY = E * (P * U + Dy) * s
    assert br == wY + E * U * Dx * s + N * U * Do * s + 4 * (N + 1) + 4 * E
    assert bs == wY + N * U * Dx * s + N * U * Do * s + 2 * E * U * Do * s + 4 * (N + 1) + 8 * E
    assert choice == uvu.UVU_FWD_RECEIVER
    q = uvu.Plan("32x0e+32x1e+32x2e+32x3e+32x4e", "1x0e", 0)
    assert q.fwd_model(N, E)[0] == uvu.UVU_FWD_SENDER


def test_mixing_host_checks():
    from clebsch_gordan_tensor_receiver_gb300 import uvu
    import pytest
    p = uvu.Plan("128x0e+128x1o", "1x0e+1x1o+1x2e+1x3o", 3)
    r = lambda b: (b + 255) // 256 * 256
    N, W, U, Do, P = 5000, 64, 128, 55, 13
    fwd, bwd = p.mix_workspace_bytes(N, W)
    # the tensor-core products' pre-split M tiles: per path, N tile and 32-wide K chunk one hi and
    # one lo tile of BN rows x 128 bytes (BN = 128 columns when N >= 128, else 64; forward: K = U,
    # N = W = 64; input gradient: K = W, N = U = 128)
    tile = lambda bn: 2 * bn * 128
    assert fwd == r(N * Do * U * 4) + r(N * Do * W * 4) + r(P * 1 * (U // 32) * tile(64))
    chunks = (7 * N + 1023) // 1024  # widest path (l3 = 3) over 1024-row chunks
    assert bwd == (r(N * Do * W * 4) + 2 * r(N * Do * U * 4) + r(P * U * W * 4) + r(chunks * P * U * W * 8) +
                   r(P * 1 * (W // 32) * tile(128)))
    for bad in (0, 5000):
        with pytest.raises(uvu.UVUError):
            p.mix_workspace_bytes(10, bad)


def test_fused_radial_host_checks_and_module():
    """The fused radial forward: its module compiles on the host for the plan's paths and the
    hidden width (weights in registers, the last layer's channel slice in shared memory when it
    fits, no spills on MACE-medium), a plan keeps one hidden width, and bad radial-network
    arguments are refused before any device work."""
    import numpy as np
    import torch
    from clebsch_gordan_tensor_receiver_gb300 import uvu
    p = uvu.Plan("128x0e+128x1o", "1x0e+1x1o+1x2e+1x3o", 3)
    src, log = p.radial_source(64)
    assert "uvu_fwd_radial" in src and "#define RD_H 64" in src and "#define RD_WSM 1" in src
    assert "#define RD_NSL 4" in src
    m = re.search(r"Function properties for uvu_fwd_radial\n.*?(\d+) bytes spill stores", log, re.S)
    assert m and int(m.group(1)) == 0, log
    with pytest.raises(uvu.UVUError) as ei:
        p.radial_source(32)
    assert ei.value.status == 2
    big = uvu.Plan("128x0e+128x1o", "1x0e+1x1o+1x2e+1x3o", 3)
    assert "#define RD_WSM 0" in big.radial_source(128)[0]  # 128 x 13 x 32 fp32 > the shared-memory budget
    q = uvu.Plan("16x0e+16x1o", "1x0e+1x1o+1x2e", 2)
    for bad in (0, 6, 260):
        with pytest.raises(uvu.UVUError) as ei:
            q.radial_source(bad)
        assert ei.value.status == 1
    import types
    r = torch.zeros(0)
    h = torch.zeros(0, 8)
    Wt = torch.zeros(64)
    st = types.SimpleNamespace(cuda_stream=0)  # no device here: the calls return before any launch
    for widths, pe, rc in (([8, 6], 5, 5.0), ([0, 8], 5, 5.0), ([8, 8], 0, 5.0), ([8, 8], 5, 0.0),
                           ([8, 8, 8, 8, 8, 8], 5, 5.0), ([65, 8], 5, 5.0), ([8, 132], 5, 5.0)):
        with pytest.raises(uvu.UVUError) as ei:
            q.radial_hidden(r, rc, pe, widths, Wt, h, stream=st)
        assert ei.value.status == 1, widths
    q.radial_hidden(r, 5.0, 5, [8, 8], Wt, h, stream=st)  # no edges: nothing to do


def test_fused_radial_forward_argument_errors():
    """uvu_conv_fwd_radial refuses bad arguments on the host, before any device work: a hidden
    width that is not a multiple of 4, NULL or misaligned tensors, negative sizes."""
    import ctypes
    import types
    import torch
    from clebsch_gordan_tensor_receiver_gb300 import uvu
    p = uvu.Plan("32x0e+32x1o", "1x0e+1x1o+1x2e+1x3o", 3)
    i = p.info
    st = types.SimpleNamespace(cuda_stream=0)
    x = torch.zeros(4, 32, i.dim_x)
    Y = torch.zeros(6, i.dim_sh)
    h = torch.zeros(6, 8)
    wl = torch.zeros(8, i.n_paths, 32)
    off = torch.zeros(5, dtype=torch.int32)
    src = torch.zeros(6, dtype=torch.int32)
    out = torch.zeros(4, 32, i.dim_out)
    vp = lambda t, k=0: ctypes.c_void_p(t.data_ptr() + k)

    def call(n_nodes=4, n_edges=6, xx=None, hidden=8, oo=None, ww=None):
        pick = lambda a, b: b if a is None else a
        uvu.uvu_conv_fwd_radial(p.handle, n_nodes, n_edges, pick(xx, vp(x)), vp(Y), vp(h), hidden, pick(ww, vp(wl)),
                                vp(off), vp(src), pick(oo, vp(out)), ctypes.c_void_p(st.cuda_stream))
    for kw, status in ((dict(hidden=6), 1), (dict(n_nodes=-1), 1), (dict(oo=ctypes.c_void_p(0)), 1),
                       (dict(xx=vp(x, 4)), 1), (dict(ww=vp(wl, 8)), 1)):
        with pytest.raises(uvu.UVUError) as ei:
            call(**kw)
        assert ei.value.status == status, kw
    call(n_nodes=0, n_edges=0)  # nothing to do: no device work
