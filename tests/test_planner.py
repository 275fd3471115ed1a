"""The host planner: its CG derivation (highest-weight state + lowering operator) agrees with the
oracle's (Racah closed form) to rounding for every triple with l <= 4; its path list and layout
match the oracle's; the emitted source compiles for sm_103a without register spills."""
import re

import numpy as np
import pytest

from clebsch_gordan_tensor_receiver_gb300 import uvu, workloads
from oracle import cg as ocg, paths as opaths

SH4 = "1x0e+1x1o+1x2e+1x3o+1x4e"


@pytest.mark.parametrize("l1", range(5))
def test_planner_cg_matches_oracle(l1):
    p = uvu.Plan(f"1x{l1}e", SH4, 8)
    triples = p.info.paths
    assert len(triples) == sum(min(l1 + l2, 8) - abs(l1 - l2) + 1 for l2 in range(5))
    for i, (a, b, c) in enumerate(triples):
        np.testing.assert_allclose(p.cg(i), ocg.real_cg(a, b, c), atol=2e-15, rtol=0,
                                   err_msg=str((a, b, c)))


@pytest.mark.parametrize("key", sorted(workloads.SPECS))
def test_paths_and_layout_match_oracle(key):
    spec = workloads.SPECS[key]
    p = uvu.Plan(spec.irreps_x, spec.irreps_sh, spec.lmax_out, spec.dtype)
    lay = opaths.layout(spec.irreps_x, spec.irreps_sh, spec.lmax_out)
    assert p.info.paths == [(q.l1, q.l2, q.l3) for q in lay.paths]
    assert (p.info.mul, p.info.dim_x, p.info.dim_sh, p.info.dim_out) == \
        (lay.mul, lay.dim_x, lay.dim_y, lay.dim_out)
    assert p.info.n_paths == {0: 9, 1: 13, 2: 24, 3: 24, 4: 24}[key]
    src, log = p.source()
    for k in ("uvu_fwd", "uvu_bwd_edge", "uvu_bwd_dx"):
        assert f"void __launch_bounds__" in src and k in src
        m = re.search(rf"Function properties for {k}\n.*?(\d+) bytes spill stores, (\d+) bytes spill loads",
                      log, re.S)
        # small spills are tolerated: a register save around the producer call, and the wide
        # (U=256, 106 output components) edge kernel, which holds the whole d_out row in
        # registers and measured faster with its staged d_out block despite a few spills
        assert m and int(m.group(1)) <= 256 and int(m.group(2)) <= 256, (k, log)


def test_cg_immediates_present_in_source():
    p = uvu.Plan("4x1o", "1x1o", 1)
    src, _ = p.source()
    # the (1,1,1) coupling is the cross product / sqrt(2): 0.707106781 appears as an immediate
    assert "7.071067" in src


def test_plan_is_identical_across_processes():
    # The planner's register-budget choice reads ptxas's report; it must see a full report in
    # every process (no cross-process compile cache short-circuiting it), so two processes emit
    # the same source.
    import subprocess
    import sys
    code = ("import hashlib; from clebsch_gordan_tensor_receiver_gb300 import uvu, workloads; "
            "s = workloads.SPECS[1]; p = uvu.Plan(s.irreps_x, s.irreps_sh, s.lmax_out, s.dtype); "
            "src, log = p.source(); print(hashlib.sha256(src.encode()).hexdigest(), 'Used' in log)")
    outs = [subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, check=True,
                           cwd=__import__("conftest").ROOT).stdout.split() for _ in range(2)]
    assert outs[0] == outs[1] and outs[0][1] == "True"


@pytest.mark.parametrize("key", sorted(workloads.SPECS))
def test_hvp_kernels_build_on_the_host(key):
    """The double-backward module compiles without a device; plans with U >= 32 get the
    bulk-copy pipelined kernels (stages carrying the cotangent rows too), smaller ones the
    direct-load kernels."""
    spec = workloads.SPECS[key]
    p = uvu.Plan(spec.irreps_x, spec.irreps_sh, spec.lmax_out, spec.dtype)
    src, log = p.hvp_source()
    for k in ("uvu_hvp_fwd", "uvu_hvp_edge"):
        assert f"Function properties for {k}" in log
    assert ("cp.async.bulk" in src) == (p.info.mul >= 32)
    if p.info.mul >= 32:
        assert "if (hm & 4) bulk_g2s" in src  # aw rows staged only when present
    assert p.hvp_source()[0] == src  # compiled once per plan


def _run_child(code, env):
    import os, subprocess, sys
    e = dict(os.environ)
    e.update(env)
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    return subprocess.run([sys.executable, "-c", code], cwd=root, env=e, capture_output=True, text=True, timeout=300)


_CHILD = """
from clebsch_gordan_tensor_receiver_gb300 import uvu
try:
    p = uvu.Plan("48x0e+48x1o", "1x0e+1x1o+1x2e", 2)
    src, log = p.source()
    print("OK", len(src), "Function properties for uvu_fwd" in log)
except uvu.UVUError as e:
    print("ERR", e.status, str(e))
"""


def test_compile_failure_injection():
    """UVU_FAIL_COMPILE=1 (host-side fault injection): plan creation reports UVU_ERR_COMPILE with
    the injected message and nothing crashes."""
    r = _run_child(_CHILD, {"UVU_FAIL_COMPILE": "1"})
    assert r.returncode == 0, r.stderr
    assert r.stdout.startswith("ERR 3") and "injected" in r.stdout, r.stdout


def test_disk_cache_and_source_dump(tmp_path):
    """UVU_CACHE_DIR keeps one file per emitted source with the cubin and the NVRTC log (the
    register/spill report survives a cache hit); UVU_DUMP_SOURCE writes the emitted CUDA C++."""
    cache, dump = tmp_path / "cache", tmp_path / "dump"
    cache.mkdir()
    dump.mkdir()
    env = {"UVU_CACHE_DIR": str(cache), "UVU_DUMP_SOURCE": str(dump)}
    first = _run_child(_CHILD, env)
    assert first.stdout.startswith("OK") and first.stdout.strip().endswith("True"), first.stdout + first.stderr
    files = sorted(f.name for f in cache.iterdir())
    assert files and all(f.startswith("uvu_") and f.endswith(".bin") for f in files)
    stamp = {f.name: f.stat().st_mtime_ns for f in cache.iterdir()}
    second = _run_child(_CHILD, env)
    assert second.stdout == first.stdout
    assert {f.name: f.stat().st_mtime_ns for f in cache.iterdir()} == stamp  # served from the cache
    dumped = list(dump.glob("uvu_*.cu"))
    assert dumped and "uvu_fwd" in dumped[0].read_text()


def test_unwritable_cache_dir_is_harmless(tmp_path):
    """A cache directory that cannot be written (here: a path under a regular file) does not fail
    plan creation; the plan compiles and runs from memory."""
    blocker = tmp_path / "file"
    blocker.write_text("x")
    r = _run_child(_CHILD, {"UVU_CACHE_DIR": str(blocker / "sub")})
    assert r.returncode == 0 and r.stdout.startswith("OK"), r.stdout + r.stderr


@pytest.mark.parametrize("env", [
    {"UVU_RAD_SPLIT": "2", "UVU_RAD_RW": "8", "UVU_RAD_MINB": "2"},
    {"UVU_RAD_PACK": "0"},
    {"UVU_RAD_PREFETCH": "2"},
    {"UVU_PACK_PRODUCTS": "0"},
], ids=["radial-split", "radial-unpaired", "radial-prefetch-h", "scalar-products"])
def test_tuning_variants_build_on_the_host(env, monkeypatch):
    """The emission variants selected by tuning switches (measured, not the defaults) still
    generate code that compiles for sm_103a without spills on MACE-medium, and differ from the
    default source (which pairs the fp32 products)."""
    for k, v in env.items():
        monkeypatch.setenv(k, v)
    p = uvu.Plan("128x0e+128x1o", "1x0e+1x1o+1x2e+1x3o", 3)
    for monkey_k in env:
        monkeypatch.delenv(monkey_k)
    base = uvu.Plan("128x0e+128x1o", "1x0e+1x1o+1x2e+1x3o", 3)
    for k, v in env.items():
        monkeypatch.setenv(k, v)
    if "UVU_PACK_PRODUCTS" in env:
        src, log = p.source()
        assert "mul.rn.f32x2" not in src and "mul.rn.f32x2" in base.source()[0]
        names = ("uvu_fwd", "uvu_bwd_edge")
    else:
        src, log = p.radial_source(64)
        for k in env:
            monkeypatch.delenv(k)
        assert src != base.radial_source(64)[0]
        names = ("uvu_fwd_radial",)
    for k in names:
        m = re.search(rf"Function properties for {k}\n.*?(\d+) bytes spill stores", log, re.S)
        assert m and int(m.group(1)) == 0, (k, log)


_EDGE_SWITCHES = [("UVU_COL_SCALE", "0"), ("UVU_PAIR_CONTRACT", "0"), ("UVU_ID_FOLD", "0"),
                  ("UVU_EDGE_BULK_OUT", "0"), ("UVU_GSM_VEC", "0"), ("UVU_DY_SMEM", "0"),
                  ("UVU_REDUCE_GROUP", "4")]


def test_edge_kernel_forms_present_by_default():
    """The default emission carries the edge-kernel forms measured faster: on MACE-medium the
    column-scaled d_out row, the folded identity paths and the paired dY/dx contractions; on
    MACE-large (staged d_out rows) the paired staged reads, the shared-memory dY tile and the
    dw / dx-partial bulk copies out of the stage; on both the flat-row dx reduction."""
    med = uvu.Plan("128x0e+128x1o", "1x0e+1x1o+1x2e+1x3o", 3).source()[0]
    assert "zi_1" in med and "uvu_f2fma(xb_" in med and "gv_19 = 5.773502" in med
    assert "reinterpret_cast<float4*>(dx + (size_t)sn * (UVU_U * UVU_DX))[c]" in med
    large = uvu.Plan("128x0e+128x1o+128x2e", "1x0e+1x1o+1x2e+1x3o", 3).source()[0]
    assert "gq2_" in large and "EG_DYT" in large and "bulk_s2g(dw" in large and "gw[" in large


@pytest.mark.parametrize("name,value", _EDGE_SWITCHES, ids=[n for n, _ in _EDGE_SWITCHES])
def test_edge_kernel_switches_build_on_the_host(name, value, monkeypatch):
    """Each edge-kernel tuning switch changes the emitted source of a plan it applies to, and the
    result still compiles for sm_103a with at most a call-site register save of spill."""
    irreps = "128x0e+128x1o+128x2e" if name in ("UVU_GSM_VEC", "UVU_DY_SMEM", "UVU_EDGE_BULK_OUT") else "128x0e+128x1o"
    base = uvu.Plan(irreps, "1x0e+1x1o+1x2e+1x3o", 3).source()[0]
    monkeypatch.setenv(name, value)
    p = uvu.Plan(irreps, "1x0e+1x1o+1x2e+1x3o", 3)
    src, log = p.source()
    assert src != base
    for k in ("uvu_bwd_edge", "uvu_bwd_dx_reduce"):
        m = re.search(rf"Function properties for {k}\n.*?(\d+) bytes spill stores", log, re.S)
        assert m and int(m.group(1)) <= 64, (k, log)
