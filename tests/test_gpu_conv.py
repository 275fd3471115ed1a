"""GPU parity of the convolution kernels against the fp64 oracle, through the C ABI.

Small workloads are compared element by element over every output; the full-size workloads in
the configuration the benchmark times are compared on sampled receivers, edges and senders
(each sampled element computed by the oracle from its full definition) and by the adjoint
identities, which hold at any size."""
import numpy as np
import pytest
import torch

from clebsch_gordan_tensor_receiver_gb300 import uvu, workloads
from gpu_util import Problem, check, dev

pytestmark = pytest.mark.gpu

SH3 = "1x0e+1x1o+1x2e+1x3o"
MODES = (uvu.UVU_DX_SENDER, uvu.UVU_DX_ATOMIC, uvu.UVU_DX_STAGED)


def _full_compare(P):
    out = P.fwd().cpu().numpy()
    check(out, P.ref_out(), P.f64, "out")
    rdY, rdw = P.ref_edges()
    rdx = P.ref_dx()
    for mode in MODES:
        dx, dY, dw = (t.cpu().numpy() for t in P.bwd(mode))
        check(dY, rdY, P.f64, "dY")
        check(dw, rdw, P.f64, "dw")
        check(dx, rdx, P.f64, f"dx mode {mode}")
    assert P.status_ok()


def test_tiny_workload_all_outputs():
    _full_compare(Problem.from_spec(0))


CUSTOM = [
    # irreps_x, irreps_sh, lmax_out, dtype, N, max degree
    ("48x0e+48x1o+48x2e", SH3, 3, "float32", 37, 12),     # channel padding, ragged degrees
    ("96x0e+96x1o", SH3, 3, "float32", 21, 9),            # three warps per owner
    ("32x0e", "1x0e", 0, "float32", 40, 7),               # scalar path only
    ("8x1o+8x2e", "1x0e+1x1o+1x2e", 4, "float64", 19, 6),  # narrow fp64, pseudo-tensor outputs
    ("64x0e+64x1o+64x2e", SH3, 3, "float64", 23, 8),      # fp64 with register groups
    ("3x0e+3x1o", "1x0e+1x1o+1x2e", 2, "float32", 11, 5),  # three channels
    ("128x0e+128x1o", SH3, 3, "float32", 300, 70),        # medium shapes, ragged, many chunks
    ("33x0e+33x1o+33x2e", SH3, 3, "float32", 29, 9),      # pipelined, x rows not 16-byte multiples (no bulk x)
    ("40x1o", "1x0e+1x1o+1x2e", 2, "float64", 17, 7),     # pipelined, Y rows not bulk, even D_out (padded stride)
    ("32x1o+32x4e", "1x0e+1x1o+1x2e+1x3o+1x4e", 4, "float32", 13, 6),  # l = 4 everywhere: 27 paths, D_out 159
]


@pytest.mark.parametrize("case", CUSTOM, ids=[c[0] + "-" + c[3] for c in CUSTOM])
def test_custom_workloads_all_outputs(case):
    irx, irs, lo, dt, N, dmax = case
    spec = workloads.custom_spec(100 + CUSTOM.index(case), N, irx, irs, lo, dt)
    rng = np.random.default_rng(CUSTOM.index(case))
    deg = rng.integers(0, dmax + 1, size=N)
    deg[[0, N // 2, N - 1]] = [0, dmax, 0]
    recv, src = workloads.random_degree_graph(N, deg, rng)
    vec = workloads.unit_vectors(src.size, rng)
    lsh = int(irs.split("+")[-1].split("x")[1][:-1])
    # Y is an input of the convolution: SH values up to l = 3, plain normal values beyond
    Y = (workloads.sh_inputs(vec, lsh) if lsh <= 3 else rng.standard_normal((src.size, workloads.dim_of(irs)))).astype(dt)
    mul = int(irx.split("x")[0])
    x = rng.standard_normal((N, mul, workloads.dim_of(irx))).astype(dt)
    _full_compare(Problem(spec, recv, src, x, Y, N))


def test_no_edges_writes_zeros():
    spec = workloads.custom_spec(150, 9, "32x0e+32x1o", SH3, 3)
    recv = np.zeros(0, np.int32)
    src = np.zeros(0, np.int32)
    x = np.ones((9, 32, 4), np.float32)
    P = Problem(spec, recv, src, x, np.zeros((0, 16), np.float32), 9)
    assert torch.all(P.fwd() == 0)
    for mode in MODES:
        dx, dY, dw = P.bwd(mode)
        assert torch.all(dx == 0) and dY.numel() == 0 and dw.numel() == 0


def _sample(n, k, rng):
    s = rng.choice(n, size=min(k, n), replace=False)
    return np.unique(np.concatenate([s, [0, n - 1]]))


@pytest.mark.parametrize("key", [1, 2, 3, 4])
def test_full_size_sampled(key):
    P = Problem.from_spec(key)
    rng = np.random.default_rng(1000 + key)
    rs = _sample(P.N, 48, rng)
    es = _sample(P.E, 192, rng)
    ss = _sample(P.N, 48, rng)
    rs_t, es_t, ss_t = (torch.from_numpy(a).cuda() for a in (rs, es, ss))
    out = P.fwd()
    check(out[rs_t].cpu().numpy(), P.ref_out(rs), P.f64, "out")
    rdY, rdw = P.ref_edges(es)
    rdx = P.ref_dx(ss)
    for mode in MODES:
        dx, dY, dw = P.bwd(mode)
        check(dY[es_t].cpu().numpy(), rdY, P.f64, "dY")
        check(dw[es_t].cpu().numpy(), rdw, P.f64, "dw")
        check(dx[ss_t].cpu().numpy(), rdx, P.f64, f"dx mode {mode}")
        assert not torch.isnan(dx).any() and not torch.isnan(dY).any() and not torch.isnan(dw).any()
    assert not torch.isnan(out).any()
    # adjoint identities over the whole problem: <d_out,out> = <dx,x> = <dY,Y> = <dw,w>
    dx, dY, dw = P.bwd(uvu.UVU_DX_SENDER)
    s = lambda a, b: float((a.double() * b.double()).sum())
    ref = s(out, P.d["g"])
    tol = 1e-10 if P.f64 else 2e-5
    for a, b, name in ((dx, P.d["x"], "dx"), (dY, P.d["Y"], "dY"), (dw, P.d["w"], "dw")):
        assert s(a, b) == pytest.approx(ref, rel=tol), name
    assert P.status_ok()


@pytest.mark.parametrize("mode", [uvu.UVU_DX_SENDER, uvu.UVU_DX_STAGED])
def test_deterministic_kernels_repeat_bitwise(mode):
    P = Problem.from_spec(1)
    o1 = P.fwd()
    a1 = P.bwd(mode)
    for _ in range(2):
        assert torch.equal(P.fwd(), o1)
        a2 = P.bwd(mode)
        for t1, t2 in zip(a1, a2):
            assert torch.equal(t1, t2)
    assert P.status_ok()


def test_graph_validate():
    P = Problem.from_spec(0)
    ws = torch.zeros(2, dtype=torch.int64, device="cuda")
    import ctypes
    nbad = ctypes.c_int64(-1)
    uvu.uvu_graph_validate(P.N, P.E, ctypes.c_void_p(P.G.recv_offsets.data_ptr()),
                           ctypes.c_void_p(P.d["src"].data_ptr()), ctypes.c_void_p(ws.data_ptr()),
                           ctypes.byref(nbad), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert nbad.value == 0
    bad_src = P.d["src"].clone()
    bad_src[5] = P.N + 3
    bad_src[7] = -1
    uvu.uvu_graph_validate(P.N, P.E, ctypes.c_void_p(P.G.recv_offsets.data_ptr()),
                           ctypes.c_void_p(bad_src.data_ptr()), ctypes.c_void_p(ws.data_ptr()),
                           ctypes.byref(nbad), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert nbad.value == 2


def test_receiver_subranges_match_whole_graph():
    # offsets are absolute edge indices, so recv_offsets + r0 with n_nodes = r1 - r0 computes the
    # receivers [r0, r1) exactly as a whole-graph call does (the chunked host pipeline relies on it)
    P = Problem.from_spec(workloads.custom_spec(160, 333, "64x0e+64x1o+64x2e", SH3, 3, degree=9))
    i = P.plan.info
    out_ref = P.fwd()
    dxe_ref = torch.empty(P.E, i.mul, i.dim_x, device="cuda")
    dY_ref = torch.empty(P.E, i.dim_sh, device="cuda")
    dw_ref = torch.empty(P.E, i.n_paths, i.mul, device="cuda")
    P.plan.bwd_edge(P.N, P.d["x"], P.d["Y"], P.d["w"], P.G.recv_offsets, P.d["src"], P.d["g"],
                    dY=dY_ref, dw=dw_ref, dx_edge=dxe_ref)
    out = torch.full_like(out_ref, float("nan"))
    dxe, dY, dw = (torch.full_like(t, float("nan")) for t in (dxe_ref, dY_ref, dw_ref))
    for a, b in ((0, 17), (17, 200), (200, 333)):
        ro = P.G.recv_offsets[a:]
        P.plan.fwd(b - a, P.d["x"], P.d["Y"], P.d["w"], ro, P.d["src"], out[a:])
        P.plan.bwd_edge(b - a, P.d["x"], P.d["Y"], P.d["w"], ro, P.d["src"], P.d["g"][a:],
                        dY=dY, dw=dw, dx_edge=dxe)
    for got, want in ((out, out_ref), (dxe, dxe_ref), (dY, dY_ref), (dw, dw_ref)):
        assert torch.equal(got, want)
    assert P.status_ok()


def test_one_plan_over_changing_graphs():
    """One plan serves graphs of any size in sequence (the plan depends on the irreps only):
    growing, shrinking and empty graphs, each checked against the oracle."""
    spec0 = workloads.custom_spec(170, 10, "32x0e+32x1o", SH3, 3)
    plan = None
    rng = np.random.default_rng(17)
    for N, dmax in ((10, 4), (57, 20), (3, 0), (31, 9), (1, 2)):
        spec = workloads.custom_spec(170, N, "32x0e+32x1o", SH3, 3)
        deg = rng.integers(0, dmax + 1, size=N)
        recv, src = workloads.random_degree_graph(N, deg, rng)
        Y = workloads.sh_inputs(workloads.unit_vectors(src.size, rng), 3).astype(np.float32)
        x = rng.standard_normal((N, 32, 4)).astype(np.float32)
        P = Problem(spec, recv, src, x, Y, N)
        if plan is None:
            plan = P.plan
        P.plan = plan  # the same plan object for every graph
        _full_compare(P)
    assert spec0.n_nodes == 10
