"""GPU parity of the double backward (uvu_conv_hvp) against the fp64 oracle.

The oracle's double backward (oracle.hvp) is pinned by finite differences of its VJP; here the
CUDA kernels are compared with it element by element on small workloads (including absent
cotangents, a plan with several register groups whose pipelined edge kernel sums the per-edge
grad_x partials across groups in shared memory, and a direct-load plan with U < 32) and on
sampled outputs of the full MACE-medium workload."""
import numpy as np
import pytest
import torch

from clebsch_gordan_tensor_receiver_gb300 import workloads
from gpu_util import Problem, check, dev
from oracle import conv, hvp

pytestmark = pytest.mark.gpu

SH3 = "1x0e+1x1o+1x2e+1x3o"


def _cotangents(P, seed):
    rng = np.random.default_rng(seed)
    dt = np.float64 if P.f64 else np.float32
    return (rng.standard_normal(P.x.shape).astype(dt), rng.standard_normal(P.Y.shape).astype(dt),
            rng.standard_normal(P.w.shape).astype(dt))


def _gpu_hvp(P, ax, aY, aw):
    i = P.plan.info
    outs = [P.empty(P.N, i.mul, i.dim_out), P.empty(P.N, i.mul, i.dim_x),
            P.empty(max(P.E, 1), i.dim_sh), P.empty(max(P.E, 1), i.n_paths, i.mul)]
    for t in outs:
        t.fill_(float("nan"))
    P.plan.hvp(P.N, P.d["x"], P.d["Y"], P.d["w"], P.G.recv_offsets, P.d["src"], P.G.send_offsets,
               P.G.send_eids, P.d["g"], ax=None if ax is None else dev(ax),
               aY=None if aY is None else dev(aY), aw=None if aw is None else dev(aw),
               grad_d_out=outs[0], grad_x=outs[1], grad_Y=outs[2], grad_w=outs[3])
    torch.cuda.synchronize()
    assert P.status_ok()
    return outs[0], outs[1], outs[2][:P.E], outs[3][:P.E]


def _full_compare(P, seed, drop=()):
    ax, aY, aw = _cotangents(P, seed)
    ax = None if "ax" in drop else ax
    aY = None if "aY" in drop else aY
    aw = None if "aw" in drop else aw
    got = _gpu_hvp(P, ax, aY, aw)
    ref = hvp.hvp(P.lay, P.off_host, P.src, P.x, P.Y, P.w, P.g, ax, aY, aw, P.N)
    for name, a, b in zip(("grad_d_out", "grad_x", "grad_Y", "grad_w"), got, ref):
        check(a.cpu().numpy(), b, P.f64, name)


def test_tiny_workload_all_outputs():
    _full_compare(Problem.from_spec(0), 1)


CUSTOM = [
    ("48x0e+48x1o+48x2e", SH3, 3, "float32", 29, 9),
    ("64x0e+64x1o+64x2e", SH3, 3, "float64", 17, 6),   # several register groups
    ("8x1o+8x2e", "1x0e+1x1o+1x2e", 4, "float32", 13, 5),
    ("33x0e+33x1o+33x2e", SH3, 3, "float32", 15, 6),      # pipelined, x and ax rows read directly
    ("40x1o", "1x0e+1x1o+1x2e", 2, "float64", 11, 5),     # pipelined, Y and aY rows read directly
    ("32x2e+32x4e", "1x0e+1x2e+1x4e", 4, "float32", 9, 4),  # l = 4 paths
]


@pytest.mark.parametrize("case", CUSTOM, ids=[c[0] + "-" + c[3] for c in CUSTOM])
def test_custom_workloads(case):
    irx, irs, lo, dt, N, dmax = case
    spec = workloads.custom_spec(200 + CUSTOM.index(case), N, irx, irs, lo, dt)
    rng = np.random.default_rng(50 + CUSTOM.index(case))
    deg = rng.integers(0, dmax + 1, size=N)
    deg[0] = 0
    recv, src = workloads.random_degree_graph(N, deg, rng)
    lsh = int(irs.split("+")[-1].split("x")[1][:-1])
    # Y is an input of the convolution: SH values up to l = 3, plain normal values beyond
    Y = (workloads.sh_inputs(workloads.unit_vectors(src.size, rng), lsh) if lsh <= 3
         else rng.standard_normal((src.size, workloads.dim_of(irs)))).astype(dt)
    x = rng.standard_normal((N, int(irx.split("x")[0]), workloads.dim_of(irx))).astype(dt)
    _full_compare(Problem(spec, recv, src, x, Y, N), 7)


@pytest.mark.parametrize("drop", [("ax",), ("aY",), ("aw",), ("ax", "aY", "aw")])
def test_absent_cotangents_count_as_zero(drop):
    _full_compare(Problem.from_spec(0), 3, drop)


def test_full_size_sampled():
    P = Problem.from_spec(1)
    ax, aY, aw = _cotangents(P, 11)
    got = _gpu_hvp(P, ax, aY, aw)
    rng = np.random.default_rng(12)
    rs = np.unique(np.concatenate([rng.choice(P.N, 24, replace=False), [0, P.N - 1]]))
    es = np.unique(np.concatenate([rng.choice(P.E, 96, replace=False), [0, P.E - 1]]))
    L, off, s = P.lay, P.off_host, P.src
    ref_g = (conv.fwd(L, off, s, ax, P.Y, P.w, rs) + conv.fwd(L, off, s, P.x, aY, P.w, rs)
             + conv.fwd(L, off, s, P.x, P.Y, aw, rs))
    ref_x = (conv.bwd_dx(L, off, s, aY, P.w, P.g, P.N, rs) + conv.bwd_dx(L, off, s, P.Y, aw, P.g, P.N, rs))
    dY_a, dw_a = conv.bwd_edges(L, off, s, ax, P.Y, P.w, P.g, es)
    dY_w, _ = conv.bwd_edges(L, off, s, P.x, P.Y, aw, P.g, es)
    _, dw_y = conv.bwd_edges(L, off, s, P.x, aY, P.w, P.g, es)
    r_t, e_t = torch.from_numpy(rs).cuda(), torch.from_numpy(es).cuda()
    check(got[0][r_t].cpu().numpy(), ref_g, False, "grad_d_out")
    check(got[1][r_t].cpu().numpy(), ref_x, False, "grad_x")
    check(got[2][e_t].cpu().numpy(), dY_a + dY_w, False, "grad_Y")
    check(got[3][e_t].cpu().numpy(), dw_a + dw_y, False, "grad_w")
    for t in got:
        assert not torch.isnan(t).any()


def test_deterministic_repeat():
    P = Problem.from_spec(1)
    ax, aY, aw = _cotangents(P, 5)
    a = _gpu_hvp(P, ax, aY, aw)
    b = _gpu_hvp(P, ax, aY, aw)
    for t1, t2 in zip(a, b):
        assert torch.equal(t1, t2)
