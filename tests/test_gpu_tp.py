"""GPU parity of the batched (non-convolution) tensor product (uvu_tp_fwd / uvu_tp_bwd) against
the fp64 oracle (oracle.tp), with per-sample and batch-shared weights: element by element on
small batches (several register groups, fp64, a batch smaller than the grid), on sampled rows
of a 60,000-sample MACE-medium batch (its shared dw over the whole batch), the empty batch, and bitwise repeatability of the shared
dw (fixed-order block sums)."""
import numpy as np
import pytest
import torch

from clebsch_gordan_tensor_receiver_gb300 import uvu, workloads
from gpu_util import check, dev
from oracle import conv, paths, tp

pytestmark = pytest.mark.gpu

SH3 = "1x0e+1x1o+1x2e+1x3o"


def _run(plan, B, x, y, w, g, shared, f64):
    i = plan.info
    dt = torch.float64 if f64 else torch.float32
    out = torch.full((B, i.mul, i.dim_out), float("nan"), dtype=dt, device="cuda")
    dx = torch.full((B, i.mul, i.dim_x), float("nan"), dtype=dt, device="cuda")
    dy = torch.full((B, i.dim_sh), float("nan"), dtype=dt, device="cuda")
    dw = torch.full(w.shape, float("nan"), dtype=dt, device="cuda")
    X, Yd, W, G = dev(x), dev(y), dev(w), dev(g)
    plan.tp_fwd(B, X, Yd, W, out, w_shared=shared)
    plan.tp_bwd(B, X, Yd, W, G, dx=dx, dy=dy, dw=dw, w_shared=shared)
    torch.cuda.synchronize()
    assert plan.device_status() == 0
    return out, dx, dy, dw


CASES = [
    ("32x0e+32x1o", SH3, 3, "float32", 7),
    ("48x0e+48x1o+48x2e", SH3, 3, "float32", 40),
    ("128x0e+128x1o", SH3, 3, "float32", 300),
    ("64x0e+64x1o+64x2e", SH3, 3, "float64", 25),   # several register groups
    ("33x0e+33x1o+33x2e", SH3, 3, "float32", 13),   # x rows read directly (not 16-byte multiples)
    ("40x1o", "1x0e+1x1o+1x2e", 2, "float64", 9),   # y rows read directly, even D_out
]


@pytest.mark.parametrize("shared", [False, True], ids=["per_sample", "shared"])
@pytest.mark.parametrize("case", CASES, ids=[c[0] + "-" + c[3] for c in CASES])
def test_small_batches_all_outputs(case, shared):
    irx, irs, lo, dt, B = case
    spec = workloads.custom_spec(300 + CASES.index(case), B, irx, irs, lo, dt)
    plan = uvu.Plan(irx, irs, lo, dt)
    lay = paths.layout(irx, irs, lo)
    x, y, w, g = workloads.tp_inputs(spec, B, len(lay.paths), lay.dim_out, shared, seed=1)
    got = _run(plan, B, x, y, w, g, shared, dt == "float64")
    ref = (tp.fwd(lay, x, y, w, shared),) + tp.vjp(lay, x, y, w, g, shared)
    for name, a, b in zip(("out", "dx", "dy", "dw"), got, ref):
        check(a.cpu().numpy(), b, dt == "float64", name)


@pytest.mark.parametrize("shared", [False, True], ids=["per_sample", "shared"])
def test_medium_batch_sampled(shared):
    spec = workloads.SPECS[1]
    plan = uvu.Plan(spec.irreps_x, spec.irreps_sh, spec.lmax_out, spec.dtype)
    lay = paths.layout(spec.irreps_x, spec.irreps_sh, spec.lmax_out)
    B = 60000
    x, y, w, g = workloads.tp_inputs(spec, B, len(lay.paths), lay.dim_out, shared, seed=2)
    out, dx, dy, dw = _run(plan, B, x, y, w, g, shared, False)
    rng = np.random.default_rng(3)
    rows = np.unique(np.concatenate([rng.choice(B, 64, replace=False), [0, B - 1]]))
    ws = w if shared else w[rows]
    r_out = tp.fwd(lay, x[rows], y[rows], ws, shared)
    r_dx, r_dy, r_dw = tp.vjp(lay, x[rows], y[rows], ws, g[rows], shared)
    rt = torch.from_numpy(rows).cuda()
    check(out[rt].cpu().numpy(), r_out, False, "out")
    check(dx[rt].cpu().numpy(), r_dx, False, "dx")
    check(dy[rt].cpu().numpy(), r_dy, False, "dy")
    if shared:
        # The shared dw sums all 60,000 samples.  The oracle's C loops give it: the batched
        # product is the convolution on self loops (sample b = receiver b with the one edge b
        # from sender b, a reading the oracle's own pins tie to oracle.tp), so the per-sample dw
        # of oracle.conv.bwd_edges, summed over the batch in fp64, is the reference.  Also
        # <dw, w> = <d_out, out>, because out is linear in w.
        ref_dw = np.zeros(w.shape)
        for b0 in range(0, B, 10000):
            b1 = min(B, b0 + 10000)
            n = b1 - b0
            wb = np.broadcast_to(w, (n,) + w.shape)
            _, dwb = conv.bwd_edges(lay, np.arange(n + 1), np.arange(n), x[b0:b1], y[b0:b1], wb, g[b0:b1])
            ref_dw += dwb.sum(axis=0)
        check(dw.cpu().numpy(), ref_dw, False, "shared dw vs oracle")
        G = dev(g)
        lhs = float((dw.double() * dev(w).double()).sum())
        rhs = float((out.double() * G.double()).sum())
        assert abs(lhs - rhs) <= 1e-5 * abs(rhs), (lhs, rhs)
    else:
        check(dw[rt].cpu().numpy(), r_dw, False, "dw")
    for t in (out, dx, dy, dw):
        assert not torch.isnan(t).any()


def test_empty_batch():
    spec = workloads.SPECS[1]
    plan = uvu.Plan(spec.irreps_x, spec.irreps_sh, spec.lmax_out, spec.dtype)
    i = plan.info
    dw = torch.full((i.n_paths, i.mul), float("nan"), device="cuda")
    e = torch.empty(0, device="cuda")
    plan.tp_fwd(0, e, e, dw, torch.empty(0, 16, device="cuda"), w_shared=True)
    plan.tp_bwd(0, e, e, dw, e, dw=dw, w_shared=True)
    torch.cuda.synchronize()
    assert torch.equal(dw, torch.zeros_like(dw))


def test_shared_dw_is_bitwise_repeatable():
    spec = workloads.SPECS[1]
    plan = uvu.Plan(spec.irreps_x, spec.irreps_sh, spec.lmax_out, spec.dtype)
    lay = paths.layout(spec.irreps_x, spec.irreps_sh, spec.lmax_out)
    B = 20000
    x, y, w, g = (dev(a) for a in workloads.tp_inputs(spec, B, len(lay.paths), lay.dim_out, True, seed=4))
    a, b = torch.empty_like(w), torch.empty_like(w)
    plan.tp_bwd(B, x, y, w, g, dw=a, w_shared=True)
    plan.tp_bwd(B, x, y, w, g, dw=b, w_shared=True)
    torch.cuda.synchronize()
    assert torch.equal(a, b)
