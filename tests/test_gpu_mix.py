"""GPU parity of the channel mixing (uvu_mix_fwd / uvu_mix_bwd) and of the factorised UVW
convolution (uvu_conv_uvw_fwd) against the fp64 oracle (oracle.mix): small plans in fp32 and
fp64 with W different from U, the UVW convolution against its edge-by-edge brute force, the
full MACE-medium size (5,000 receivers, W = 128) and bitwise repeatability of dM."""
import numpy as np
import pytest
import torch

from clebsch_gordan_tensor_receiver_gb300 import uvu, workloads
from gpu_util import Problem, check, dev
from oracle import mix, paths

pytestmark = pytest.mark.gpu

SH3 = "1x0e+1x1o+1x2e+1x3o"


def _mix_all(plan, lay, N, W, inp, M, g, f64):
    dt = torch.float64 if f64 else torch.float32
    out = torch.full((N, W, lay.dim_out), float("nan"), dtype=dt, device="cuda")
    d_in = torch.full(inp.shape, float("nan"), dtype=dt, device="cuda")
    dM = torch.full(M.shape, float("nan"), dtype=dt, device="cuda")
    I, Md, G = dev(inp), dev(M), dev(g)
    plan.mix_fwd(N, W, I, Md, out)
    plan.mix_bwd(N, W, I, Md, G, d_in=d_in, dM=dM)
    torch.cuda.synchronize()
    return out, d_in, dM


CASES = [("16x0e+16x1o", "1x0e+1x1o+1x2e", 2, "float32", 11, 24),
         ("48x0e+48x1o+48x2e", SH3, 3, "float32", 9, 200),
         ("64x0e+64x1o+64x2e", SH3, 3, "float64", 7, 64)]


@pytest.mark.parametrize("case", CASES, ids=[c[0] + "-" + c[3] for c in CASES])
def test_mixing_small(case):
    irx, irs, lo, dt, N, W = case
    plan = uvu.Plan(irx, irs, lo, dt)
    lay = paths.layout(irx, irs, lo)
    rng = np.random.default_rng(CASES.index(case))
    U = lay.mul
    inp = rng.standard_normal((N, U, lay.dim_out)).astype(dt)
    M = rng.standard_normal((len(lay.paths), U, W)).astype(dt)
    g = rng.standard_normal((N, W, lay.dim_out)).astype(dt)
    got = _mix_all(plan, lay, N, W, inp, M, g, dt == "float64")
    ref = (mix.fwd(lay, inp, M),) + mix.vjp(lay, inp, M, g)
    for name, a, b in zip(("out", "d_in", "dM"), got, ref):
        check(a.cpu().numpy(), b, dt == "float64", name)


def test_factorised_uvw_convolution():
    spec = workloads.custom_spec(500, 19, "32x0e+32x1o+32x2e", SH3, 3, "float32")
    rng = np.random.default_rng(50)
    deg = rng.integers(0, 6, size=19)
    recv, src = workloads.random_degree_graph(19, deg, rng)
    Y = workloads.sh_inputs(workloads.unit_vectors(src.size, rng), 3).astype(np.float32)
    x = rng.standard_normal((19, 32, 9)).astype(np.float32)
    P = Problem(spec, recv, src, x, Y, 19)
    W = 40
    M = rng.standard_normal((len(P.lay.paths), 32, W)).astype(np.float32)
    uvu_out = P.empty(19, 32, P.lay.dim_out)
    out = P.empty(19, W, P.lay.dim_out).fill_(float("nan"))
    P.plan.uvw_fwd(19, P.d["x"], P.d["Y"], P.d["w"], P.G.recv_offsets, P.d["src"], dev(M), W, uvu_out, out)
    torch.cuda.synchronize()
    ref = mix.uvw_conv_brute(P.lay, recv, src, x, Y, P.w, M, 19)
    check(out.cpu().numpy(), ref, False, "uvw out")


def test_mixing_medium_size():
    spec = workloads.SPECS[1]
    plan = uvu.Plan(spec.irreps_x, spec.irreps_sh, spec.lmax_out, spec.dtype)
    lay = paths.layout(spec.irreps_x, spec.irreps_sh, spec.lmax_out)
    N, W = 5000, 128
    rng = np.random.default_rng(7)
    inp = rng.standard_normal((N, 128, lay.dim_out), dtype=np.float32)
    M = (rng.standard_normal((len(lay.paths), 128, W), dtype=np.float32) / np.float32(np.sqrt(128)))
    g = rng.standard_normal((N, W, lay.dim_out), dtype=np.float32)
    out, d_in, dM = _mix_all(plan, lay, N, W, inp, M, g, False)
    rows = np.unique(np.concatenate([rng.choice(N, 48, replace=False), [0, N - 1]]))
    rt = torch.from_numpy(rows).cuda()
    check(out[rt].cpu().numpy(), mix.fwd(lay, inp[rows], M), False, "out")
    r_din, r_dM = mix.vjp(lay, inp, M, g)
    check(d_in[rt].cpu().numpy(), r_din[rows], False, "d_in")
    check(dM.cpu().numpy(), r_dM, False, "dM")
    dM2 = torch.empty_like(dM)
    plan.mix_bwd(N, W, dev(inp), dev(M), dev(g), dM=dM2)
    torch.cuda.synchronize()
    assert torch.equal(dM, dM2)
