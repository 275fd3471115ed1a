"""The tensor-core product kernel at shapes away from the MACE sizes, against fp64 products of the
same inputs: the radial last layer and its input gradient for hidden widths whose K is not a
multiple of the 32-wide chunk (4, 36, 100) or spans several accumulation ranges (dh: K = P U up to
3,328), output widths that leave a partial 64- or 128-column tile, and the channel mixing with
W != U, widths that are not multiples of 32, and row counts that leave partial 128-row tiles in
every path segment.  Tolerance: relative Frobenius <= 1e-5 and |d| <= 1e-4 (1 + |ref|)."""
import numpy as np
import pytest
import torch

from clebsch_gordan_tensor_receiver_gb300 import uvu, workloads
from gpu_util import check, dev
from oracle import mix as omix
from oracle import paths

pytestmark = pytest.mark.gpu

SH3 = "1x0e+1x1o+1x2e+1x3o"


@pytest.mark.parametrize("hidden,U,E", [(4, 32, 300), (36, 36, 1000), (100, 20, 777), (132, 64, 513), (256, 128, 129)])
def test_radial_products(hidden, U, E):
    spec = workloads.custom_spec(900 + hidden, 30, f"{U}x0e+{U}x1o", SH3, 3, "float32")
    plan = uvu.Plan(spec.irreps_x, spec.irreps_sh, spec.lmax_out, spec.dtype)
    P = plan.info.n_paths
    rng = np.random.default_rng(hidden * 7 + U)
    h = rng.standard_normal((E, hidden)).astype(np.float32)
    wl = (rng.standard_normal((hidden, P, U)) / np.sqrt(hidden)).astype(np.float32)
    dw = rng.standard_normal((E, P, U)).astype(np.float32)
    w = torch.empty(E, P, U, device="cuda")
    plan.radial_weights(dev(h), dev(wl), w)
    dh = torch.empty(E, hidden, device="cuda")
    plan.radial_weights_bwd(dev(h), dev(wl), dev(dw), dh=dh)
    torch.cuda.synchronize()
    check(w.cpu().numpy(), np.einsum("ek,kpu->epu", h.astype(np.float64), wl.astype(np.float64)), False, "w")
    check(dh.cpu().numpy(), np.einsum("epu,kpu->ek", dw.astype(np.float64), wl.astype(np.float64)), False, "dh")
    assert plan.device_status() == 0


@pytest.mark.parametrize("U,W,N", [(36, 20, 97), (64, 132, 301), (128, 260, 130), (32, 128, 1)])
def test_mixing_products(U, W, N):
    spec = workloads.custom_spec(950 + U, 40, f"{U}x0e+{U}x1o", SH3, 3, "float32")
    plan = uvu.Plan(spec.irreps_x, spec.irreps_sh, spec.lmax_out, spec.dtype)
    lay = paths.layout(spec.irreps_x, spec.irreps_sh, spec.lmax_out)
    P, Do = plan.info.n_paths, plan.info.dim_out
    rng = np.random.default_rng(U * 3 + W + N)
    inp = rng.standard_normal((N, U, Do)).astype(np.float32)
    M = (rng.standard_normal((P, U, W)) / np.sqrt(U)).astype(np.float32)
    g = rng.standard_normal((N, W, Do)).astype(np.float32)
    out = torch.empty(N, W, Do, device="cuda")
    plan.mix_fwd(N, W, dev(inp), dev(M), out)
    d_in = torch.empty(N, U, Do, device="cuda")
    dM = torch.empty(P, U, W, device="cuda")
    plan.mix_bwd(N, W, dev(inp), dev(M), dev(g), d_in=d_in, dM=dM)
    torch.cuda.synchronize()
    check(out.cpu().numpy(), omix.fwd(lay, inp, M), False, "out")
    r_din, r_dM = omix.vjp(lay, inp, M, g)
    check(d_in.cpu().numpy(), r_din, False, "d_in")
    check(dM.cpu().numpy(), r_dM, False, "dM")
    assert plan.device_status() == 0
