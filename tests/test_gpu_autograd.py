"""PyTorch autograd through the library (autograd.uvu_conv): first derivatives against the oracle's
VJP and second derivatives (create_graph=True, then a second grad) against the oracle's double
backward, on the tiny workload and a pipelined MACE-medium-irreps graph."""
import numpy as np
import pytest
import torch

from clebsch_gordan_tensor_receiver_gb300 import autograd, uvu, workloads
from gpu_util import Problem, check, dev
from oracle import conv, hvp

pytestmark = pytest.mark.gpu


def _problems():
    yield Problem.from_spec(0)
    spec = workloads.custom_spec(700, 40, "64x0e+64x1o", "1x0e+1x1o+1x2e+1x3o", 3, "float32")
    rng = np.random.default_rng(70)
    recv, src = workloads.random_degree_graph(40, rng.integers(0, 9, size=40), rng)
    Y = workloads.sh_inputs(workloads.unit_vectors(src.size, rng), 3).astype(np.float32)
    x = rng.standard_normal((40, 64, 4)).astype(np.float32)
    yield Problem(spec, recv, src, x, Y, 40)


@pytest.mark.parametrize("which", [0, 1], ids=["tiny", "pipelined"])
def test_first_and_second_derivatives(which):
    P = list(_problems())[which]
    rng = np.random.default_rng(5)
    x, Y, w = (dev(a).requires_grad_(True) for a in (P.x, P.Y, P.w))
    out = autograd.uvu_conv(x, Y, w, P.plan, P.G)
    check(out.detach().cpu().numpy(), conv.fwd(P.lay, P.off_host, P.src, P.x, P.Y, P.w), False, "out")
    c = P.g  # the cotangent of out
    gx, gY, gw = torch.autograd.grad((out * dev(c)).sum(), (x, Y, w), create_graph=True)
    r_dY, r_dw = conv.bwd_edges(P.lay, P.off_host, P.src, P.x, P.Y, P.w, c)
    check(gx.detach().cpu().numpy(), conv.bwd_dx(P.lay, P.off_host, P.src, P.Y, P.w, c, P.N), False, "dx")
    check(gY.detach().cpu().numpy(), r_dY, False, "dY")
    check(gw.detach().cpu().numpy(), r_dw, False, "dw")
    ax, aY, aw = (rng.standard_normal(a.shape).astype(np.float32) for a in (P.x, P.Y, P.w))
    l2 = (gx * dev(ax)).sum() + (gY * dev(aY)).sum() + (gw * dev(aw)).sum()
    hx, hY, hw = torch.autograd.grad(l2, (x, Y, w))
    _, r_x, r_Y, r_w = hvp.hvp(P.lay, P.off_host, P.src, P.x, P.Y, P.w, c, ax, aY, aw, P.N)
    check(hx.cpu().numpy(), r_x, False, "d2 x")
    check(hY.cpu().numpy(), r_Y, False, "d2 Y")
    check(hw.cpu().numpy(), r_w, False, "d2 w")
    assert P.status_ok()
