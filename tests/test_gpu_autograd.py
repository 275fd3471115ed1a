"""PyTorch autograd through the library (autograd.uvu_conv): first derivatives against the oracle's
VJP and second derivatives (create_graph=True, then a second grad) against the oracle's double
backward, on the tiny workload and a pipelined MACE-medium-irreps graph; and autograd.radial_conv
(edge lengths -> radial network -> last layer -> convolution): the edge-length, input, layer and
last-layer gradients against the oracle's composition."""
import numpy as np
import pytest
import torch

from clebsch_gordan_tensor_receiver_gb300 import autograd, uvu, workloads
from gpu_util import Problem, check, dev
from oracle import conv, hvp, paths

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


def test_radial_conv_gradients():
    """autograd.radial_conv: the gradients with respect to the edge lengths, x, Y, the radial
    layers and W_last against the oracle's composition of the same steps."""
    from oracle import graph, radial
    spec = workloads.custom_spec(710, 30, "64x0e+64x1o", "1x0e+1x1o+1x2e+1x3o", 3, "float32")
    rng = np.random.default_rng(71)
    recv, src = workloads.random_degree_graph(30, rng.integers(0, 12, size=30), rng)
    E, N = src.size, 30
    Y = workloads.sh_inputs(workloads.unit_vectors(E, rng), 3).astype(np.float32)
    x = rng.standard_normal((N, 64, 4)).astype(np.float32)
    plan = uvu.Plan(spec.irreps_x, spec.irreps_sh, spec.lmax_out, spec.dtype)
    lay = paths.layout(spec.irreps_x, spec.irreps_sh, spec.lmax_out)
    widths = [8, 32, 32]
    r, layers, Wl = workloads.radial_inputs(spec, E, plan.info.n_paths, 8, (32, 32), seed=7)
    G = uvu.Graph(N, dev(recv), dev(src))
    rt, xt, Yt = dev(r).requires_grad_(True), dev(x).requires_grad_(True), dev(Y).requires_grad_(True)
    Wt = dev(np.concatenate([a.reshape(-1) for a in layers])).requires_grad_(True)
    Wlt = dev(Wl).requires_grad_(True)
    out = autograd.radial_conv(rt, xt, Yt, Wt, Wlt, plan, G, 5.0, 5, widths)
    c = rng.standard_normal(out.shape).astype(np.float32)
    grads = torch.autograd.grad((out * dev(c)).sum(), (rt, xt, Yt, Wt, Wlt))
    off = graph.recv_offsets(recv, N)
    h = radial.hidden(r, 5.0, 5, layers)
    w = radial.weights(h, Wl)
    check(out.detach().cpu().numpy(), conv.fwd(lay, off, src, x, Y, w), False, "out")
    r_dY, r_dw = conv.bwd_edges(lay, off, src, x, Y, w, c)
    r_dx = conv.bwd_dx(lay, off, src, Y, w, c, N)
    r_dh, r_dWl = radial.weights_vjp(h, Wl, r_dw)
    r_dr, r_dW = radial.hidden_vjp(r, 5.0, 5, layers, r_dh)
    check(grads[0].cpu().numpy(), r_dr, False, "dr")
    check(grads[1].cpu().numpy(), r_dx, False, "dx")
    check(grads[2].cpu().numpy(), r_dY, False, "dY")
    check(grads[3].cpu().numpy(), np.concatenate([a.reshape(-1) for a in r_dW]), False, "dW")
    check(grads[4].cpu().numpy(), r_dWl, False, "dW_last")
    assert plan.device_status() == 0
