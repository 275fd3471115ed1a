"""Every entry point that takes a caller workspace or writes caller outputs stays inside them: each
buffer is handed over as the exact size the library asks for, cut from a larger allocation whose
tail holds a known pattern, and the tail must be unchanged after the call.  Covers the radial
last layer and its gradients at hidden widths whose two products have different shapes (the
input-gradient product dh = dw W_last^T has K = P U and N = hidden), the radial network's reverse
pass, the channel mixing, the staged convolution VJP and the double backward."""
import numpy as np
import pytest
import torch

from clebsch_gordan_tensor_receiver_gb300 import uvu, workloads
from gpu_util import dev

pytestmark = pytest.mark.gpu

TAIL = 4096
SH3 = "1x0e+1x1o+1x2e+1x3o"


class Guarded:
    """Buffers cut from allocations with a patterned tail of TAIL bytes."""

    def __init__(self):
        self.bufs = []

    def ws(self, nbytes):
        n = max(int(nbytes), 16)
        buf = torch.full((n + TAIL,), 0xA5, dtype=torch.uint8, device="cuda")
        self.bufs.append(("workspace", buf, n))
        return buf[:n]

    def out(self, *shape, dtype=torch.float32):
        n = int(np.prod(shape))
        es = torch.empty((), dtype=dtype).element_size()
        buf = torch.full((n * es + TAIL,), 0x5A, dtype=torch.uint8, device="cuda")
        self.bufs.append(("output", buf, n * es))
        return buf[:n * es].view(dtype).view(*shape)

    def check(self):
        torch.cuda.synchronize()
        for kind, buf, n in self.bufs:
            tail = buf[n:]
            want = 0xA5 if kind == "workspace" else 0x5A
            bad = int((tail != want).sum())
            assert bad == 0, f"{kind} of {n} bytes: {bad} bytes written past its end"


def _radial_case(hidden, U, seed):
    spec = workloads.custom_spec(780 + hidden, 30, f"{U}x0e+{U}x1o", SH3, 3, "float32")
    plan = uvu.Plan(spec.irreps_x, spec.irreps_sh, spec.lmax_out, spec.dtype)
    return spec, plan


@pytest.mark.parametrize("hidden,U,E", [(32, 64, 149), (64, 128, 700), (16, 32, 2000), (128, 32, 300)])
def test_radial_last_layer_and_gradients(hidden, U, E):
    spec, plan = _radial_case(hidden, U, 1)
    P = plan.info.n_paths
    rng = np.random.default_rng(hidden + U)
    h = dev(rng.standard_normal((E, hidden)).astype(np.float32))
    wl = dev((rng.standard_normal((hidden, P, U)) / np.sqrt(hidden)).astype(np.float32))
    g = Guarded()
    w = g.out(E, P, U)
    plan.radial_weights(h, wl, w, workspace=g.ws(plan.radial_weights_workspace(hidden)))
    dw = dev(rng.standard_normal((E, P, U)).astype(np.float32))
    dh = g.out(E, hidden)
    dwl = g.out(hidden, P, U)
    plan.radial_weights_bwd(h, wl, dw, dh=dh, dw_last=dwl, workspace=g.ws(plan.radial_weights_bwd_workspace(E, hidden)))
    g.check()
    # and the values: the products against fp64 (each sum is short enough for the fp32 tolerance)
    hd, wld, dwd = (t.double().cpu().numpy() for t in (h, wl, dw))
    ref_w = np.einsum("ek,kpu->epu", hd, wld)
    assert np.linalg.norm(w.cpu().numpy() - ref_w) <= 1e-5 * np.linalg.norm(ref_w)
    ref_dh = np.einsum("epu,kpu->ek", dwd, wld)
    assert np.linalg.norm(dh.cpu().numpy() - ref_dh) <= 1e-5 * np.linalg.norm(ref_dh)
    ref_dwl = np.einsum("ek,epu->kpu", hd, dwd)
    assert np.linalg.norm(dwl.cpu().numpy() - ref_dwl) <= 1e-5 * np.linalg.norm(ref_dwl)


@pytest.mark.parametrize("widths", [[8, 32, 32], [8, 64, 64, 64], [4, 16]])
def test_radial_network_reverse_pass(widths):
    spec, plan = _radial_case(widths[-1], 16, 2)
    E = 777
    r, layers, _ = workloads.radial_inputs(spec, E, plan.info.n_paths, widths[0], tuple(widths[1:]), seed=9)
    wflat = dev(np.concatenate([a.reshape(-1) for a in layers]))
    rng = np.random.default_rng(4)
    g = Guarded()
    h = g.out(E, widths[-1])
    plan.radial_hidden(dev(r), 5.0, 5, widths, wflat, h)
    dh = dev(rng.standard_normal((E, widths[-1])).astype(np.float32))
    dr = g.out(E)
    dW = g.out(wflat.numel())
    plan.radial_hidden_bwd(dev(r), 5.0, 5, widths, wflat, dh, dr, dW,
                           workspace=g.ws(plan.radial_hidden_bwd_workspace(E, widths)))
    g.check()


@pytest.mark.parametrize("U,W", [(64, 128), (32, 16)])
def test_mixing(U, W):
    spec = workloads.custom_spec(790, 40, f"{U}x0e+{U}x1o", SH3, 3, "float32")
    plan = uvu.Plan(spec.irreps_x, spec.irreps_sh, spec.lmax_out, spec.dtype)
    N, P, Do = 333, plan.info.n_paths, plan.info.dim_out
    rng = np.random.default_rng(U + W)
    inp = dev(rng.standard_normal((N, U, Do)).astype(np.float32))
    M = dev((rng.standard_normal((P, U, W)) / np.sqrt(U)).astype(np.float32))
    fb, bb = plan.mix_workspace_bytes(N, W)
    g = Guarded()
    out = g.out(N, W, Do)
    plan.mix_fwd(N, W, inp, M, out, workspace=g.ws(fb))
    d_out = dev(rng.standard_normal((N, W, Do)).astype(np.float32))
    d_in = g.out(N, U, Do)
    dM = g.out(P, U, W)
    plan.mix_bwd(N, W, inp, M, d_out, d_in=d_in, dM=dM, workspace=g.ws(bb))
    g.check()


def test_conv_staged_vjp_and_hvp():
    spec = workloads.custom_spec(795, 40, "64x0e+64x1o", SH3, 3, "float32")
    plan = uvu.Plan(spec.irreps_x, spec.irreps_sh, spec.lmax_out, spec.dtype)
    rng = np.random.default_rng(795)
    N = 40
    recv, src = workloads.random_degree_graph(N, rng.integers(0, 14, size=N), rng)
    E = src.size
    i = plan.info
    Y = dev(workloads.sh_inputs(workloads.unit_vectors(E, rng), 3).astype(np.float32))
    x = dev(rng.standard_normal((N, i.mul, i.dim_x)).astype(np.float32))
    w = dev(rng.standard_normal((E, i.n_paths, i.mul)).astype(np.float32))
    d_out = dev(rng.standard_normal((N, i.mul, i.dim_out)).astype(np.float32))
    G = uvu.Graph(N, dev(recv), dev(src))
    g = Guarded()
    dx, dY, dw = g.out(N, i.mul, i.dim_x), g.out(E, i.dim_sh), g.out(E, i.n_paths, i.mul)
    plan.bwd(N, x, Y, w, G.recv_offsets, G.src, G.send_offsets, G.send_eids, G.send_recv, d_out, dx=dx, dY=dY,
             dw=dw, dx_mode=uvu.UVU_DX_STAGED, workspace=g.ws(plan.workspace_bytes(N, E, uvu.UVU_DX_STAGED)))
    ax, aY, aw = (dev(rng.standard_normal(t.shape).astype(np.float32)) for t in (x, Y, w))
    gd, gx, gY, gw = g.out(N, i.mul, i.dim_out), g.out(N, i.mul, i.dim_x), g.out(E, i.dim_sh), g.out(E, i.n_paths, i.mul)
    import ctypes
    b = ctypes.c_size_t()
    uvu.uvu_conv_hvp_workspace(plan.handle, N, E, ctypes.byref(b))
    plan.hvp(N, x, Y, w, G.recv_offsets, G.src, G.send_offsets, G.send_eids, d_out, ax=ax, aY=aY, aw=aw,
             grad_d_out=gd, grad_x=gx, grad_Y=gY, grad_w=gw, workspace=g.ws(b.value))
    g.check()
    assert plan.device_status() == 0
