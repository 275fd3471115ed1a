"""GPU parity of the radial network's last layer and reverse pass against the fp64 oracle, through
the C ABI: the materialised last layer (uvu_radial_weights, tensor cores in fp32 plans), its
gradients dh and dW_last (uvu_radial_weights_bwd) and the edge-length and layer gradients of the
network (uvu_radial_hidden_bwd); the whole chain radial network -> weights -> convolution VJP ->
gradients on a small graph; MACE-medium size (280,000 edges, hidden 64, 13 paths x 128
channels) on sampled rows and columns, with the sums over all edges compared in full."""
import numpy as np
import pytest
import torch

from clebsch_gordan_tensor_receiver_gb300 import uvu, workloads
from gpu_util import check, dev
from oracle import conv, graph, paths, radial

pytestmark = pytest.mark.gpu

SH3 = "1x0e+1x1o+1x2e+1x3o"
RC = 5.0


def _flat(layers):
    return dev(np.concatenate([W.reshape(-1) for W in layers]))


def _unflat(v, widths):
    out, o = [], 0
    for i in range(len(widths) - 1):
        n = widths[i] * widths[i + 1]
        out.append(v[o:o + n].reshape(widths[i], widths[i + 1]))
        o += n
    return out


CASES = [
    # irreps_x, dtype, E, n_basis, hidden
    ("128x0e+128x1o", "float32", 300, 8, (64, 64, 64)),
    ("48x0e+48x1o+48x2e", "float32", 257, 6, (16, 12)),     # n_basis not a multiple of 4, ragged tiles
    ("16x0e+16x1o", "float32", 5, 8, (8,)),                 # fewer edges than a tile, one layer
    ("64x0e+64x1o+64x2e", "float64", 129, 8, (16, 20)),     # fp64: CUDA-core products
    ("32x0e+32x1o", "float32", 77, 8, (128, 128, 128)),     # widest layers: 16-edge tiles, weights read globally
]


@pytest.mark.parametrize("case", CASES, ids=[f"{c[0]}-{c[1]}-E{c[2]}-H{c[4][-1]}" for c in CASES])
def test_last_layer_and_reverse_pass_all_outputs(case):
    irx, dt, E, nb, hidden = case
    k = CASES.index(case)
    spec = workloads.custom_spec(700 + k, 10, irx, SH3, 3, dt)
    plan = uvu.Plan(irx, SH3, 3, dt)
    P, U = plan.info.n_paths, plan.info.mul
    f64 = dt == "float64"
    tdt = torch.float64 if f64 else torch.float32
    r, layers, Wl = workloads.radial_inputs(spec, E, P, nb, hidden, seed=k)
    r = r.copy()
    r[-1] = 5.5  # one edge beyond the cutoff
    widths = [nb, *hidden]
    H = hidden[-1]
    rng = np.random.default_rng(70 + k)
    h = radial.hidden(r, RC, 5, layers).astype(dt)
    dw = rng.standard_normal((E, P, U)).astype(dt)
    dh_in = rng.standard_normal((E, H)).astype(dt)
    # last layer and its gradients
    w = torch.full((E, P, U), float("nan"), dtype=tdt, device="cuda")
    plan.radial_weights(dev(h), dev(Wl), w)
    dh = torch.full((E, H), float("nan"), dtype=tdt, device="cuda")
    dWl = torch.full(Wl.shape, float("nan"), dtype=tdt, device="cuda")
    plan.radial_weights_bwd(dev(h), dev(Wl), dev(dw), dh=dh, dw_last=dWl)
    # reverse pass of the network
    dr = torch.full((E,), float("nan"), dtype=tdt, device="cuda")
    dW = torch.full((sum(widths[i] * widths[i + 1] for i in range(len(hidden))),), float("nan"), dtype=tdt, device="cuda")
    plan.radial_hidden_bwd(dev(r), RC, 5, widths, _flat(layers), dev(dh_in), dr, dW)
    torch.cuda.synchronize()
    assert plan.device_status() == 0
    check(w.cpu().numpy(), radial.weights(h, Wl), f64, "w")
    r_dh, r_dWl = radial.weights_vjp(h, Wl, dw)
    check(dh.cpu().numpy(), r_dh, f64, "dh")
    check(dWl.cpu().numpy(), r_dWl, f64, "dW_last")
    r_dr, r_dW = radial.hidden_vjp(r, RC, 5, layers, dh_in)
    check(dr.cpu().numpy(), r_dr, f64, "dr")
    assert float(dr[-1]) == 0.0
    for i, (a, b) in enumerate(zip(_unflat(dW.cpu().numpy(), widths), r_dW)):
        check(a, b, f64, f"dW_{i + 1}")


def test_empty_edge_set():
    plan = uvu.Plan("32x0e+32x1o", SH3, 3)
    P, U = plan.info.n_paths, plan.info.mul
    e = torch.empty(0, 16, device="cuda")
    dWl = torch.full((16, P, U), float("nan"), device="cuda")
    plan.radial_weights_bwd(e, torch.zeros(16, P, U, device="cuda"), torch.empty(0, P, U, device="cuda"), dw_last=dWl)
    dW = torch.full((8 * 16,), float("nan"), device="cuda")
    plan.radial_hidden_bwd(torch.empty(0, device="cuda"), RC, 5, [8, 16], torch.zeros(8 * 16, device="cuda"), e,
                           torch.empty(0, device="cuda"), dW)
    torch.cuda.synchronize()
    assert torch.equal(dWl, torch.zeros_like(dWl)) and torch.equal(dW, torch.zeros_like(dW))


def test_chain_through_the_convolution_vjp():
    """Radial network -> materialised weights -> convolution -> VJP -> last-layer and network
    gradients, against the oracle's composition (w = weights(h, W_last), then conv.bwd_edges and
    bwd_dx with those weights, then weights_vjp and hidden_vjp)."""
    spec = workloads.custom_spec(750, 40, "128x0e+128x1o", SH3, 3, "float32")
    rng = np.random.default_rng(75)
    deg = rng.integers(0, 30, size=40)
    recv, src = workloads.random_degree_graph(40, deg, rng)
    E, N = src.size, 40
    Y = workloads.sh_inputs(workloads.unit_vectors(E, rng), 3).astype(np.float32)
    x = rng.standard_normal((N, 128, 4)).astype(np.float32)
    plan = uvu.Plan(spec.irreps_x, spec.irreps_sh, spec.lmax_out, spec.dtype)
    lay = paths.layout(spec.irreps_x, spec.irreps_sh, spec.lmax_out)
    info = plan.info
    r, layers, Wl = workloads.radial_inputs(spec, E, info.n_paths, 8, (64, 64), seed=3)
    widths = [8, 64, 64]
    g = rng.standard_normal((N, 128, info.dim_out)).astype(np.float32)
    G = uvu.Graph(N, dev(recv), dev(src))
    h = torch.empty(E, 64, device="cuda")
    plan.radial_hidden(dev(r), RC, 5, widths, _flat(layers), h)
    w = torch.empty(E, info.n_paths, 128, device="cuda")
    plan.radial_weights(h, dev(Wl), w)
    dx = torch.empty(N, 128, info.dim_x, device="cuda")
    dY = torch.empty(E, info.dim_sh, device="cuda")
    dw = torch.empty_like(w)
    plan.bwd(N, dev(x), dev(Y), w, G.recv_offsets, dev(src), G.send_offsets, G.send_eids, G.send_recv, dev(g),
             dx=dx, dY=dY, dw=dw, dx_mode=uvu.UVU_DX_STAGED)
    dh = torch.empty(E, 64, device="cuda")
    dWl = torch.empty(Wl.shape, device="cuda")
    plan.radial_weights_bwd(h, dev(Wl), dw, dh=dh, dw_last=dWl)
    dr = torch.empty(E, device="cuda")
    dW = torch.empty(8 * 64 + 64 * 64, device="cuda")
    plan.radial_hidden_bwd(dev(r), RC, 5, widths, _flat(layers), dh, dr, dW)
    torch.cuda.synchronize()
    assert plan.device_status() == 0
    off = graph.recv_offsets(recv, N)
    h_ref = radial.hidden(r, RC, 5, layers)
    w_ref = radial.weights(h_ref, Wl)
    r_dY, r_dw = conv.bwd_edges(lay, off, src, x, Y, w_ref, g)
    r_dx = conv.bwd_dx(lay, off, src, Y, w_ref, g, N)
    r_dh, r_dWl = radial.weights_vjp(h_ref, Wl, r_dw)
    r_dr, r_dW = radial.hidden_vjp(r, RC, 5, layers, r_dh)
    check(dx.cpu().numpy(), r_dx, False, "dx")
    check(dY.cpu().numpy(), r_dY, False, "dY")
    check(dWl.cpu().numpy(), r_dWl, False, "dW_last")
    check(dr.cpu().numpy(), r_dr, False, "dr")
    for i, (a, b) in enumerate(zip(_unflat(dW.cpu().numpy(), widths), r_dW)):
        check(a, b, False, f"dW_{i + 1}")


def test_mace_medium_size_sampled():
    """280,000 edges, hidden 8-64-64-64, 13 paths x 128 channels: w and dh on sampled edges,
    dW_last on sampled columns (each a sum over all edges), dr on sampled edges and the layer
    gradients in full."""
    spec = workloads.SPECS[1]
    plan = uvu.Plan(spec.irreps_x, spec.irreps_sh, spec.lmax_out, spec.dtype)
    P, U = plan.info.n_paths, plan.info.mul
    E = 280_000
    widths = [8, 64, 64, 64]
    r, layers, Wl = workloads.radial_inputs(spec, E, P, 8, (64, 64, 64), seed=5)
    rng = np.random.default_rng(55)
    dw = (rng.standard_normal((E, P, U), dtype=np.float32) * np.float32(0.1))
    h = torch.empty(E, 64, device="cuda")
    plan.radial_hidden(dev(r), RC, 5, widths, _flat(layers), h)
    w = torch.empty(E, P, U, device="cuda")
    plan.radial_weights(h, dev(Wl), w)
    dh = torch.empty(E, 64, device="cuda")
    dWl = torch.empty(Wl.shape, device="cuda")
    plan.radial_weights_bwd(h, dev(Wl), dev(dw), dh=dh, dw_last=dWl)
    dr = torch.empty(E, device="cuda")
    dW = torch.empty(8 * 64 + 2 * 64 * 64, device="cuda")
    plan.radial_hidden_bwd(dev(r), RC, 5, widths, _flat(layers), dh, dr, dW)
    torch.cuda.synchronize()
    assert plan.device_status() == 0
    h_ref = radial.hidden(r, RC, 5, layers)
    rows = np.unique(np.concatenate([rng.choice(E, 200, replace=False), [0, E - 1]]))
    rt = torch.from_numpy(rows).cuda()
    check(w[rt].cpu().numpy(), radial.weights(h_ref[rows], Wl), False, "w (sampled edges)")
    r_dh = np.einsum("epu,kpu->ek", dw[rows].astype(np.float64), Wl.astype(np.float64))
    check(dh[rt].cpu().numpy(), r_dh, False, "dh (sampled edges)")
    cols = rng.choice(P * U, 48, replace=False)
    dwc = dw.reshape(E, P * U)[:, cols].astype(np.float64)
    r_dWl = h_ref.T @ dwc
    check(dWl.reshape(64, P * U)[:, torch.from_numpy(cols).cuda()].cpu().numpy(), r_dWl, False, "dW_last (sampled columns)")
    # the network's gradients for the cotangent the GPU produced (so the comparison isolates this step)
    dh_gpu = dh.double().cpu().numpy()
    r_dr, r_dW = radial.hidden_vjp(r, RC, 5, layers, dh_gpu)
    check(dr[rt].cpu().numpy(), r_dr[rows], False, "dr (sampled edges)")
    for i, (a, b) in enumerate(zip(_unflat(dW.cpu().numpy(), widths), r_dW)):
        check(a, b, False, f"dW_{i + 1}")
