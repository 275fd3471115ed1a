"""GPU parity of the fused-radial-weight path against the fp64 oracle, through the C ABI: the
radial network (uvu_radial_hidden) and the convolution whose per-edge weights are formed in
registers from it (uvu_conv_fwd_radial).  Small workloads are compared over every output; the
MACE-medium workload in the benchmark's launch configuration on sampled receivers."""
import numpy as np
import pytest
import torch

from clebsch_gordan_tensor_receiver_gb300 import uvu, workloads
from gpu_util import check, dev
from oracle import graph, paths, radial

pytestmark = pytest.mark.gpu

SH3 = "1x0e+1x1o+1x2e+1x3o"
RC = 5.0


def _flat(layers):
    return dev(np.concatenate([W.reshape(-1) for W in layers]))


def _run(spec, recv, src, x, Y, N, n_basis=8, hidden=(64, 64, 64), p_env=5, r=None, seed=0, receivers=None):
    plan = uvu.Plan(spec.irreps_x, spec.irreps_sh, spec.lmax_out, spec.dtype)
    lay = paths.layout(spec.irreps_x, spec.irreps_sh, spec.lmax_out)
    f64 = spec.dtype == "float64"
    rr, layers, Wl = workloads.radial_inputs(spec, src.size, plan.info.n_paths, n_basis, hidden, seed=seed)
    if r is not None:
        rr = r.astype(rr.dtype)
    dt = torch.float64 if f64 else torch.float32
    h = torch.full((max(src.size, 1), hidden[-1]), float("nan"), dtype=dt, device="cuda")[:src.size]
    plan.radial_hidden(dev(rr), RC, p_env, [n_basis, *hidden], _flat(layers), h)
    G = uvu.Graph(N, dev(recv), dev(src))
    out = torch.full((N, plan.info.mul, plan.info.dim_out), float("nan"), dtype=dt, device="cuda")
    plan.fwd_radial(N, dev(x), dev(Y), h, dev(Wl), G.recv_offsets, dev(src), out)
    off = graph.recv_offsets(recv, N)
    h_ref = radial.hidden(rr, RC, p_env, layers)
    ref = radial.conv_fwd(lay, off, src, x, Y, h_ref, Wl, receivers=receivers)
    assert plan.device_status(reset=True) == 0
    return h, out, h_ref, ref, f64, plan


CASES = [
    # irreps_x, irreps_sh, lmax_out, dtype, N, max degree, hidden
    ("128x0e+128x1o", SH3, 3, "float32", 60, 70, (64, 64, 64)),          # MACE-medium irreps, ragged degrees
    ("48x0e+48x1o+48x2e", SH3, 3, "float32", 37, 12, (32, 16)),         # two channel slices, the second half empty
    ("16x0e+16x1o", "1x0e+1x1o+1x2e", 2, "float32", 23, 9, (12, 8)),    # fewer channels than a warp
    ("64x0e+64x1o+64x2e", SH3, 3, "float64", 21, 8, (16, 20)),          # fp64, register groups
    ("128x0e+128x1o", SH3, 3, "float32", 19, 40, (64, 128)),            # last layer too large for shared memory
    ("32x1o+32x4e", "1x0e+1x1o+1x2e+1x3o+1x4e", 4, "float32", 13, 6, (8, 12)),  # l = 4 paths
]


@pytest.mark.parametrize("case", CASES, ids=[f"{c[0]}-{c[3]}-H{c[6][-1]}" for c in CASES])
def test_small_workloads_all_outputs(case):
    irx, irs, lo, dt, N, dmax, hidden = case
    k = CASES.index(case)
    spec = workloads.custom_spec(200 + k, N, irx, irs, lo, dt)
    rng = np.random.default_rng(200 + k)
    deg = rng.integers(0, dmax + 1, size=N)
    deg[[0, N // 2, N - 1]] = [0, dmax, 0]
    recv, src = workloads.random_degree_graph(N, deg, rng)
    lsh = int(irs.split("+")[-1].split("x")[1][:-1])
    Y = (workloads.sh_inputs(workloads.unit_vectors(src.size, rng), lsh) if lsh <= 3
         else rng.standard_normal((src.size, workloads.dim_of(irs)))).astype(dt)
    x = rng.standard_normal((N, spec.mul, workloads.dim_of(irx))).astype(dt)
    nb = 5 if dt == "float64" else 8
    h, out, h_ref, ref, f64, _ = _run(spec, recv, src, x, Y, N, n_basis=nb, hidden=hidden, seed=k)
    check(h.cpu().numpy(), h_ref, f64, "h")
    check(out.cpu().numpy(), ref, f64, "out")


def test_cutoff_and_empty_receivers():
    """Edges at or beyond the cutoff get h = 0 exactly and add nothing; empty receivers are zero."""
    spec = workloads.custom_spec(220, 17, "32x0e+32x1o", SH3, 3)
    rng = np.random.default_rng(220)
    deg = rng.integers(0, 6, size=17)
    deg[::4] = 0
    recv, src = workloads.random_degree_graph(17, deg, rng)
    Y = workloads.sh_inputs(workloads.unit_vectors(src.size, rng), 3).astype(np.float32)
    x = rng.standard_normal((17, 32, 4)).astype(np.float32)
    r = rng.uniform(1.0, 7.0, size=src.size)
    r[:3] = RC
    h, out, h_ref, ref, f64, _ = _run(spec, recv, src, x, Y, 17, r=r)
    beyond = torch.from_numpy(r.astype(np.float32) >= np.float32(RC)).cuda()
    assert beyond.sum() > 3 and torch.all(h[beyond] == 0)
    check(out.cpu().numpy(), ref, False, "out")
    empty = torch.from_numpy(deg == 0).cuda()
    assert torch.all(out[empty] == 0)


def test_no_edges():
    spec = workloads.custom_spec(221, 5, "32x0e+32x1o", SH3, 3)
    plan = uvu.Plan(spec.irreps_x, spec.irreps_sh, spec.lmax_out, spec.dtype)
    Wl = dev(np.ones((8, plan.info.n_paths, 32), np.float32))
    G = uvu.Graph(5, dev(np.zeros(0, np.int32)), dev(np.zeros(0, np.int32)))
    out = torch.full((5, 32, plan.info.dim_out), float("nan"), device="cuda")
    plan.fwd_radial(5, None, None, None, Wl, G.recv_offsets, dev(np.zeros(0, np.int32)), out)
    assert torch.all(out == 0)
    plan.radial_hidden(torch.zeros(0, device="cuda"), RC, 5, [8, 8], dev(np.ones(64, np.float32)),
                       torch.zeros(0, 8, device="cuda"))


def test_one_hidden_width_per_plan():
    spec = workloads.custom_spec(222, 4, "32x0e+32x1o", SH3, 3)
    plan = uvu.Plan(spec.irreps_x, spec.irreps_sh, spec.lmax_out, spec.dtype)
    plan.radial_source(16)
    with pytest.raises(uvu.UVUError, match="UNSUPPORTED"):
        plan.radial_source(32)


@pytest.mark.parametrize("key", [1, 2, 3, 4])
def test_full_size_sampled_receivers(key):
    """The full-size workloads (MACE-medium in the launch configuration the benchmark times;
    MACE-large; the wide proxy with U = 256, 24 paths and eight channel slices; the irregular fp64
    graph with the last layer read through the cache), checked on sampled receivers (and every
    receiver against non-NaN)."""
    wl = workloads.make_workload(key)
    rng = np.random.default_rng(1234 + key)
    rs = np.unique(np.concatenate([rng.choice(wl.n_nodes, 40, replace=False), [0, wl.n_nodes - 1]]))
    h, out, h_ref, ref, f64, _ = _run(wl.spec, wl.recv, wl.src, wl.x, wl.Y, wl.n_nodes, receivers=rs)
    es = rng.choice(wl.n_edges, 2000, replace=False)
    check(h[torch.from_numpy(es).cuda()].cpu().numpy(), h_ref[es], f64, "h")
    check(out[torch.from_numpy(rs).cuda()].cpu().numpy(), ref, f64, "out")
    assert not torch.isnan(out).any()


def test_repeat_bitwise():
    wl = workloads.make_workload(0)
    h, out, *_rest, plan = _run(wl.spec, wl.recv, wl.src, wl.x, wl.Y, wl.n_nodes, hidden=(16, 16))
    plan2_out = torch.empty_like(out)
    r, layers, Wl = workloads.radial_inputs(wl.spec, wl.n_edges, plan.info.n_paths, 8, (16, 16))
    G = uvu.Graph(wl.n_nodes, dev(wl.recv), dev(wl.src))
    h2 = torch.empty_like(h)
    plan.radial_hidden(dev(r), RC, 5, [8, 16, 16], _flat(layers), h2)
    plan.fwd_radial(wl.n_nodes, dev(wl.x), dev(wl.Y), h2, dev(Wl), G.recv_offsets, dev(wl.src), plan2_out)
    assert torch.equal(h, h2) and torch.equal(out, plan2_out)
