"""GPU parity of the sender-stationary forward (uvu_conv_fwd_sender) and of the mode dispatch
(uvu_conv_fwd_mode) against the fp64 oracle: small graphs with empty senders and receivers,
several register groups, fp64, a plan for which the data-movement model picks the sender
forward, and sampled receivers of the full MACE-medium workload."""
import numpy as np
import pytest
import torch

from clebsch_gordan_tensor_receiver_gb300 import uvu, workloads
from gpu_util import Problem, check
from oracle import conv

pytestmark = pytest.mark.gpu

SH3 = "1x0e+1x1o+1x2e+1x3o"


def _sender(P):
    i = P.plan.info
    out = P.empty(P.N, i.mul, i.dim_out).fill_(float("nan"))
    P.plan.fwd_sender(P.N, P.E, P.d["x"], P.d["Y"], P.d["w"], P.G.send_offsets, P.G.send_eids,
                      P.G.send_recv, out)
    torch.cuda.synchronize()
    return out


CASES = [
    ("16x0e+16x1o", "1x0e+1x1o+1x2e", 2, "float32", 23, 7),
    ("48x0e+48x1o+48x2e", SH3, 3, "float32", 31, 9),
    ("64x0e+64x1o+64x2e", SH3, 3, "float64", 17, 6),   # several register groups
    ("32x0e+32x1e+32x2e+32x3e+32x4e", "1x0e", 0, "float32", 40, 12),  # the model picks the sender forward
]


@pytest.mark.parametrize("case", CASES, ids=[c[0] + "-" + c[3] for c in CASES])
def test_sender_forward_small_graphs(case):
    irx, irs, lo, dt, N, dmax = case
    spec = workloads.custom_spec(400 + CASES.index(case), N, irx, irs, lo, dt)
    rng = np.random.default_rng(60 + CASES.index(case))
    deg = rng.integers(0, dmax + 1, size=N)
    deg[0] = 0
    recv, src = workloads.random_degree_graph(N, deg, rng)
    lsh = int(irs.split("+")[-1].split("x")[1][:-1])
    Y = workloads.sh_inputs(workloads.unit_vectors(src.size, rng), lsh).astype(dt)
    x = rng.standard_normal((N, int(irx.split("x")[0]), workloads.dim_of(irx))).astype(dt)
    P = Problem(spec, recv, src, x, Y, N)
    ref = conv.fwd(P.lay, P.off_host, P.src, P.x, P.Y, P.w)
    check(_sender(P).cpu().numpy(), ref, P.f64, "sender out")
    mode, _, _ = P.plan.fwd_model(P.N, P.E)
    out = P.empty(P.N, P.plan.info.mul, P.plan.info.dim_out).fill_(float("nan"))
    P.plan.fwd_mode(uvu.UVU_FWD_AUTO, P.N, P.E, P.d["x"], P.d["Y"], P.d["w"], P.G, out)
    torch.cuda.synchronize()
    check(out.cpu().numpy(), ref, P.f64, f"auto ({mode}) out")
    assert P.status_ok()


def test_sender_forward_medium_sampled():
    P = Problem.from_spec(1)
    assert P.plan.fwd_model(P.N, P.E)[0] == uvu.UVU_FWD_RECEIVER
    out = _sender(P)
    rng = np.random.default_rng(8)
    rs = np.unique(np.concatenate([rng.choice(P.N, 32, replace=False), [0, P.N - 1]]))
    ref = conv.fwd(P.lay, P.off_host, P.src, P.x, P.Y, P.w, rs)
    check(out[torch.from_numpy(rs).cuda()].cpu().numpy(), ref, False, "sender out")
    assert not torch.isnan(out).any()
