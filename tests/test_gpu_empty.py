"""Empty inputs of the newer entry points: a graph without edges for the sender forward and the
double backward (zeros written where the definition gives zero), and zero receivers for the
channel mixing (nothing written; a requested dM is zero)."""
import numpy as np
import pytest
import torch

from clebsch_gordan_tensor_receiver_gb300 import uvu, workloads
from gpu_util import Problem, dev

pytestmark = pytest.mark.gpu

SH3 = "1x0e+1x1o+1x2e+1x3o"


def _edgeless():
    spec = workloads.custom_spec(950, 9, "32x0e+32x1o", SH3, 3)
    z = np.zeros(0, np.int32)
    return Problem(spec, z, z, np.ones((9, 32, 4), np.float32), np.zeros((0, 16), np.float32), 9)


def test_sender_forward_without_edges():
    P = _edgeless()
    i = P.plan.info
    out = torch.full((9, i.mul, i.dim_out), float("nan"), device="cuda")
    P.plan.fwd_sender(9, 0, P.d["x"], P.d["Y"], P.d["w"], P.G.send_offsets, P.G.send_eids, P.G.send_recv, out)
    torch.cuda.synchronize()
    assert torch.all(out == 0)


def test_double_backward_without_edges():
    P = _edgeless()
    i = P.plan.info
    gg = torch.full((9, i.mul, i.dim_out), float("nan"), device="cuda")
    gx = torch.full((9, i.mul, i.dim_x), float("nan"), device="cuda")
    ax = torch.ones(9, i.mul, i.dim_x, device="cuda")
    P.plan.hvp(9, P.d["x"], P.d["Y"], P.d["w"], P.G.recv_offsets, P.d["src"], P.G.send_offsets, P.G.send_eids,
               P.d["g"], ax=ax, grad_d_out=gg, grad_x=gx)
    torch.cuda.synchronize()
    assert torch.all(gg == 0) and torch.all(gx == 0)
    assert P.status_ok()


def test_mixing_without_receivers():
    plan = uvu.Plan("32x0e+32x1o", SH3, 3)
    i = plan.info
    e = torch.empty(0, device="cuda")
    M = dev(np.ones((i.n_paths, i.mul, 8), np.float32))
    dM = torch.full((i.n_paths, i.mul, 8), float("nan"), device="cuda")
    plan.mix_fwd(0, 8, e, M, e)
    plan.mix_bwd(0, 8, e, M, e, dM=dM)
    torch.cuda.synchronize()
    assert torch.all(dM == 0)
