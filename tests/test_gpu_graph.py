"""The C-ABI calls of one convolution step (forward, edge backward, staged dx reduction) recorded
into a CUDA graph by stream capture and replayed: the replay writes the same bits as the eager
calls, and replays with new inputs copied into the captured buffers follow the new inputs."""
import pytest
import torch

from clebsch_gordan_tensor_receiver_gb300 import uvu
from gpu_util import Problem, check
from oracle import conv

pytestmark = pytest.mark.gpu


def test_step_captured_in_a_cuda_graph_replays_bitwise():
    P = Problem.from_spec(1)
    i = P.plan.info
    N, E = P.N, P.E
    out, dx = P.empty(N, i.mul, i.dim_out), P.empty(N, i.mul, i.dim_x)
    dY, dw = P.empty(E, i.dim_sh), P.empty(E, i.n_paths, i.mul)
    ws = torch.empty(P.plan.workspace_bytes(N, E, uvu.UVU_DX_STAGED), dtype=torch.uint8, device="cuda")
    d, G = P.d, P.G

    def step(st):
        P.plan.fwd(N, d["x"], d["Y"], d["w"], G.recv_offsets, d["src"], out, st)
        P.plan.bwd_edge(N, d["x"], d["Y"], d["w"], G.recv_offsets, d["src"], d["g"], dY=dY, dw=dw,
                        dx_edge=ws, stream=st)
        P.plan.bwd_dx_reduce(N, E, G.send_offsets, G.send_eids, ws, dx, st)

    step(torch.cuda.current_stream())  # eager: also loads the modules
    torch.cuda.synchronize()
    ref = [t.clone() for t in (out, dx, dY, dw)]
    g = torch.cuda.CUDAGraph()
    cap = torch.cuda.Stream()
    cap.wait_stream(torch.cuda.current_stream())
    with torch.cuda.graph(g, stream=cap):
        step(cap)
    for t in (out, dx, dY, dw):
        t.fill_(float("nan"))
    g.replay()
    torch.cuda.synchronize()
    for a, b in zip((out, dx, dY, dw), ref):
        assert torch.equal(a, b)
    # new inputs in the captured buffers: the replay follows them (checked against the oracle on samples)
    d["w"].mul_(-0.5)
    g.replay()
    torch.cuda.synchronize()
    rs = torch.arange(0, N, 997)
    ref_new = conv.fwd(P.lay, P.off_host, P.src, P.x, P.Y, d["w"].cpu().numpy(), rs.numpy())
    check(out[rs.cuda()].cpu().numpy(), ref_new, P.f64, "out after new w")
    assert P.status_ok()
