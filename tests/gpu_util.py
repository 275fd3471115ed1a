"""Helpers shared by the GPU parity tests: device copies, one call of each C-ABI entry point,
and the tolerance check (fp32: relative Frobenius <= 1e-5 and |d| <= 1e-4 (1 + |ref|); fp64:
relative Frobenius <= 1e-11 and |d| <= 1e-10 (1 + |ref|))."""
import numpy as np
import torch

from clebsch_gordan_tensor_receiver_gb300 import uvu, workloads
from oracle import conv, graph, paths


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def check(got, ref, f64, what=""):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (what, got.shape, ref.shape)
    d = got - ref
    nr = np.linalg.norm(ref)
    rel = np.linalg.norm(d) / nr if nr > 0 else np.linalg.norm(d)
    rtol, etol = (1e-11, 1e-10) if f64 else (1e-5, 1e-4)
    assert rel <= rtol, f"{what}: relative Frobenius error {rel:.3e} > {rtol}"
    bad = np.abs(d) > etol * (1 + np.abs(ref))
    assert not bad.any(), f"{what}: {bad.sum()} elements beyond {etol}(1+|ref|), max {np.abs(d).max():.3e}"
    return rel


class Problem:
    """A workload resident on the device plus its plan and graph."""

    def __init__(self, spec, recv, src, x, Y, n_nodes, seed_w=None):
        self.spec = spec
        self.f64 = spec.dtype == "float64"
        self.plan = uvu.Plan(spec.irreps_x, spec.irreps_sh, spec.lmax_out, spec.dtype)
        self.lay = paths.layout(spec.irreps_x, spec.irreps_sh, spec.lmax_out)
        self.N = n_nodes
        self.E = int(src.size)
        self.recv, self.src, self.x, self.Y = recv, src, x, Y
        i = self.plan.info
        assert Y.shape == (self.E, i.dim_sh) and x.shape == (n_nodes, i.mul, i.dim_x), \
            ("inputs do not match the plan's layout", Y.shape, x.shape)
        self.w = workloads.make_weights(spec, self.E, self.plan.info.n_paths)
        self.g = workloads.make_cotangent(spec, n_nodes, self.plan.info.dim_out)
        self.off_host = graph.recv_offsets(recv, n_nodes)
        self.d = {k: dev(v) for k, v in dict(x=x, Y=Y, w=self.w, g=self.g, recv=recv, src=src).items()}
        self.G = uvu.Graph(n_nodes, self.d["recv"], self.d["src"])

    @classmethod
    def from_spec(cls, key_or_spec):
        wl = workloads.make_workload(key_or_spec)
        return cls(wl.spec, wl.recv, wl.src, wl.x, wl.Y, wl.n_nodes)

    def empty(self, *shape):
        dt = torch.float64 if self.f64 else torch.float32
        return torch.empty(*shape, dtype=dt, device="cuda")

    def status_ok(self):
        """No kernel of this plan reported a bounded-wait timeout on the device."""
        return self.plan.device_status(reset=True) == 0

    def fwd(self):
        i = self.plan.info
        out = self.empty(self.N, i.mul, i.dim_out)
        out.fill_(float("nan"))  # every element must be written
        self.plan.fwd(self.N, self.d["x"], self.d["Y"], self.d["w"], self.G.recv_offsets,
                      self.d["src"], out)
        return out

    def bwd(self, mode):
        i = self.plan.info
        dx = self.empty(self.N, i.mul, i.dim_x).fill_(float("nan"))
        dY = self.empty(max(self.E, 1), i.dim_sh).fill_(float("nan"))
        dw = self.empty(max(self.E, 1), i.n_paths, i.mul).fill_(float("nan"))
        self.plan.bwd(self.N, self.d["x"], self.d["Y"], self.d["w"], self.G.recv_offsets,
                      self.d["src"], self.G.send_offsets, self.G.send_eids, self.G.send_recv,
                      self.d["g"], dx=dx, dY=dY, dw=dw, dx_mode=mode)
        return dx, dY[:self.E], dw[:self.E]

    # oracle on chosen owners
    def ref_out(self, receivers=None):
        return conv.fwd(self.lay, self.off_host, self.src, self.x, self.Y, self.w, receivers)

    def ref_edges(self, edges=None):
        return conv.bwd_edges(self.lay, self.off_host, self.src, self.x, self.Y, self.w, self.g, edges)

    def ref_dx(self, senders=None):
        return conv.bwd_dx(self.lay, self.off_host, self.src, self.Y, self.w, self.g, self.N, senders)
