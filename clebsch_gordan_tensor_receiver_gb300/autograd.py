"""PyTorch autograd for the UVU convolution, through the library's C ABI only.

`uvu_conv(x, Y, w, plan, graph)` returns out [N][U][D_out].  Its backward is the VJP
(uvu_conv_bwd: dx, dY, dw), and the VJP's own backward is the double backward (uvu_conv_hvp), so
`torch.autograd.grad(..., create_graph=True)` followed by a second `grad` (forces in training, as
in "Receiver-streaming convolutions for channel-wise UVU tensor products", results table: HVP
column) runs on the library's kernels.  Third derivatives are not provided.

Every tensor is a contiguous CUDA tensor of the plan's dtype in the layouts of include/uvu.h;
`graph` is a `uvu.Graph` (receiver CSR and transposed CSR) of the same edges.  This module only
marshals arguments: every step runs in the library.
"""

from __future__ import annotations

import torch
from torch.autograd.function import once_differentiable

from . import uvu


def _c(t):
    return t.contiguous()


class _ConvVJP(torch.autograd.Function):
    """(x, Y, w, g) -> (dx, dY, dw); backward = the double backward."""

    @staticmethod
    def forward(ctx, x, Y, w, g, plan, graph, dx_mode):
        n, e, i = graph.n_nodes, graph.n_edges, plan.info
        dx = torch.empty_like(x)
        dY = torch.empty(max(e, 1), i.dim_sh, dtype=x.dtype, device=x.device)[:e]
        dw = torch.empty(max(e, 1), i.n_paths, i.mul, dtype=x.dtype, device=x.device)[:e]
        plan.bwd(n, x, Y, w, graph.recv_offsets, graph.src, graph.send_offsets, graph.send_eids,
                 graph.send_recv, g, dx=dx, dY=dY, dw=dw, dx_mode=dx_mode)
        ctx.save_for_backward(x, Y, w, g)
        ctx.plan, ctx.graph = plan, graph
        return dx, dY, dw

    @staticmethod
    @once_differentiable
    def backward(ctx, ax, aY, aw):
        x, Y, w, g = ctx.saved_tensors
        plan, graph = ctx.plan, ctx.graph
        n, e = graph.n_nodes, graph.n_edges
        need = ctx.needs_input_grad
        gx = torch.empty_like(x) if need[0] else None
        gY = torch.empty_like(Y) if need[1] and e > 0 else (torch.zeros_like(Y) if need[1] else None)
        gw = torch.empty_like(w) if need[2] and e > 0 else (torch.zeros_like(w) if need[2] else None)
        gg = torch.empty_like(g) if need[3] else None
        plan.hvp(n, x, Y, w, graph.recv_offsets, graph.src, graph.send_offsets, graph.send_eids, g,
                 ax=None if ax is None else _c(ax), aY=None if aY is None else _c(aY),
                 aw=None if aw is None else _c(aw), grad_d_out=gg, grad_x=gx,
                 grad_Y=gY if e > 0 else None, grad_w=gw if e > 0 else None)
        return gx, gY, gw, gg, None, None, None


class _Conv(torch.autograd.Function):
    """(x, Y, w) -> out; backward = the VJP (itself differentiable once more)."""

    @staticmethod
    def forward(ctx, x, Y, w, plan, graph, dx_mode):
        i = plan.info
        out = torch.empty(graph.n_nodes, i.mul, i.dim_out, dtype=x.dtype, device=x.device)
        plan.fwd(graph.n_nodes, x, Y, w, graph.recv_offsets, graph.src, out)
        ctx.save_for_backward(x, Y, w)
        ctx.plan, ctx.graph, ctx.dx_mode = plan, graph, dx_mode
        return out

    @staticmethod
    def backward(ctx, g):
        x, Y, w = ctx.saved_tensors
        dx, dY, dw = _ConvVJP.apply(x, Y, w, _c(g), ctx.plan, ctx.graph, ctx.dx_mode)
        return dx, dY, dw, None, None, None


def uvu_conv(x, Y, w, plan: "uvu.Plan", graph: "uvu.Graph", dx_mode: int = uvu.UVU_DX_STAGED):
    """out = the UVU convolution of x [N][U][D_x], Y [E][D_Y], w [E][P][U] over `graph`, with
    autograd support up to second order (VJP and double backward run in the library)."""
    return _Conv.apply(_c(x), _c(Y), _c(w), plan, graph, dx_mode)


class _RadialHidden(torch.autograd.Function):
    """r [E] -> h [E][widths[-1]] (uvu_radial_hidden); backward = uvu_radial_hidden_bwd (dr and
    the layers' gradients)."""

    @staticmethod
    def forward(ctx, r, weights, plan, r_cut, p_env, widths):
        h = torch.empty(r.numel(), widths[-1], dtype=r.dtype, device=r.device)
        plan.radial_hidden(r, r_cut, p_env, widths, weights, h)
        ctx.save_for_backward(r, weights)
        ctx.plan, ctx.r_cut, ctx.p_env, ctx.widths = plan, r_cut, p_env, widths
        return h

    @staticmethod
    @once_differentiable
    def backward(ctx, dh):
        r, weights = ctx.saved_tensors
        dr = torch.empty_like(r)
        dW = torch.empty_like(weights)
        ctx.plan.radial_hidden_bwd(r, ctx.r_cut, ctx.p_env, ctx.widths, weights, _c(dh), dr, dW)
        return dr, dW, None, None, None, None


class _RadialWeights(torch.autograd.Function):
    """(h, W_last) -> w = h W_last (uvu_radial_weights); backward = uvu_radial_weights_bwd."""

    @staticmethod
    def forward(ctx, h, w_last, plan):
        i = plan.info
        w = torch.empty(h.shape[0], i.n_paths, i.mul, dtype=h.dtype, device=h.device)
        plan.radial_weights(h, w_last, w)
        ctx.save_for_backward(h, w_last)
        ctx.plan = plan
        return w

    @staticmethod
    @once_differentiable
    def backward(ctx, dw):
        h, w_last = ctx.saved_tensors
        need = ctx.needs_input_grad
        dh = torch.empty_like(h) if need[0] else None
        dwl = torch.empty_like(w_last) if need[1] else None
        ctx.plan.radial_weights_bwd(h, w_last, _c(dw), dh=dh, dw_last=dwl)
        return dh, dwl, None


def radial_conv(r, x, Y, weights, w_last, plan: "uvu.Plan", graph: "uvu.Graph", r_cut: float, p_env: int,
                widths, dx_mode: int = uvu.UVU_DX_STAGED):
    """The convolution with radial weights from edge lengths r [E]: h = uvu_radial_hidden(r) (the
    SiLU network, layers back to back in `weights`), w = h W_last (materialised on the tensor
    cores), out = uvu_conv(x, Y, w).  First derivatives with respect to r (forces), x, Y, the
    layers and W_last run in the library; second derivatives through the radial network are not
    provided."""
    h = _RadialHidden.apply(_c(r), _c(weights), plan, float(r_cut), int(p_env), [int(v) for v in widths])
    w = _RadialWeights.apply(h, _c(w_last), plan)
    return uvu_conv(x, Y, w, plan, graph, dx_mode)
