"""Python binding of libuvu.so (argument marshalling only).

Every function named ``uvu_*`` here calls the C entry point of the same name in
``include/uvu.h`` and raises ``UVUError`` when it returns a status other than UVU_OK.  All
arithmetic runs in the library's CUDA kernels; there is no fallback path: if the library cannot
be loaded, importing this module raises.

``Plan`` is a small convenience wrapper that passes torch tensors' device pointers and the
current CUDA stream; torch is used only for memory and streams.
"""

from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libuvu.so")

UVU_F32, UVU_F64 = 0, 1
UVU_DX_SENDER, UVU_DX_ATOMIC, UVU_DX_STAGED = 0, 1, 2
UVU_MODULE_CONV, UVU_MODULE_HVP, UVU_MODULE_TP, UVU_MODULE_TP_SHARED = 0, 1, 2, 3
UVU_FWD_AUTO, UVU_FWD_RECEIVER, UVU_FWD_SENDER = 0, 1, 2
STATUS = {0: "UVU_OK", 1: "UVU_ERR_INVALID_ARGUMENT", 2: "UVU_ERR_UNSUPPORTED",
          3: "UVU_ERR_COMPILE", 4: "UVU_ERR_CUDA", 5: "UVU_ERR_OUT_OF_MEMORY"}

# every symbol declared in include/uvu.h
EXPORTS = (
    "uvu_plan_create", "uvu_plan_destroy", "uvu_plan_info", "uvu_plan_cg", "uvu_plan_source",
    "uvu_plan_module_source", "uvu_plan_device_status",
    "uvu_csr_from_sorted_recv", "uvu_csr_transpose_workspace", "uvu_csr_transpose",
    "uvu_csr_transpose_noalloc", "uvu_graph_validate", "uvu_conv_fwd", "uvu_conv_bwd_edge",
    "uvu_conv_bwd_dx", "uvu_conv_bwd_dx_reduce", "uvu_conv_bwd_workspace", "uvu_conv_bwd",
    "uvu_conv_hvp", "uvu_conv_hvp_workspace", "uvu_tp_fwd", "uvu_tp_bwd", "uvu_tp_bwd_workspace",
    "uvu_conv_fwd_model", "uvu_conv_fwd_sender", "uvu_conv_fwd_mode",
    "uvu_mix_fwd", "uvu_mix_bwd", "uvu_mix_workspace", "uvu_conv_uvw_fwd",
    "uvu_radial_hidden", "uvu_conv_fwd_radial", "uvu_radial_module_source",
    "uvu_radial_weights", "uvu_radial_weights_workspace", "uvu_radial_weights_bwd", "uvu_radial_weights_bwd_workspace",
    "uvu_radial_hidden_bwd", "uvu_radial_hidden_bwd_workspace",
    "uvu_fma_rate_probe", "uvu_status_string", "uvu_last_error_message",
)


class UVUError(RuntimeError):
    def __init__(self, status: int, fn: str, msg: str):
        super().__init__(f"{fn}: {STATUS.get(status, status)}: {msg}")
        self.status = status


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"libuvu.so is not built ({LIB_PATH}); run __graft_entry__.build()")
    lib = ctypes.CDLL(LIB_PATH)
    P, I, I64, SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t
    sig = {
        "uvu_plan_create": [ctypes.c_char_p, ctypes.c_char_p, I, I, ctypes.POINTER(P)],
        "uvu_plan_destroy": [P],
        "uvu_plan_info": [P, P, P, P, P, P, P],
        "uvu_plan_cg": [P, I, P],
        "uvu_plan_source": [P, ctypes.POINTER(ctypes.c_char_p), ctypes.POINTER(ctypes.c_char_p)],
        "uvu_plan_module_source": [P, I, ctypes.POINTER(ctypes.c_char_p), ctypes.POINTER(ctypes.c_char_p)],
        "uvu_plan_device_status": [P, ctypes.POINTER(ctypes.c_uint), I],
        "uvu_csr_from_sorted_recv": [I64, I64, P, P, P],
        "uvu_csr_transpose_workspace": [I64, I64, ctypes.POINTER(SZ)],
        "uvu_csr_transpose": [I64, I64, P, P, P, P, P, P, SZ, P],
        "uvu_csr_transpose_noalloc": [I64, I64, P, P, P, P, P, P],
        "uvu_graph_validate": [I64, I64, P, P, P, ctypes.POINTER(I64), P],
        "uvu_conv_fwd": [P, I64, I64, P, P, P, P, P, P, P],
        "uvu_conv_bwd_edge": [P, I64, I64, P, P, P, P, P, P, P, P, P, P, P],
        "uvu_conv_bwd_dx": [P, I64, I64, P, P, P, P, P, P, P, P],
        "uvu_conv_bwd_dx_reduce": [P, I64, I64, P, P, P, P, P],
        "uvu_conv_bwd_workspace": [P, I64, I64, I, ctypes.POINTER(SZ)],
        "uvu_conv_bwd": [P, I64, I64, P, P, P, P, P, P, P, P, P, P, P, P, I, P, SZ, P],
        "uvu_conv_hvp": [P, I64, I64] + [P] * 16 + [SZ, P],
        "uvu_conv_hvp_workspace": [P, I64, I64, ctypes.POINTER(SZ)],
        "uvu_tp_fwd": [P, I64, P, P, P, I, P, P],
        "uvu_tp_bwd": [P, I64, P, P, P, I, P, P, P, P, P, SZ, P],
        "uvu_tp_bwd_workspace": [P, I64, I, ctypes.POINTER(SZ)],
        "uvu_conv_fwd_model": [P, I64, I64, ctypes.POINTER(I), ctypes.POINTER(ctypes.c_double),
                               ctypes.POINTER(ctypes.c_double)],
        "uvu_conv_fwd_sender": [P, I64, I64, P, P, P, P, P, P, P, P],
        "uvu_conv_fwd_mode": [P, I, I64, I64, P, P, P, P, P, P, P, P, P, P],
        "uvu_mix_fwd": [P, I64, I, P, P, P, P, SZ, P],
        "uvu_mix_bwd": [P, I64, I, P, P, P, P, P, P, SZ, P],
        "uvu_mix_workspace": [P, I64, I, ctypes.POINTER(SZ), ctypes.POINTER(SZ)],
        "uvu_conv_uvw_fwd": [P, I64, I64, P, P, P, P, P, P, I, P, P, P, SZ, P],
        "uvu_radial_hidden": [P, I64, P, ctypes.c_double, I, I, ctypes.POINTER(I), P, P, P],
        "uvu_conv_fwd_radial": [P, I64, I64, P, P, P, I, P, P, P, P, P],
        "uvu_radial_module_source": [P, I, ctypes.POINTER(ctypes.c_char_p), ctypes.POINTER(ctypes.c_char_p)],
        "uvu_fma_rate_probe": [I, I, I, P, ctypes.POINTER(ctypes.c_double), P],
        "uvu_radial_weights": [P, I64, P, I, P, P, P, SZ, P],
        "uvu_radial_weights_workspace": [P, I, ctypes.POINTER(SZ)],
        "uvu_radial_weights_bwd": [P, I64, P, I, P, P, P, P, P, SZ, P],
        "uvu_radial_weights_bwd_workspace": [P, I64, I, ctypes.POINTER(SZ)],
        "uvu_radial_hidden_bwd": [P, I64, P, ctypes.c_double, I, I, ctypes.POINTER(I), P, P, P, P, P, SZ, P],
        "uvu_radial_hidden_bwd_workspace": [P, I64, I, ctypes.POINTER(I), ctypes.POINTER(SZ)],
    }
    for name, args in sig.items():
        f = getattr(lib, name)
        f.argtypes = args
        f.restype = ctypes.c_int
    lib.uvu_status_string.argtypes = [ctypes.c_int]
    lib.uvu_status_string.restype = ctypes.c_char_p
    lib.uvu_last_error_message.argtypes = []
    lib.uvu_last_error_message.restype = ctypes.c_char_p
    return lib


lib = _load()


def _check(st: int, fn: str):
    if st != 0:
        raise UVUError(st, fn, lib.uvu_last_error_message().decode())


def _wrap(name):
    f = getattr(lib, name)

    def call(*args):
        _check(f(*args), name)

    call.__name__ = name
    call.__doc__ = f"Calls {name} of include/uvu.h; raises UVUError on failure."
    return call


for _n in ("uvu_plan_destroy", "uvu_plan_info", "uvu_plan_cg", "uvu_plan_source", "uvu_plan_module_source",
           "uvu_plan_device_status",
           "uvu_csr_from_sorted_recv", "uvu_csr_transpose_workspace", "uvu_csr_transpose",
           "uvu_csr_transpose_noalloc", "uvu_graph_validate", "uvu_conv_fwd", "uvu_conv_bwd_edge",
           "uvu_conv_bwd_dx", "uvu_conv_bwd_dx_reduce", "uvu_conv_bwd_workspace", "uvu_conv_bwd",
           "uvu_conv_hvp", "uvu_conv_hvp_workspace", "uvu_tp_fwd", "uvu_tp_bwd", "uvu_tp_bwd_workspace",
           "uvu_conv_fwd_model", "uvu_conv_fwd_sender", "uvu_conv_fwd_mode",
           "uvu_mix_fwd", "uvu_mix_bwd", "uvu_mix_workspace", "uvu_conv_uvw_fwd",
           "uvu_radial_hidden", "uvu_conv_fwd_radial", "uvu_radial_module_source", "uvu_fma_rate_probe",
           "uvu_radial_weights", "uvu_radial_weights_workspace", "uvu_radial_weights_bwd",
           "uvu_radial_weights_bwd_workspace", "uvu_radial_hidden_bwd", "uvu_radial_hidden_bwd_workspace"):
    globals()[_n] = _wrap(_n)


def fma_rate_probe(out, f64: bool, blocks: int, iters: int, stream=None) -> float:
    """Enqueue one launch of the FMA-chain probe into `out` (a device tensor of at least
    blocks * 256 elements of the dtype); returns the FMAs that launch performs."""
    n = ctypes.c_double()
    uvu_fma_rate_probe(UVU_F64 if f64 else UVU_F32, blocks, iters, _ptr(out), ctypes.byref(n), _stream(stream))
    return n.value


def uvu_plan_create(irreps_x: str, irreps_sh: str, lmax_out: int, dtype: int) -> int:
    h = ctypes.c_void_p()
    _check(lib.uvu_plan_create(irreps_x.encode(), irreps_sh.encode(), lmax_out, dtype,
                               ctypes.byref(h)), "uvu_plan_create")
    return h.value


def uvu_status_string(s: int) -> str:
    return lib.uvu_status_string(s).decode()


def uvu_last_error_message() -> str:
    return lib.uvu_last_error_message().decode()


# ----------------------------------------------------------------------- torch convenience

def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    import torch
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


@dataclass
class PlanInfo:
    mul: int
    dim_x: int
    dim_sh: int
    dim_out: int
    n_paths: int
    paths: list


class Plan:
    """Owns a uvu plan handle; methods take torch tensors already on the current device."""

    def __init__(self, irreps_x: str, irreps_sh: str, lmax_out: int, dtype: str = "float32"):
        self.dtype_name = dtype
        self.handle = uvu_plan_create(irreps_x, irreps_sh, lmax_out,
                                      UVU_F64 if dtype == "float64" else UVU_F32)
        vals = [ctypes.c_int() for _ in range(5)]
        uvu_plan_info(self.handle, *[ctypes.byref(v) for v in vals], None)
        P = vals[4].value
        arr = (ctypes.c_int * (3 * P))()
        uvu_plan_info(self.handle, None, None, None, None, None, arr)
        self.info = PlanInfo(vals[0].value, vals[1].value, vals[2].value, vals[3].value, P,
                             [tuple(arr[3 * i:3 * i + 3]) for i in range(P)])

    def __del__(self):
        h = getattr(self, "handle", None)
        if h:
            lib.uvu_plan_destroy(h)
            self.handle = None

    def cg(self, path: int):
        import numpy as np
        l1, l2, l3 = self.info.paths[path]
        out = np.zeros((2 * l1 + 1, 2 * l2 + 1, 2 * l3 + 1))
        uvu_plan_cg(self.handle, path, out.ctypes.data_as(ctypes.c_void_p))
        return out

    def device_status(self, reset: bool = True) -> int:
        """Status word of the plan's kernels on the current device (0 = no timeout)."""
        w = ctypes.c_uint()
        uvu_plan_device_status(self.handle, ctypes.byref(w), int(reset))
        return w.value

    def source(self):
        s, l = ctypes.c_char_p(), ctypes.c_char_p()
        uvu_plan_source(self.handle, ctypes.byref(s), ctypes.byref(l))
        return s.value.decode(), l.value.decode()

    def module_source(self, module: int):
        """(source, NVRTC log) of one of the plan's modules (UVU_MODULE_*); compiles it on the host
        if needed."""
        s, l = ctypes.c_char_p(), ctypes.c_char_p()
        uvu_plan_module_source(self.handle, module, ctypes.byref(s), ctypes.byref(l))
        return s.value.decode(), l.value.decode()

    def hvp_source(self):
        return self.module_source(UVU_MODULE_HVP)

    def radial_source(self, hidden: int):
        """(source, NVRTC log) of the fused radial forward for `hidden` (fixes the plan's hidden
        width); compiles it on the host if needed."""
        s, l = ctypes.c_char_p(), ctypes.c_char_p()
        uvu_radial_module_source(self.handle, int(hidden), ctypes.byref(s), ctypes.byref(l))
        return s.value.decode(), l.value.decode()

    def radial_hidden(self, r, r_cut, p_env, widths, weights, h, stream=None):
        """Radial network h = silu(... silu(basis(r) W_1) ... W_L) (see uvu_radial_hidden);
        `widths` = [n_basis, H_1, ..., H_L] (host ints), `weights` the layers back to back."""
        wd = (ctypes.c_int * len(widths))(*[int(v) for v in widths])
        uvu_radial_hidden(self.handle, r.numel(), _ptr(r), float(r_cut), int(p_env), len(widths) - 1, wd,
                          _ptr(weights), _ptr(h), _stream(stream))

    def fwd_radial(self, n_nodes, x, Y, h, w_last, recv_offsets, src, out, stream=None):
        """Convolution with fused radial weights w = h W_last (see uvu_conv_fwd_radial)."""
        uvu_conv_fwd_radial(self.handle, n_nodes, src.numel() if src is not None else 0, _ptr(x), _ptr(Y), _ptr(h),
                            int(w_last.shape[0]), _ptr(w_last), _ptr(recv_offsets), _ptr(src), _ptr(out),
                            _stream(stream))

    def radial_weights_workspace(self, hidden) -> int:
        b = ctypes.c_size_t()
        uvu_radial_weights_workspace(self.handle, int(hidden), ctypes.byref(b))
        return b.value

    def radial_weights(self, h, w_last, w, workspace=None, stream=None):
        """Materialised last layer w = h W_last (see uvu_radial_weights)."""
        import torch
        if workspace is None:
            workspace = torch.empty(max(16, self.radial_weights_workspace(h.shape[1])), dtype=torch.uint8, device=h.device)
        uvu_radial_weights(self.handle, h.shape[0], _ptr(h), int(h.shape[1]), _ptr(w_last), _ptr(w), _ptr(workspace),
                           workspace.numel(), _stream(stream))

    def radial_weights_bwd_workspace(self, n_edges, hidden) -> int:
        b = ctypes.c_size_t()
        uvu_radial_weights_bwd_workspace(self.handle, n_edges, int(hidden), ctypes.byref(b))
        return b.value

    def radial_weights_bwd(self, h, w_last, dw, dh=None, dw_last=None, workspace=None, stream=None):
        """dh = dw W_last^T and dW_last = h^T dw (see uvu_radial_weights_bwd)."""
        import torch
        E, H = h.shape
        if workspace is None:
            workspace = torch.empty(max(16, self.radial_weights_bwd_workspace(E, H)), dtype=torch.uint8, device=h.device)
        uvu_radial_weights_bwd(self.handle, E, _ptr(h), int(H), _ptr(w_last), _ptr(dw), _ptr(dh), _ptr(dw_last),
                               _ptr(workspace), workspace.numel(), _stream(stream))

    def radial_hidden_bwd_workspace(self, n_edges, widths) -> int:
        wd = (ctypes.c_int * len(widths))(*[int(v) for v in widths])
        b = ctypes.c_size_t()
        uvu_radial_hidden_bwd_workspace(self.handle, n_edges, len(widths) - 1, wd, ctypes.byref(b))
        return b.value

    def radial_hidden_bwd(self, r, r_cut, p_env, widths, weights, dh, dr, dweights, workspace=None, stream=None):
        """Edge-length and layer gradients of <dh, h> (see uvu_radial_hidden_bwd)."""
        import torch
        wd = (ctypes.c_int * len(widths))(*[int(v) for v in widths])
        if workspace is None:
            workspace = torch.empty(max(16, self.radial_hidden_bwd_workspace(r.numel(), widths)), dtype=torch.uint8,
                                    device=r.device)
        uvu_radial_hidden_bwd(self.handle, r.numel(), _ptr(r), float(r_cut), int(p_env), len(widths) - 1, wd,
                              _ptr(weights), _ptr(dh), _ptr(dr), _ptr(dweights), _ptr(workspace), workspace.numel(),
                              _stream(stream))

    def tp_fwd(self, batch, x, y, w, out, w_shared=False, stream=None):
        """Batched tensor product (see uvu_tp_fwd)."""
        uvu_tp_fwd(self.handle, batch, _ptr(x), _ptr(y), _ptr(w), int(bool(w_shared)), _ptr(out),
                   _stream(stream))

    def tp_workspace_bytes(self, batch, w_shared) -> int:
        b = ctypes.c_size_t()
        uvu_tp_bwd_workspace(self.handle, batch, int(bool(w_shared)), ctypes.byref(b))
        return b.value

    def tp_bwd(self, batch, x, y, w, d_out, dx=None, dy=None, dw=None, w_shared=False,
               workspace=None, stream=None):
        """VJP of the batched tensor product (see uvu_tp_bwd); a shared dw needs `workspace`
        (a uint8 device tensor of tp_workspace_bytes() bytes), allocated here with torch if None."""
        ws_ptr, ws_bytes = None, 0
        need = self.tp_workspace_bytes(batch, w_shared) if dw is not None else 0
        if need:
            if workspace is None:
                import torch
                workspace = torch.empty(need, dtype=torch.uint8, device=d_out.device)
            ws_ptr, ws_bytes = _ptr(workspace), workspace.numel() * workspace.element_size()
        uvu_tp_bwd(self.handle, batch, _ptr(x), _ptr(y), _ptr(w), int(bool(w_shared)), _ptr(d_out),
                   _ptr(dx), _ptr(dy), _ptr(dw), ws_ptr, ws_bytes, _stream(stream))

    def fwd(self, n_nodes, x, Y, w, recv_offsets, src, out, stream=None):
        uvu_conv_fwd(self.handle, n_nodes, src.numel() if src is not None else 0, _ptr(x), _ptr(Y),
                     _ptr(w), _ptr(recv_offsets), _ptr(src), _ptr(out), _stream(stream))

    def fwd_model(self, n_nodes, n_edges):
        """(chosen UVU_FWD_* mode, bytes of the receiver forward, bytes of the sender forward)."""
        c, br, bs = ctypes.c_int(), ctypes.c_double(), ctypes.c_double()
        uvu_conv_fwd_model(self.handle, n_nodes, n_edges, ctypes.byref(c), ctypes.byref(br), ctypes.byref(bs))
        return c.value, br.value, bs.value

    def fwd_sender(self, n_nodes, n_edges, x, Y, w, send_offsets, send_eids, send_recv, out, stream=None):
        uvu_conv_fwd_sender(self.handle, n_nodes, n_edges, _ptr(x), _ptr(Y), _ptr(w), _ptr(send_offsets),
                            _ptr(send_eids), _ptr(send_recv), _ptr(out), _stream(stream))

    def fwd_mode(self, mode, n_nodes, n_edges, x, Y, w, graph, out, stream=None):
        """Forward by mode (UVU_FWD_*) over a Graph holding both CSRs."""
        uvu_conv_fwd_mode(self.handle, mode, n_nodes, n_edges, _ptr(x), _ptr(Y), _ptr(w),
                          _ptr(graph.recv_offsets), _ptr(graph.src), _ptr(graph.send_offsets),
                          _ptr(graph.send_eids), _ptr(graph.send_recv), _ptr(out), _stream(stream))

    def mix_workspace_bytes(self, n_nodes, w_out):
        """(forward bytes, backward bytes) of device workspace for the channel mixing."""
        f, b = ctypes.c_size_t(), ctypes.c_size_t()
        uvu_mix_workspace(self.handle, n_nodes, w_out, ctypes.byref(f), ctypes.byref(b))
        return f.value, b.value

    def _mix_ws(self, n_nodes, w_out, bwd, workspace, device):
        need = self.mix_workspace_bytes(n_nodes, w_out)[1 if bwd else 0]
        if workspace is None:
            import torch
            workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=device)
        return _ptr(workspace), workspace.numel() * workspace.element_size()

    def mix_fwd(self, n_nodes, w_out, inp, M, out, workspace=None, stream=None):
        """Per-path channel mixing of a UVU output (see uvu_mix_fwd); `workspace` (uint8) is
        allocated here with torch if None."""
        ws, nb = self._mix_ws(n_nodes, w_out, False, workspace, out.device)
        uvu_mix_fwd(self.handle, n_nodes, w_out, _ptr(inp), _ptr(M), _ptr(out), ws, nb, _stream(stream))

    def mix_bwd(self, n_nodes, w_out, inp, M, d_out, d_in=None, dM=None, workspace=None, stream=None):
        """VJP of mix_fwd (see uvu_mix_bwd)."""
        ws, nb = self._mix_ws(n_nodes, w_out, True, workspace, d_out.device)
        uvu_mix_bwd(self.handle, n_nodes, w_out, _ptr(inp), _ptr(M), _ptr(d_out), _ptr(d_in), _ptr(dM),
                    ws, nb, _stream(stream))

    def uvw_fwd(self, n_nodes, x, Y, w, recv_offsets, src, M, w_out, uvu_out, out, workspace=None, stream=None):
        """Factorised UVW convolution (see uvu_conv_uvw_fwd)."""
        ws, nb = self._mix_ws(n_nodes, w_out, False, workspace, out.device)
        uvu_conv_uvw_fwd(self.handle, n_nodes, src.numel(), _ptr(x), _ptr(Y), _ptr(w), _ptr(recv_offsets),
                         _ptr(src), _ptr(M), w_out, _ptr(uvu_out), _ptr(out), ws, nb, _stream(stream))

    def bwd_edge(self, n_nodes, x, Y, w, recv_offsets, src, d_out, dY=None, dw=None,
                 dx_atomic=None, dx_edge=None, stream=None):
        uvu_conv_bwd_edge(self.handle, n_nodes, src.numel(), _ptr(x), _ptr(Y), _ptr(w),
                          _ptr(recv_offsets), _ptr(src), _ptr(d_out), _ptr(dY), _ptr(dw),
                          _ptr(dx_atomic), _ptr(dx_edge), _stream(stream))

    def bwd_dx(self, n_nodes, n_edges, Y, w, send_offsets, send_eids, send_recv, d_out, dx,
               stream=None):
        uvu_conv_bwd_dx(self.handle, n_nodes, n_edges, _ptr(Y), _ptr(w), _ptr(send_offsets),
                        _ptr(send_eids), _ptr(send_recv), _ptr(d_out), _ptr(dx), _stream(stream))

    def bwd_dx_reduce(self, n_nodes, n_edges, send_offsets, send_eids, dx_edge, dx, stream=None):
        uvu_conv_bwd_dx_reduce(self.handle, n_nodes, n_edges, _ptr(send_offsets), _ptr(send_eids),
                               _ptr(dx_edge), _ptr(dx), _stream(stream))

    def workspace_bytes(self, n_nodes, n_edges, dx_mode) -> int:
        b = ctypes.c_size_t()
        uvu_conv_bwd_workspace(self.handle, n_nodes, n_edges, dx_mode, ctypes.byref(b))
        return b.value

    def bwd(self, n_nodes, x, Y, w, recv_offsets, src, send_offsets, send_eids, send_recv,
            d_out, dx=None, dY=None, dw=None, dx_mode=UVU_DX_SENDER, workspace=None,
            stream=None):
        """Full VJP.  UVU_DX_STAGED needs `workspace` (a uint8 device tensor of at least
        workspace_bytes() bytes); pass None to let this wrapper allocate it with torch."""
        n_edges = src.numel()
        ws_ptr, ws_bytes = None, 0
        if dx_mode == UVU_DX_STAGED and dx is not None:
            need = self.workspace_bytes(n_nodes, n_edges, dx_mode)
            if workspace is None:
                import torch
                workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=src.device)
            ws_ptr, ws_bytes = _ptr(workspace), workspace.numel() * workspace.element_size()
        uvu_conv_bwd(self.handle, n_nodes, n_edges, _ptr(x), _ptr(Y), _ptr(w),
                     _ptr(recv_offsets), _ptr(src), _ptr(send_offsets), _ptr(send_eids),
                     _ptr(send_recv), _ptr(d_out), _ptr(dx), _ptr(dY), _ptr(dw), dx_mode,
                     ws_ptr, ws_bytes, _stream(stream))


def _hvp_method(self, n_nodes, x, Y, w, recv_offsets, src, send_offsets, send_eids, d_out,
                ax=None, aY=None, aw=None, grad_d_out=None, grad_x=None, grad_Y=None, grad_w=None,
                workspace=None, stream=None):
    """Double backward: gradients of <ax,dx> + <aY,dY> + <aw,dw> (see uvu_conv_hvp)."""
    n_edges = src.numel()
    ws_ptr, ws_bytes = None, 0
    if grad_x is not None:
        b = ctypes.c_size_t()
        uvu_conv_hvp_workspace(self.handle, n_nodes, n_edges, ctypes.byref(b))
        if b.value:
            if workspace is None:
                import torch
                workspace = torch.empty(b.value, dtype=torch.uint8, device=src.device)
            ws_ptr, ws_bytes = _ptr(workspace), workspace.numel() * workspace.element_size()
    uvu_conv_hvp(self.handle, n_nodes, n_edges, _ptr(x), _ptr(Y), _ptr(w), _ptr(recv_offsets),
                 _ptr(src), _ptr(send_offsets), _ptr(send_eids), _ptr(d_out), _ptr(ax), _ptr(aY),
                 _ptr(aw), _ptr(grad_d_out), _ptr(grad_x), _ptr(grad_Y), _ptr(grad_w), ws_ptr,
                 ws_bytes, _stream(stream))


Plan.hvp = _hvp_method


class Graph:
    """Receiver CSR and transposed CSR built on the device by the library's kernels."""

    def __init__(self, n_nodes: int, recv, src, stream=None):
        import torch
        dev = src.device
        self.n_nodes = n_nodes
        self.n_edges = src.numel()
        self.src = src
        self.recv_offsets = torch.empty(n_nodes + 1, dtype=torch.int32, device=dev)
        uvu_csr_from_sorted_recv(n_nodes, self.n_edges, _ptr(recv), _ptr(self.recv_offsets),
                                 _stream(stream))
        nb = ctypes.c_size_t()
        uvu_csr_transpose_workspace(n_nodes, self.n_edges, ctypes.byref(nb))
        ws = torch.empty(max(nb.value, 16), dtype=torch.uint8, device=dev)
        self.send_offsets = torch.empty(n_nodes + 1, dtype=torch.int32, device=dev)
        self.send_eids = torch.empty(max(self.n_edges, 1), dtype=torch.int32, device=dev)
        self.send_recv = torch.empty(max(self.n_edges, 1), dtype=torch.int32, device=dev)
        uvu_csr_transpose(n_nodes, self.n_edges, _ptr(self.recv_offsets), _ptr(src),
                          _ptr(self.send_offsets), _ptr(self.send_eids), _ptr(self.send_recv),
                          _ptr(ws), nb.value, _stream(stream))
        self._ws = ws
