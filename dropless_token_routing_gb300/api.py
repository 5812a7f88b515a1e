"""Torch-facing wrappers of the C ABI: device memory and streams come from PyTorch,
every computation runs in libmoe's kernels.  Names follow include/moe.h."""
from __future__ import annotations

import ctypes
from dataclasses import dataclass
from typing import Optional

import torch

from . import _native as N

__all__ = ["make_dims", "Workspace", "router_logits", "route_topk", "permute", "permute_rows",
           "grouped_swiglu_fwd", "unpermute_combine", "grouped_bwd_dx", "grouped_bwd_dw",
           "route_topk_bwd", "LayerParams", "MoELayer", "get_device_error", "debug_timeout_probe"]


def _p(t: Optional[torch.Tensor]):
    return None if t is None else t.data_ptr()


def _s(stream=None):
    return (stream if stream is not None else torch.cuda.current_stream()).cuda_stream


def _dt(dtype) -> int:
    if dtype in (torch.float32, "f32"):
        return N.MOE_F32
    if dtype in (torch.bfloat16, "bf16"):
        return N.MOE_BF16
    raise ValueError(f"unsupported dtype {dtype}")


def make_dims(T, d, E, k, f, S=0, f_s=0, dtype=torch.bfloat16, capacity=0, rearrange=0) -> N.MoeDims:
    """capacity = 0: dropless; C > 0: drop-and-pad with C rows per expert.
    rearrange (flags) = 0: rearranged copies; 1: rearrangement fused into the GEMM loads;
    2: the second expert GEMM writes its rows in token-major order for the combine; 3: both."""
    return N.MoeDims(int(T), int(d), int(E), int(k), int(f), int(S), int(f_s) if S else 0, _dt(dtype),
                     int(capacity), int(rearrange))


def perm_rows(dims: N.MoeDims) -> int:
    """Rows of the permuted buffers: T*k dropless, E*C with a capacity C."""
    return dims.E * dims.capacity if dims.capacity > 0 else dims.T * dims.k


class Workspace:
    """Device workspace of moe_workspace_bytes(dims) bytes, initialised once."""

    def __init__(self, dims: N.MoeDims, device="cuda", stream=None):
        self.dims = dims
        self.nbytes = int(N.lib().moe_workspace_bytes(ctypes.byref(dims)))
        if self.nbytes == 0:
            raise N.MoeError(N.STATUS_CODE["MOE_ERR_BAD_DIMS"], "moe_workspace_bytes")
        self.buf = torch.empty(self.nbytes + 256, dtype=torch.uint8, device=device)
        off = (-self.buf.data_ptr()) % 256
        self.ptr = self.buf.data_ptr() + off
        N.check(N.lib().moe_workspace_init(self.ptr, self.nbytes, ctypes.byref(dims), _s(stream)),
                "moe_workspace_init")


def get_device_error(ws: Workspace, stream=None) -> int:
    out = ctypes.c_int(0)
    N.check(N.lib().moe_get_device_error(ws.ptr, _s(stream), ctypes.byref(out)), "moe_get_device_error")
    return out.value


def debug_timeout_probe(ws: Workspace, limit_ns: int, stream=None) -> None:
    N.check(N.lib().moe_debug_timeout_probe(ws.ptr, ws.nbytes, int(limit_ns), _s(stream)),
            "moe_debug_timeout_probe")


def router_logits(x, w_r, dims, logits, ws: Workspace, stream=None):
    N.check(N.lib().moe_router_logits(_p(x), _p(w_r), ctypes.byref(dims), _p(logits), ws.ptr,
                                      ws.nbytes, _s(stream)), "moe_router_logits")


def route_topk(logits, bias, k, topk_idx, topk_w, counts, ws: Workspace, stream=None):
    T, E = logits.shape
    N.check(N.lib().moe_route_topk(_p(logits), _p(bias), T, E, k, _p(topk_idx), _p(topk_w),
                                   _p(counts), ws.ptr, ws.nbytes, _s(stream)), "moe_route_topk")


def permute(x, topk_idx, topk_w, dims, x_perm, dest, row_src, offsets, w_perm, ws: Workspace,
            stream=None):
    N.check(N.lib().moe_permute(_p(x), _p(topk_idx), _p(topk_w), ctypes.byref(dims), _p(x_perm),
                                _p(dest), _p(row_src), _p(offsets), _p(w_perm), ws.ptr, ws.nbytes,
                                _s(stream)), "moe_permute")


def permute_rows(x, dest, dims, x_perm, stream=None):
    N.check(N.lib().moe_permute_rows(_p(x), _p(dest), ctypes.byref(dims), _p(x_perm), _s(stream)),
            "moe_permute_rows")


def grouped_swiglu_fwd(x_perm, x, w13, w2, ws13, ws2, offsets, dims, z, h, z_sh, h_sh, y_perm, y_sh,
                       ws: Workspace, stream=None):
    N.check(N.lib().moe_grouped_swiglu_fwd(
        _p(x_perm), _p(x), _p(w13), _p(w2), _p(ws13), _p(ws2), _p(offsets), ctypes.byref(dims),
        _p(z), _p(h), _p(z_sh), _p(h_sh), _p(y_perm), _p(y_sh), ws.ptr, ws.nbytes, _s(stream)),
        "moe_grouped_swiglu_fwd")


def unpermute_combine(y_perm, dest, topk_w, y_sh, dims, y, stream=None):
    N.check(N.lib().moe_unpermute_combine(_p(y_perm), _p(dest), _p(topk_w), _p(y_sh),
                                          ctypes.byref(dims), _p(y), _s(stream)),
            "moe_unpermute_combine")


def grouped_bwd_dx(dy_perm, dy, z, z_sh, w13, w2, ws13, ws2, w_perm, offsets, dest, dims, dz, dz_sh,
                   hw, hw_sh, dx_perm, dx_sh, dgate, ws: Workspace, stream=None):
    N.check(N.lib().moe_grouped_bwd_dx(
        _p(dy_perm), _p(dy), _p(z), _p(z_sh), _p(w13), _p(w2), _p(ws13), _p(ws2), _p(w_perm),
        _p(offsets), _p(dest), ctypes.byref(dims), _p(dz), _p(dz_sh), _p(hw), _p(hw_sh),
        _p(dx_perm), _p(dx_sh), _p(dgate), ws.ptr, ws.nbytes, _s(stream)), "moe_grouped_bwd_dx")


def grouped_bwd_dw(x_perm, x, hw, hw_sh, dz, dz_sh, dy_perm, dy, offsets, dims, dw13, dw2, dws13,
                   dws2, ws: Workspace, stream=None):
    N.check(N.lib().moe_grouped_bwd_dw(
        _p(x_perm), _p(x), _p(hw), _p(hw_sh), _p(dz), _p(dz_sh), _p(dy_perm), _p(dy), _p(offsets),
        ctypes.byref(dims), _p(dw13), _p(dw2), _p(dws13), _p(dws2), ws.ptr, ws.nbytes, _s(stream)),
        "moe_grouped_bwd_dw")


def route_topk_bwd(topk_idx, topk_w, dgate, E, dlogits, stream=None):
    T, k = topk_idx.shape
    N.check(N.lib().moe_route_topk_bwd(_p(topk_idx), _p(topk_w), _p(dgate), T, E, k, _p(dlogits),
                                       _s(stream)), "moe_route_topk_bwd")


def route_balance(logits, bias, counts, k, alpha, prob_mean, aux_loss, ws: Workspace, stream=None):
    T, E = logits.shape
    N.check(N.lib().moe_route_balance(_p(logits), _p(bias), _p(counts), T, E, k, float(alpha),
                                      _p(prob_mean), _p(aux_loss), ws.ptr, ws.nbytes, _s(stream)),
            "moe_route_balance")


def route_topk_balance(logits, bias, k, alpha, topk_idx, topk_w, counts, prob_mean, aux_loss, ws: Workspace,
                       stream=None):
    T, E = logits.shape
    N.check(N.lib().moe_route_topk_balance(_p(logits), _p(bias), T, E, k, float(alpha), _p(topk_idx),
                                           _p(topk_w), _p(counts), _p(prob_mean), _p(aux_loss), ws.ptr,
                                           ws.nbytes, _s(stream)), "moe_route_topk_balance")


def route_balance_bwd(logits, bias, counts, k, alpha, grad, dlogits, stream=None):
    T, E = logits.shape
    N.check(N.lib().moe_route_balance_bwd(_p(logits), _p(bias), _p(counts), T, E, k, float(alpha),
                                          float(grad), _p(dlogits), _s(stream)),
            "moe_route_balance_bwd")


def route_balance_seq(logits, bias, topk_idx, k, group_len, alpha, prob_mean, counts, aux_loss,
                      ws: Workspace, stream=None):
    T, E = logits.shape
    N.check(N.lib().moe_route_balance_seq(_p(logits), _p(bias), _p(topk_idx), T, E, k, int(group_len),
                                          float(alpha), _p(prob_mean), _p(counts), _p(aux_loss), ws.ptr,
                                          ws.nbytes, _s(stream)), "moe_route_balance_seq")


def route_balance_seq_bwd(logits, bias, counts, k, group_len, n_groups, alpha, grad, dlogits, stream=None):
    T, E = logits.shape
    N.check(N.lib().moe_route_balance_seq_bwd(_p(logits), _p(bias), _p(counts), T, E, k, int(group_len),
                                              int(n_groups), float(alpha), float(grad), _p(dlogits),
                                              _s(stream)), "moe_route_balance_seq_bwd")


@dataclass
class LayerParams:
    w13: torch.Tensor
    w2: torch.Tensor
    w_r: Optional[torch.Tensor] = None
    bias: Optional[torch.Tensor] = None
    ws13: Optional[torch.Tensor] = None
    ws2: Optional[torch.Tensor] = None

    def c(self) -> N.LayerParams:
        return N.LayerParams(_p(self.w_r), _p(self.bias), _p(self.w13), _p(self.w2), _p(self.ws13),
                             _p(self.ws2))


class MoELayer:
    """One dropless MoE layer: caller-owned saved activations, gradients and workspace.

    ``forward(x, logits_in=None)`` runs moe_layer_fwd; ``backward(dy)`` runs
    moe_layer_bwd on the values the last forward saved. ``recompute=True`` keeps neither
    the rearranged input nor h between the two (selective recompute). ``capacity=C > 0``
    runs the drop-and-pad variant with C rows per expert instead of the dropless layer;
    ``rearrange=1`` fuses the rearrangement into the GEMMs' operand loads, ``rearrange=2`` the
    un-rearrangement into the second GEMM's stores (token-major rows), 3 both.
    """

    def __init__(self, params: LayerParams, T, d, E, k, f, S=0, f_s=0, dtype=torch.bfloat16,
                 device="cuda", logits_input=False, recompute=False, capacity=0, rearrange=0):
        self.params = params
        self.dims = make_dims(T, d, E, k, f, S, f_s, dtype, capacity, rearrange)
        self.T, self.d, self.E, self.k, self.f, self.S, self.f_s = T, d, E, k, f, S, f_s
        self.dtype = dtype
        Tk = T * k
        R = perm_rows(self.dims)
        dev = device
        emp = lambda *shape, dt=dtype: torch.empty(shape, dtype=dt, device=dev)  # noqa: E731
        self.ws = Workspace(self.dims, device=dev)
        self.saved = dict(
            logits=None if logits_input else emp(T, E, dt=torch.float32),
            topk_idx=emp(T, k, dt=torch.int32), topk_w=emp(T, k, dt=torch.float32),
            counts=emp(E, dt=torch.int32), offsets=emp(E + 1, dt=torch.int32),
            dest=emp(Tk, dt=torch.int32), row_src=emp(R, dt=torch.int32),
            w_perm=emp(R, dt=torch.float32), x_perm=None if recompute else emp(R, d),
            z=emp(R, 2 * f), h=None if recompute else emp(R, f),
            z_sh=emp(S * T, 2 * f_s) if S else None,
            h_sh=emp(S * T, f_s) if (S and not recompute) else None)
        self.y = emp(T, d)
        self.grads = None
        self._x = None

    def _saved_c(self):
        s = self.saved
        return N.LayerSaved(*[_p(s[n]) for n in ("logits", "topk_idx", "topk_w", "counts", "offsets",
                                                  "dest", "row_src", "w_perm", "x_perm", "z", "h",
                                                  "z_sh", "h_sh")])

    def alloc_grads(self, with_dlogits=None):
        T, d, E, f, S, f_s = self.T, self.d, self.E, self.f, self.S, self.f_s
        dev, dt = self.y.device, self.dtype
        want_dl = (self.params.w_r is None) if with_dlogits is None else with_dlogits
        self.grads = dict(
            dx=torch.empty(T, d, dtype=dt, device=dev),
            dw13=torch.empty(E, 2 * f, d, dtype=dt, device=dev),
            dw2=torch.empty(E, d, f, dtype=dt, device=dev),
            dws13=torch.empty(S, 2 * f_s, d, dtype=dt, device=dev) if S else None,
            dws2=torch.empty(S, d, f_s, dtype=dt, device=dev) if S else None,
            dw_r=torch.empty(d, E, dtype=torch.float32, device=dev) if self.params.w_r is not None else None,
            dlogits=torch.empty(T, E, dtype=torch.float32, device=dev) if want_dl else None)
        return self.grads

    def forward(self, x, logits_in=None, stream=None):
        self._x = x
        pc, sc = self.params.c(), self._saved_c()
        N.check(N.lib().moe_layer_fwd(ctypes.byref(pc), _p(x), _p(logits_in), ctypes.byref(self.dims),
                                      ctypes.byref(sc), _p(self.y), self.ws.ptr, self.ws.nbytes,
                                      _s(stream)), "moe_layer_fwd")
        return self.y

    def backward(self, dy, x=None, stream=None):
        if self.grads is None:
            self.alloc_grads()
        x = self._x if x is None else x
        g = self.grads
        gc = N.LayerGrads(*[_p(g[n]) for n in ("dx", "dw13", "dw2", "dws13", "dws2", "dw_r", "dlogits")])
        pc, sc = self.params.c(), self._saved_c()
        N.check(N.lib().moe_layer_bwd(ctypes.byref(pc), ctypes.byref(sc), _p(x), _p(dy),
                                      ctypes.byref(self.dims), ctypes.byref(gc), self.ws.ptr,
                                      self.ws.nbytes, _s(stream)), "moe_layer_bwd")
        return g
