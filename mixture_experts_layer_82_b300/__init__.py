"""DeepSeekMoE layer forward on one B300 (sm_103a): Python binding of libmoe.

The binding only marshals arguments: every step of the layer runs in the
CUDA kernels of ``libmoe.so`` (built in-tree by ``build.py``).  PyTorch
provides device memory and streams.  Importing this package fails loudly if
the shared library is missing: there is no CPU fallback.

Calls (same names as the C ABI in include/moe.h):
    moe_route, moe_permute, moe_experts_grouped, moe_combine,
    moe_bias_update, moe_quantize_weights_fp8, moe_get_device_error,
    moe_workspace_bytes, moe_check_cfg
and ``MoELayer``, which owns the buffers of one layer and runs the five
calls of a forward step in order on one stream.
"""

from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libmoe.so")

if not os.path.exists(LIB_PATH):
    raise ImportError(
        f"{LIB_PATH} is missing: build it with `python mixture_experts_layer_82_b300/build.py`")
_lib = ctypes.CDLL(LIB_PATH)

DTYPE_FP32, DTYPE_BF16, DTYPE_FP8_E4M3 = 0, 1, 2
_DTYPES = {"fp32": DTYPE_FP32, "bf16": DTYPE_BF16, "fp8": DTYPE_FP8_E4M3}

STATUS = {0: "MOE_OK", 1: "MOE_ERR_INVALID_ARG", 2: "MOE_ERR_SHAPE", 3: "MOE_ERR_ALIGN",
          4: "MOE_ERR_CUDA", 5: "MOE_ERR_TIMEOUT", 6: "MOE_ERR_DEVICE",
          7: "MOE_ERR_WORKSPACE"}

EXPORTED = ("moe_status_str", "moe_version", "moe_check_cfg", "moe_workspace_bytes",
            "moe_route", "moe_permute", "moe_experts_grouped", "moe_combine",
            "moe_bias_update", "moe_quantize_weights_fp8", "moe_get_device_error",
            "moe_route_static_scratch", "moe_experts_grouped_gather", "moe_balance_stat",
            "moe_selftest_wait", "moe_backward_workspace_bytes", "moe_combine_backward",
            "moe_experts_backward_input", "moe_experts_backward_weights", "moe_route_backward",
            "moe_experts_grouped_train", "moe_experts_grouped_gated", "moe_transpose_weights_fp8",
            "moe_experts_backward_input_fp8", "moe_experts_backward_weights_fp8",
            "moe_experts_grouped_train_fp8", "moe_quantize_act_fp8_128x1")


class MoeCfg(ctypes.Structure):
    """Mirror of moe_cfg_t."""
    _fields_ = [("T", ctypes.c_int32), ("d", ctypes.c_int32), ("E", ctypes.c_int32),
                ("n_groups", ctypes.c_int32), ("topk_groups", ctypes.c_int32),
                ("K", ctypes.c_int32), ("n_shared", ctypes.c_int32), ("inter", ctypes.c_int32),
                ("group_score_topn", ctypes.c_int32), ("route_scale", ctypes.c_float),
                ("gamma", ctypes.c_float), ("dtype", ctypes.c_int32)]


class MoeError(RuntimeError):
    def __init__(self, fn, status):
        self.status = status
        super().__init__(f"{fn}: {STATUS.get(status, status)} "
                         f"({_lib.moe_status_str(status).decode()})")


_P = ctypes.c_void_p
_CFG = ctypes.POINTER(MoeCfg)
_lib.moe_status_str.restype = ctypes.c_char_p
_lib.moe_status_str.argtypes = [ctypes.c_int]
_lib.moe_version.restype = ctypes.c_int32
_lib.moe_version.argtypes = []
_lib.moe_check_cfg.restype = ctypes.c_int
_lib.moe_check_cfg.argtypes = [_CFG]
_lib.moe_workspace_bytes.restype = ctypes.c_size_t
_lib.moe_workspace_bytes.argtypes = [_CFG]
_lib.moe_route.restype = ctypes.c_int
_lib.moe_route.argtypes = [_CFG] + [_P] * 11 + [_P, ctypes.c_size_t, _P]
_lib.moe_permute.restype = ctypes.c_int
_lib.moe_permute.argtypes = [_CFG] + [_P] * 6 + [_P]
_lib.moe_experts_grouped.restype = ctypes.c_int
_lib.moe_experts_grouped.argtypes = [_CFG] + [_P] * 15 + [_P, ctypes.c_size_t, _P]
_lib.moe_experts_grouped_gated.restype = ctypes.c_int
_lib.moe_experts_grouped_gated.argtypes = [_CFG] + [_P] * 17 + [_P, ctypes.c_size_t, _P]
_lib.moe_experts_grouped_gather.restype = ctypes.c_int
_lib.moe_experts_grouped_gather.argtypes = [_CFG] + [_P] * 14 + [_P, ctypes.c_size_t, _P]
_lib.moe_balance_stat.restype = ctypes.c_int
_lib.moe_balance_stat.argtypes = [_CFG, _P, _P, ctypes.c_int32, ctypes.c_float, _P, _P, _P, _P,
                                  ctypes.c_size_t, _P]
_lib.moe_combine.restype = ctypes.c_int
_lib.moe_combine.argtypes = [_CFG] + [_P] * 5 + [_P]
_lib.moe_bias_update.restype = ctypes.c_int
_lib.moe_bias_update.argtypes = [_CFG, _P, _P, _P]
_lib.moe_quantize_weights_fp8.restype = ctypes.c_int
_lib.moe_quantize_weights_fp8.argtypes = [_P, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                                          _P, _P, _P]
_lib.moe_selftest_wait.restype = ctypes.c_int
_lib.moe_selftest_wait.argtypes = [ctypes.c_int64, _P]
_lib.moe_get_device_error.restype = ctypes.c_int
_lib.moe_get_device_error.argtypes = [_P]
_lib.moe_route_static_scratch.restype = ctypes.c_int
_lib.moe_route_static_scratch.argtypes = [_CFG] + [_P] * 11 + [_P]


_lib.moe_backward_workspace_bytes.restype = ctypes.c_size_t
_lib.moe_backward_workspace_bytes.argtypes = [_CFG]
_lib.moe_combine_backward.argtypes = [_CFG] + [_P] * 6 + [_P]
_lib.moe_experts_backward_input.argtypes = ([_CFG] + [_P] * 11 + [ctypes.c_int32] +
                                            [_P, ctypes.c_size_t, _P])
_lib.moe_experts_grouped_train.argtypes = ([_CFG] + [_P] * 10 + [ctypes.c_size_t] +
                                           [_P, ctypes.c_size_t, _P])
_lib.moe_experts_backward_weights.argtypes = [_CFG] + [_P] * 9 + [_P, ctypes.c_size_t, _P]
_lib.moe_route_backward.argtypes = [_CFG] + [_P] * 13 + [_P, ctypes.c_size_t, _P]
_lib.moe_transpose_weights_fp8.restype = ctypes.c_int
_lib.moe_transpose_weights_fp8.argtypes = [_P, _P, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                                           _P, _P, _P]
_lib.moe_experts_backward_input_fp8.restype = ctypes.c_int
_lib.moe_experts_backward_input_fp8.argtypes = ([_CFG] + [_P] * 21 +
                                                [ctypes.c_int32, _P, ctypes.c_size_t, _P])
_lib.moe_quantize_act_fp8_128x1.restype = ctypes.c_int
_lib.moe_quantize_act_fp8_128x1.argtypes = [_P, ctypes.c_int32, ctypes.c_int32, _P, _P, _P]
_lib.moe_experts_grouped_train_fp8.restype = ctypes.c_int
_lib.moe_experts_grouped_train_fp8.argtypes = ([_CFG] + [_P] * 16 +
                                               [ctypes.c_size_t, _P, ctypes.c_size_t, _P])
_lib.moe_experts_backward_weights_fp8.restype = ctypes.c_int
_lib.moe_experts_backward_weights_fp8.argtypes = [_CFG] + [_P] * 11 + [_P, ctypes.c_size_t, _P]


def library():
    """The loaded ctypes handle of libmoe.so."""
    return _lib


@dataclass
class LayerCfg:
    """Shape of one layer (mirror of moe_cfg_t with readable names)."""
    T: int
    d: int
    E: int
    n_groups: int
    topk_groups: int
    k: int
    n_shared: int
    inter: int
    route_scale: float = 1.0
    gamma: float = 1e-3
    dtype: str = "bf16"
    group_score_topn: int = 2

    def c(self) -> MoeCfg:
        return MoeCfg(self.T, self.d, self.E, self.n_groups, self.topk_groups, self.k,
                      self.n_shared, self.inter, self.group_score_topn,
                      float(self.route_scale), float(self.gamma), _DTYPES[self.dtype])

    @classmethod
    def from_shape(cls, shape, **kw):
        """From a moe_synth.LayerShape (or anything with the same fields)."""
        c = cls(shape.T, shape.d, shape.E, shape.n_groups, shape.topk_groups, shape.k,
                shape.n_shared, shape.inter, shape.route_scale, shape.gamma, shape.dtype,
                shape.group_score_topn)
        for k, v in kw.items():
            setattr(c, k, v)
        return c


def _ptr(t, name, dtype=None, allow_none=False):
    if t is None:
        if allow_none:
            return None
        raise ValueError(f"{name} is required")
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be in CUDA device memory")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype not in (dtype if isinstance(dtype, tuple) else (dtype,)):
        raise ValueError(f"{name} has dtype {t.dtype}, expected {dtype}")
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _check(fn, status):
    if status != 0:
        raise MoeError(fn, status)


def _cfg(cfg):
    return ctypes.byref(cfg.c() if isinstance(cfg, LayerCfg) else cfg)


_X = (torch.float32, torch.bfloat16)
_F8 = (torch.float8_e4m3fn, torch.uint8)


def moe_check_cfg(cfg):
    return _lib.moe_check_cfg(_cfg(cfg))


def moe_workspace_bytes(cfg):
    return int(_lib.moe_workspace_bytes(_cfg(cfg)))


def moe_route(cfg, x, router_w, bias, topk_idx, topk_w, counts, offsets, row_of_slot,
              token_of_row, ws, affinity_in=None, affinity_out=None, stream=None):
    _check("moe_route", _lib.moe_route(
        _cfg(cfg), _ptr(x, "x", _X, allow_none=affinity_in is not None),
        _ptr(router_w, "router_w", torch.float32, allow_none=affinity_in is not None),
        _ptr(bias, "bias", torch.float32),
        _ptr(affinity_in, "affinity_in", torch.float32, allow_none=True),
        _ptr(affinity_out, "affinity_out", torch.float32, allow_none=True),
        _ptr(topk_idx, "topk_idx", torch.int32), _ptr(topk_w, "topk_w", torch.float32),
        _ptr(counts, "counts", torch.int32), _ptr(offsets, "offsets", torch.int32),
        _ptr(row_of_slot, "row_of_slot", torch.int32),
        _ptr(token_of_row, "token_of_row", torch.int32),
        _ptr(ws, "ws"), ws.numel() * ws.element_size(), _stream(stream)))


def moe_route_static_scratch(cfg, x, router_w, bias, topk_idx, topk_w, counts, offsets,
                             row_of_slot, token_of_row, affinity_in=None, affinity_out=None,
                             stream=None):
    """moe_route with the library's own fixed scratch array: no workspace
    argument and no allocation (see include/moe.h)."""
    _check("moe_route_static_scratch", _lib.moe_route_static_scratch(
        _cfg(cfg), _ptr(x, "x", _X, allow_none=affinity_in is not None),
        _ptr(router_w, "router_w", torch.float32, allow_none=affinity_in is not None),
        _ptr(bias, "bias", torch.float32),
        _ptr(affinity_in, "affinity_in", torch.float32, allow_none=True),
        _ptr(affinity_out, "affinity_out", torch.float32, allow_none=True),
        _ptr(topk_idx, "topk_idx", torch.int32), _ptr(topk_w, "topk_w", torch.float32),
        _ptr(counts, "counts", torch.int32), _ptr(offsets, "offsets", torch.int32),
        _ptr(row_of_slot, "row_of_slot", torch.int32),
        _ptr(token_of_row, "token_of_row", torch.int32), _stream(stream)))


def moe_permute(cfg, x, token_of_row, x_perm, x_perm_scales=None, x_q=None, x_q_scales=None,
                stream=None):
    _check("moe_permute", _lib.moe_permute(
        _cfg(cfg), _ptr(x, "x", _X), _ptr(token_of_row, "token_of_row", torch.int32),
        _ptr(x_perm, "x_perm", _X + _F8),
        _ptr(x_perm_scales, "x_perm_scales", torch.float32, allow_none=True),
        _ptr(x_q, "x_q", _F8, allow_none=True),
        _ptr(x_q_scales, "x_q_scales", torch.float32, allow_none=True), _stream(stream)))


def moe_experts_grouped(cfg, x_perm, x, offsets, w13, w2, ws13, ws2, y_perm, y_shared, ws,
                        x_perm_scales=None, x_scales=None, w13_scales=None, w2_scales=None,
                        ws13_scales=None, ws2_scales=None, stream=None):
    _check("moe_experts_grouped", _lib.moe_experts_grouped(
        _cfg(cfg), _ptr(x_perm, "x_perm", _X + _F8),
        _ptr(x_perm_scales, "x_perm_scales", torch.float32, allow_none=True),
        _ptr(x, "x", _X + _F8, allow_none=True),
        _ptr(x_scales, "x_scales", torch.float32, allow_none=True),
        _ptr(offsets, "offsets", torch.int32), _ptr(w13, "w13", _X + _F8),
        _ptr(w13_scales, "w13_scales", torch.float32, allow_none=True),
        _ptr(w2, "w2", _X + _F8), _ptr(w2_scales, "w2_scales", torch.float32, allow_none=True),
        _ptr(ws13, "ws13", _X + _F8, allow_none=True),
        _ptr(ws13_scales, "ws13_scales", torch.float32, allow_none=True),
        _ptr(ws2, "ws2", _X + _F8, allow_none=True),
        _ptr(ws2_scales, "ws2_scales", torch.float32, allow_none=True),
        _ptr(y_perm, "y_perm", _X), _ptr(y_shared, "y_shared", _X, allow_none=True),
        _ptr(ws, "ws"), ws.numel() * ws.element_size(), _stream(stream)))



def moe_experts_grouped_gated(cfg, x_perm, x, offsets, w13, w2, ws13, ws2, row_of_slot, topk_w,
                              y_perm, y_shared, ws,
                              x_perm_scales=None, x_scales=None, w13_scales=None, w2_scales=None,
                              ws13_scales=None, ws2_scales=None, stream=None):
    """moe_experts_grouped whose routed output rows carry their gates
    (y_perm[r] = g * FFN(u) for the copy r holds); combine them with
    ``moe_combine(..., topk_w=None, ...)``."""
    _check("moe_experts_grouped_gated", _lib.moe_experts_grouped_gated(
        _cfg(cfg), _ptr(x_perm, "x_perm", _X + _F8),
        _ptr(x_perm_scales, "x_perm_scales", torch.float32, allow_none=True),
        _ptr(x, "x", _X + _F8, allow_none=True),
        _ptr(x_scales, "x_scales", torch.float32, allow_none=True),
        _ptr(offsets, "offsets", torch.int32), _ptr(w13, "w13", _X + _F8),
        _ptr(w13_scales, "w13_scales", torch.float32, allow_none=True),
        _ptr(w2, "w2", _X + _F8), _ptr(w2_scales, "w2_scales", torch.float32, allow_none=True),
        _ptr(ws13, "ws13", _X + _F8, allow_none=True),
        _ptr(ws13_scales, "ws13_scales", torch.float32, allow_none=True),
        _ptr(ws2, "ws2", _X + _F8, allow_none=True),
        _ptr(ws2_scales, "ws2_scales", torch.float32, allow_none=True),
        _ptr(row_of_slot, "row_of_slot", torch.int32), _ptr(topk_w, "topk_w", torch.float32),
        _ptr(y_perm, "y_perm", _X), _ptr(y_shared, "y_shared", _X, allow_none=True),
        _ptr(ws, "ws"), ws.numel() * ws.element_size(), _stream(stream)))


def moe_experts_grouped_gather(cfg, x, token_of_row, offsets, w13, w2, ws13, ws2, y_perm,
                               y_shared, ws, x_scales=None, w13_scales=None, w2_scales=None,
                               ws13_scales=None, ws2_scales=None, stream=None):
    """moe_experts_grouped with the permute folded into the gate/up GEMM
    (routed A rows read from x by token_of_row)."""
    _check("moe_experts_grouped_gather", _lib.moe_experts_grouped_gather(
        _cfg(cfg), _ptr(x, "x", _X + _F8),
        _ptr(x_scales, "x_scales", torch.float32, allow_none=True),
        _ptr(token_of_row, "token_of_row", torch.int32), _ptr(offsets, "offsets", torch.int32),
        _ptr(w13, "w13", _X + _F8),
        _ptr(w13_scales, "w13_scales", torch.float32, allow_none=True),
        _ptr(w2, "w2", _X + _F8), _ptr(w2_scales, "w2_scales", torch.float32, allow_none=True),
        _ptr(ws13, "ws13", _X + _F8, allow_none=True),
        _ptr(ws13_scales, "ws13_scales", torch.float32, allow_none=True),
        _ptr(ws2, "ws2", _X + _F8, allow_none=True),
        _ptr(ws2_scales, "ws2_scales", torch.float32, allow_none=True),
        _ptr(y_perm, "y_perm", _X), _ptr(y_shared, "y_shared", _X, allow_none=True),
        _ptr(ws, "ws"), ws.numel() * ws.element_size(), _stream(stream)))


def moe_balance_stat(cfg, affinity, topk_idx, seq_len, f_out, p_out, loss_out, ws, alpha=1e-4,
                     stream=None):
    """Sequence-wise balance statistic alpha * sum_i f_i P_i per sequence."""
    _check("moe_balance_stat", _lib.moe_balance_stat(
        _cfg(cfg), _ptr(affinity, "affinity", torch.float32),
        _ptr(topk_idx, "topk_idx", torch.int32), int(seq_len), float(alpha),
        _ptr(f_out, "f_out", torch.float32), _ptr(p_out, "p_out", torch.float32),
        _ptr(loss_out, "loss_out", torch.float32), _ptr(ws, "ws"),
        ws.numel() * ws.element_size(), _stream(stream)))


def moe_combine(cfg, y_perm, y_shared, row_of_slot, topk_w, out, stream=None):
    """``topk_w=None``: y_perm holds the gated rows of moe_experts_grouped_gated."""
    _check("moe_combine", _lib.moe_combine(
        _cfg(cfg), _ptr(y_perm, "y_perm", _X), _ptr(y_shared, "y_shared", _X, allow_none=True),
        _ptr(row_of_slot, "row_of_slot", torch.int32),
        _ptr(topk_w, "topk_w", torch.float32, allow_none=True),
        _ptr(out, "out", _X), _stream(stream)))


def moe_bias_update(cfg, counts, bias, stream=None):
    _check("moe_bias_update", _lib.moe_bias_update(
        _cfg(cfg), _ptr(counts, "counts", torch.int32), _ptr(bias, "bias", torch.float32),
        _stream(stream)))


# ---------------------------------------------------------------- backward
_BF = torch.bfloat16


def moe_backward_workspace_bytes(cfg):
    return int(_lib.moe_backward_workspace_bytes(_cfg(cfg)))


def moe_combine_backward(cfg, dout, y_perm, row_of_slot, topk_w, dy_perm, dgate, stream=None):
    """dy_perm[row(t,k)] = g dout[t]; dgate[t,k] = dout[t] . y_perm[row(t,k)]."""
    _check("moe_combine_backward", _lib.moe_combine_backward(
        _cfg(cfg), _ptr(dout, "dout", _BF), _ptr(y_perm, "y_perm", _BF),
        _ptr(row_of_slot, "row_of_slot", torch.int32), _ptr(topk_w, "topk_w", torch.float32),
        _ptr(dy_perm, "dy_perm", _BF), _ptr(dgate, "dgate", torch.float32), _stream(stream)))


def moe_experts_grouped_train(cfg, x_perm, x, offsets, w13, w2, ws13, ws2, y_perm, y_shared,
                              ws, bws, stream=None):
    """moe_experts_grouped (bf16) that also keeps [a | b] in the backward
    workspace bws for moe_experts_backward_input(..., ab_kept=True)."""
    _check("moe_experts_grouped_train", _lib.moe_experts_grouped_train(
        _cfg(cfg), _ptr(x_perm, "x_perm", _BF), _ptr(x, "x", _BF, allow_none=True),
        _ptr(offsets, "offsets", torch.int32), _ptr(w13, "w13", _BF), _ptr(w2, "w2", _BF),
        _ptr(ws13, "ws13", _BF, allow_none=True), _ptr(ws2, "ws2", _BF, allow_none=True),
        _ptr(y_perm, "y_perm", _BF), _ptr(y_shared, "y_shared", _BF, allow_none=True),
        _ptr(ws, "ws"), ws.numel() * ws.element_size(),
        _ptr(bws, "bws"), bws.numel() * bws.element_size(), _stream(stream)))


def moe_experts_backward_input(cfg, x_perm, x, offsets, w13, w2, ws13, ws2, dy_perm, dout,
                               dx_perm, dx_shared, ws, ab_kept=False, stream=None):
    """Dgrad of the expert FFNs; leaves [da | db] and h in ws for the Wgrad.
    ab_kept: ws holds [a | b] from this step's moe_experts_grouped_train."""
    _check("moe_experts_backward_input", _lib.moe_experts_backward_input(
        _cfg(cfg), _ptr(x_perm, "x_perm", _BF), _ptr(x, "x", _BF, allow_none=True),
        _ptr(offsets, "offsets", torch.int32), _ptr(w13, "w13", _BF), _ptr(w2, "w2", _BF),
        _ptr(ws13, "ws13", _BF, allow_none=True), _ptr(ws2, "ws2", _BF, allow_none=True),
        _ptr(dy_perm, "dy_perm", _BF), _ptr(dout, "dout", _BF, allow_none=True),
        _ptr(dx_perm, "dx_perm", _BF), _ptr(dx_shared, "dx_shared", _BF, allow_none=True),
        1 if ab_kept else 0, _ptr(ws, "ws"), ws.numel() * ws.element_size(), _stream(stream)))


def moe_experts_backward_weights(cfg, x_perm, x, offsets, dy_perm, dout, dw13, dw2, dws13, dws2,
                                 ws, stream=None):
    """Wgrad of the expert FFNs from the intermediates the input call left in ws."""
    _check("moe_experts_backward_weights", _lib.moe_experts_backward_weights(
        _cfg(cfg), _ptr(x_perm, "x_perm", _BF), _ptr(x, "x", _BF, allow_none=True),
        _ptr(offsets, "offsets", torch.int32), _ptr(dy_perm, "dy_perm", _BF),
        _ptr(dout, "dout", _BF, allow_none=True), _ptr(dw13, "dw13", _BF),
        _ptr(dw2, "dw2", _BF), _ptr(dws13, "dws13", _BF, allow_none=True),
        _ptr(dws2, "dws2", _BF, allow_none=True),
        _ptr(ws, "ws"), ws.numel() * ws.element_size(), _stream(stream)))


def moe_route_backward(cfg, x, router_w, affinity, topk_idx, dgate, row_of_slot, token_of_row,
                       offsets, dx_perm, dx_shared, dlogit, dx, drouter_w, ws, stream=None):
    """Gates -> logits -> router weights and the layer input gradient."""
    _check("moe_route_backward", _lib.moe_route_backward(
        _cfg(cfg), _ptr(x, "x", _BF), _ptr(router_w, "router_w", torch.float32),
        _ptr(affinity, "affinity", torch.float32), _ptr(topk_idx, "topk_idx", torch.int32),
        _ptr(dgate, "dgate", torch.float32), _ptr(row_of_slot, "row_of_slot", torch.int32),
        _ptr(token_of_row, "token_of_row", torch.int32), _ptr(offsets, "offsets", torch.int32),
        _ptr(dx_perm, "dx_perm", _BF), _ptr(dx_shared, "dx_shared", _BF, allow_none=True),
        _ptr(dlogit, "dlogit", torch.float32), _ptr(dx, "dx", _BF),
        _ptr(drouter_w, "drouter_w", torch.float32),
        _ptr(ws, "ws"), ws.numel() * ws.element_size(), _stream(stream)))


def moe_transpose_weights_fp8(q, scales, qt, scales_t, stream=None):
    """E4M3 matrices [n, rows, cols] and their 128 x 128 block scales,
    transposed into ``qt`` [n, cols, rows] and ``scales_t``."""
    n, rows, cols = q.shape
    _check("moe_transpose_weights_fp8", _lib.moe_transpose_weights_fp8(
        _ptr(q, "q", _F8), _ptr(scales, "scales", torch.float32), n, rows, cols,
        _ptr(qt, "qt", _F8), _ptr(scales_t, "scales_t", torch.float32), _stream(stream)))


def moe_experts_backward_input_fp8(cfg, x_perm, x_perm_scales, x_q, x_q_scales, offsets, w13,
                                   w13_scales, w13t, w13t_scales, w2t, w2t_scales, ws13,
                                   ws13_scales, ws13t, ws13t_scales, ws2t, ws2t_scales, dy_perm,
                                   dout, dx_perm, dx_shared, ws, ab_kept=False, stream=None):
    """Dgrad of every expert FFN in FP8 (gradients in 1 x 128 tiles along
    their GEMM's contraction, weights in their forward blocks).
    ab_kept: ws holds [a | b] from this step's moe_experts_grouped_train_fp8."""
    opt = dict(allow_none=True)
    _check("moe_experts_backward_input_fp8", _lib.moe_experts_backward_input_fp8(
        _cfg(cfg), _ptr(x_perm, "x_perm", _F8), _ptr(x_perm_scales, "x_perm_scales", torch.float32),
        _ptr(x_q, "x_q", _F8, **opt), _ptr(x_q_scales, "x_q_scales", torch.float32, **opt),
        _ptr(offsets, "offsets", torch.int32),
        _ptr(w13, "w13", _F8), _ptr(w13_scales, "w13_scales", torch.float32),
        _ptr(w13t, "w13t", _F8), _ptr(w13t_scales, "w13t_scales", torch.float32),
        _ptr(w2t, "w2t", _F8), _ptr(w2t_scales, "w2t_scales", torch.float32),
        _ptr(ws13, "ws13", _F8, **opt), _ptr(ws13_scales, "ws13_scales", torch.float32, **opt),
        _ptr(ws13t, "ws13t", _F8, **opt), _ptr(ws13t_scales, "ws13t_scales", torch.float32, **opt),
        _ptr(ws2t, "ws2t", _F8, **opt), _ptr(ws2t_scales, "ws2t_scales", torch.float32, **opt),
        _ptr(dy_perm, "dy_perm", _BF), _ptr(dout, "dout", _BF, **opt),
        _ptr(dx_perm, "dx_perm", _BF), _ptr(dx_shared, "dx_shared", _BF, **opt),
        1 if ab_kept else 0, _ptr(ws, "ws"), ws.numel() * ws.element_size(), _stream(stream)))


def moe_quantize_act_fp8_128x1(x, q, scales, stream=None):
    """bf16 x [rows, cols] in 128 x 1 E4M3 tiles: codes q [ceil(rows/128)*128,
    cols] (float8_e4m3fn) and fp32 scales [ceil(rows/128), cols]."""
    rows, cols = x.shape
    _check("moe_quantize_act_fp8_128x1", _lib.moe_quantize_act_fp8_128x1(
        _ptr(x, "x", _BF), rows, cols, _ptr(q, "q", _F8), _ptr(scales, "scales", torch.float32),
        _stream(stream)))


def moe_experts_grouped_train_fp8(cfg, x_perm, x_perm_scales, x, x_scales, offsets, w13,
                                  w13_scales, w2, w2_scales, ws13, ws13_scales, ws2, ws2_scales,
                                  y_perm, y_shared, ws, bws, stream=None):
    """moe_experts_grouped (FP8) that also keeps [a | b] in the backward
    workspace bws for moe_experts_backward_input_fp8(..., ab_kept=True)."""
    opt = dict(allow_none=True)
    _check("moe_experts_grouped_train_fp8", _lib.moe_experts_grouped_train_fp8(
        _cfg(cfg), _ptr(x_perm, "x_perm", _F8), _ptr(x_perm_scales, "x_perm_scales", torch.float32),
        _ptr(x, "x", _F8, **opt), _ptr(x_scales, "x_scales", torch.float32, **opt),
        _ptr(offsets, "offsets", torch.int32),
        _ptr(w13, "w13", _F8), _ptr(w13_scales, "w13_scales", torch.float32),
        _ptr(w2, "w2", _F8), _ptr(w2_scales, "w2_scales", torch.float32),
        _ptr(ws13, "ws13", _F8, **opt), _ptr(ws13_scales, "ws13_scales", torch.float32, **opt),
        _ptr(ws2, "ws2", _F8, **opt), _ptr(ws2_scales, "ws2_scales", torch.float32, **opt),
        _ptr(y_perm, "y_perm", _BF), _ptr(y_shared, "y_shared", _BF, **opt),
        _ptr(ws, "ws"), ws.numel() * ws.element_size(),
        _ptr(bws, "bws"), bws.numel() * bws.element_size(), _stream(stream)))


def moe_experts_backward_weights_fp8(cfg, x_perm, x_perm_scales, x_q, x_q_scales, offsets,
                                     dy_perm, dout, dw13, dw2, dws13, dws2, ws, stream=None):
    """Wgrad of every expert FFN in FP8 (both operands in 128 x 1 tiles along
    the segment's rows), after moe_experts_backward_input_fp8 on ``ws``."""
    opt = dict(allow_none=True)
    _check("moe_experts_backward_weights_fp8", _lib.moe_experts_backward_weights_fp8(
        _cfg(cfg), _ptr(x_perm, "x_perm", _F8), _ptr(x_perm_scales, "x_perm_scales", torch.float32),
        _ptr(x_q, "x_q", _F8, **opt), _ptr(x_q_scales, "x_q_scales", torch.float32, **opt),
        _ptr(offsets, "offsets", torch.int32), _ptr(dy_perm, "dy_perm", _BF),
        _ptr(dout, "dout", _BF, **opt), _ptr(dw13, "dw13", _BF), _ptr(dw2, "dw2", _BF),
        _ptr(dws13, "dws13", _BF, **opt), _ptr(dws2, "dws2", _BF, **opt),
        _ptr(ws, "ws"), ws.numel() * ws.element_size(), _stream(stream)))


def moe_quantize_weights_fp8(w, q, scales, stream=None):
    """w [n, rows, cols] bf16 -> q [n, rows, cols] E4M3, scales [n, rows/128, cols/128]."""
    w3 = w if w.dim() == 3 else w.unsqueeze(0)
    _check("moe_quantize_weights_fp8", _lib.moe_quantize_weights_fp8(
        _ptr(w, "w", torch.bfloat16), w3.shape[0], w3.shape[1], w3.shape[2],
        _ptr(q, "q", _F8), _ptr(scales, "scales", torch.float32), _stream(stream)))


def moe_selftest_wait(limit_ns, stream=None):
    """Failure-detection self test: a bounded device wait that must give up
    after limit_ns and set the timeout bit of the error word."""
    _check("moe_selftest_wait", _lib.moe_selftest_wait(int(limit_ns), _stream(stream)))


def moe_get_device_error(stream=None):
    """Synchronises the stream and returns (and clears) the device error status."""
    return _lib.moe_get_device_error(_stream(stream))


from .layer import MoELayer  # noqa: E402,F401
