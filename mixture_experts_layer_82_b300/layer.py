"""One DeepSeekMoE layer: the buffers of a batch and the five library calls
of a forward step (route -> permute -> experts -> combine -> bias update),
enqueued on one stream with no host synchronisation; for the bf16 kind also
the four calls of its backward pass."""

from __future__ import annotations

import torch

from .replicas import global_cfg, global_load
from . import (LayerCfg, moe_route, moe_permute, moe_experts_grouped, moe_experts_grouped_gather,
               moe_experts_grouped_gated,
               moe_combine, moe_bias_update, moe_quantize_weights_fp8, moe_workspace_bytes,
               moe_backward_workspace_bytes, moe_combine_backward, moe_experts_backward_input,
               moe_experts_backward_weights, moe_route_backward, moe_experts_grouped_train,
               moe_transpose_weights_fp8, moe_experts_backward_input_fp8,
               moe_experts_backward_weights_fp8, moe_experts_grouped_train_fp8)


def _transpose_fp8(q, s, stream=None):
    n, rows, cols = q.shape
    qt = torch.empty(n, cols, rows, dtype=q.dtype, device=q.device)
    st = torch.empty(n, cols // 128, rows // 128, dtype=torch.float32, device=q.device)
    moe_transpose_weights_fp8(q, s, qt, st, stream=stream)
    return qt, st


def _quantize(w, stream=None):
    n, rows, cols = w.shape
    q = torch.empty(n, rows, cols, dtype=torch.float8_e4m3fn, device=w.device)
    s = torch.empty(n, (rows + 127) // 128, cols // 128, dtype=torch.float32, device=w.device)
    moe_quantize_weights_fp8(w, q, s, stream=stream)
    return q, s


class MoELayer:
    """Weights and per-batch buffers of one layer on one device.

    ``router_w`` [E, d] fp32, ``bias`` [E] fp32 (updated in place by
    ``forward`` unless ``update_bias=False``), ``w13`` [E, 2I, d],
    ``w2`` [E, d, I], ``ws13``/``ws2`` the shared experts; master weights
    in bf16 (fp32 for the fp32 kind).  For the fp8 kind the expert weights
    are quantised once here (128 x 128 blocks)."""

    def __init__(self, cfg: LayerCfg, router_w, bias, w13, w2, ws13=None, ws2=None,
                 gather=False):
        self.cfg = cfg
        self.gather = gather
        dev = router_w.device
        self.router_w, self.bias = router_w, bias
        T, d, E, K, I, ns = cfg.T, cfg.d, cfg.E, cfg.k, cfg.inter, cfg.n_shared
        if cfg.dtype == "fp8":
            self.w13, self.w13_s = _quantize(w13)
            self.w2, self.w2_s = _quantize(w2)
            if ns:
                self.ws13, self.ws13_s = _quantize(ws13)
                self.ws2, self.ws2_s = _quantize(ws2)
            else:
                self.ws13 = self.ws13_s = self.ws2 = self.ws2_s = None
        else:
            self.w13, self.w2, self.ws13, self.ws2 = w13, w2, ws13, ws2
            self.w13_s = self.w2_s = self.ws13_s = self.ws2_s = None
        act = torch.float32 if cfg.dtype == "fp32" else torch.bfloat16
        i32 = dict(dtype=torch.int32, device=dev)
        self.topk_idx = torch.empty(T, K, **i32)
        self.topk_w = torch.empty(T, K, dtype=torch.float32, device=dev)
        self.counts = torch.empty(E, **i32)
        self.offsets = torch.empty(E + 1, **i32)
        self.row_of_slot = torch.empty(T, K, **i32)
        self.token_of_row = torch.empty(T * K, **i32)
        if cfg.dtype == "fp8":
            self.x_perm = torch.empty(T * K, d, dtype=torch.float8_e4m3fn, device=dev)
            self.x_perm_s = torch.empty(T * K, d // 128, dtype=torch.float32, device=dev)
            self.x_q = torch.empty(T, d, dtype=torch.float8_e4m3fn, device=dev)
            self.x_q_s = torch.empty(T, d // 128, dtype=torch.float32, device=dev)
        else:
            self.x_perm = torch.empty(T * K, d, dtype=act, device=dev)
            self.x_perm_s = self.x_q = self.x_q_s = None
        self.y_perm = torch.empty(T * K, d, dtype=act, device=dev)
        self.y_shared = torch.empty(T, d, dtype=act, device=dev) if ns else None
        self.out = torch.empty(T, d, dtype=act, device=dev)
        self.ws = torch.empty(moe_workspace_bytes(cfg), dtype=torch.uint8, device=dev)

    def forward(self, x, stream=None, update_bias=True, affinity_out=None, affinity_in=None,
                expert_events=None, gather=None, out=None, keep=False, load_group=None,
                gated=False):
        """One forward step on ``x`` [T, d]; returns the layer output, written
        to ``out`` when given (else to the layer's own buffer).
        ``expert_events`` (a pair of torch.cuda.Event) are recorded on
        ``stream`` around the grouped expert GEMMs, for timing them inside a
        step.  ``gather`` (default: ``self.gather``) folds the permute into
        the gate/up GEMM (moe_experts_grouped_gather; bf16 kind).  ``keep``
        (bf16 and fp8 kinds, permuting forward): keep the gate/up products
        for the next ``backward`` instead of having it recompute them.
        ``load_group``: a torch.distributed group of data-parallel replicas;
        the bias update then uses the whole batch's per-expert loads (one
        all-reduce of ``counts``, which afterwards hold the global loads).
        ``gated`` (permuting forward without ``keep``): the down projection
        multiplies each routed row by its gate (moe_experts_grouped_gated)
        and the combine only adds rows; ``y_perm`` then holds the gated
        rows."""
        c = self.cfg
        out = self.out if out is None else out
        gather = self.gather if gather is None else gather
        keep = keep and c.dtype in ("bf16", "fp8") and not gather
        gated = gated and not gather and not keep
        if keep and not hasattr(self, "bws"):
            self._grad_buffers()
        self._ab_kept = False
        moe_route(c, x, self.router_w, self.bias, self.topk_idx, self.topk_w, self.counts,
                  self.offsets, self.row_of_slot, self.token_of_row, self.ws,
                  affinity_in=affinity_in, affinity_out=affinity_out, stream=stream)
        if gather:
            if expert_events is not None:
                expert_events[0].record(stream)
            moe_experts_grouped_gather(c, x, self.token_of_row, self.offsets, self.w13, self.w2,
                                       self.ws13, self.ws2, self.y_perm, self.y_shared, self.ws,
                                       stream=stream)
        else:
            moe_permute(c, x, self.token_of_row, self.x_perm, self.x_perm_s, self.x_q,
                        self.x_q_s, stream=stream)
            shared_in = self.x_q if c.dtype == "fp8" else x
            if expert_events is not None:
                expert_events[0].record(stream)
            if keep and c.dtype == "fp8":
                moe_experts_grouped_train_fp8(c, self.x_perm, self.x_perm_s, self.x_q, self.x_q_s,
                                              self.offsets, self.w13, self.w13_s, self.w2,
                                              self.w2_s, self.ws13, self.ws13_s, self.ws2,
                                              self.ws2_s, self.y_perm, self.y_shared, self.ws,
                                              self.bws, stream=stream)
                self._ab_kept = True
            elif keep:
                moe_experts_grouped_train(c, self.x_perm, x, self.offsets, self.w13, self.w2,
                                          self.ws13, self.ws2, self.y_perm, self.y_shared, self.ws,
                                          self.bws, stream=stream)
                self._ab_kept = True
            elif gated:
                moe_experts_grouped_gated(c, self.x_perm, shared_in, self.offsets, self.w13,
                                          self.w2, self.ws13, self.ws2, self.row_of_slot,
                                          self.topk_w, self.y_perm, self.y_shared, self.ws,
                                          x_perm_scales=self.x_perm_s, x_scales=self.x_q_s,
                                          w13_scales=self.w13_s, w2_scales=self.w2_s,
                                          ws13_scales=self.ws13_s, ws2_scales=self.ws2_s,
                                          stream=stream)
            else:
                moe_experts_grouped(c, self.x_perm, shared_in, self.offsets, self.w13, self.w2,
                                    self.ws13, self.ws2, self.y_perm, self.y_shared, self.ws,
                                    x_perm_scales=self.x_perm_s, x_scales=self.x_q_s,
                                    w13_scales=self.w13_s, w2_scales=self.w2_s,
                                    ws13_scales=self.ws13_s, ws2_scales=self.ws2_s, stream=stream)
        if expert_events is not None:
            expert_events[1].record(stream)
        moe_combine(c, self.y_perm, self.y_shared, self.row_of_slot,
                    None if gated else self.topk_w, out, stream=stream)
        if update_bias:
            if load_group is not None:
                world = global_load(self.counts, load_group, stream=stream)
                moe_bias_update(global_cfg(c, world), self.counts, self.bias, stream=stream)
            else:
                moe_bias_update(c, self.counts, self.bias, stream=stream)
        return out

    # ------------------------------------------------------------- backward
    def _grad_buffers(self):
        c = self.cfg
        dev = self.router_w.device
        T, d, E, K, I, ns = c.T, c.d, c.E, c.k, c.inter, c.n_shared
        bf = dict(dtype=torch.bfloat16, device=dev)
        f32 = dict(dtype=torch.float32, device=dev)
        if c.dtype == "fp8":
            # Dgrad reads the weights contracted over their other dimension:
            # transposed copies of the forward's codes and blocks
            self.w13t, self.w13t_s = _transpose_fp8(self.w13, self.w13_s)
            self.w2t, self.w2t_s = _transpose_fp8(self.w2, self.w2_s)
            if ns:
                self.ws13t, self.ws13t_s = _transpose_fp8(self.ws13, self.ws13_s)
                self.ws2t, self.ws2t_s = _transpose_fp8(self.ws2, self.ws2_s)
            else:
                self.ws13t = self.ws13t_s = self.ws2t = self.ws2t_s = None
        self.dy_perm = torch.empty(T * K, d, **bf)
        self.dgate = torch.empty(T, K, **f32)
        self.dx_perm = torch.empty(T * K, d, **bf)
        self.dx_shared = torch.empty(T, d, **bf) if ns else None
        self.dlogit = torch.empty(T, K, **f32)
        self.dx = torch.empty(T, d, **bf)
        self.drouter_w = torch.empty(E, d, **f32)
        self.dw13 = torch.empty(E, 2 * I, d, **bf)
        self.dw2 = torch.empty(E, d, I, **bf)
        self.dws13 = torch.empty(ns, 2 * I, d, **bf) if ns else None
        self.dws2 = torch.empty(ns, d, I, **bf) if ns else None
        self.bws = torch.empty(moe_backward_workspace_bytes(c), dtype=torch.uint8, device=dev)

    def backward(self, x, dout, affinity, stream=None, weights=True, events=None):
        """Backward of the last ``forward(x, affinity_out=affinity)`` (bf16
        kind; with ``keep=True`` there, the gate/up products are not
        recomputed), given ``dout`` = dL/dy [T, d] bf16.  Fills ``dx``,
        ``drouter_w`` and, with ``weights``, ``dw13``, ``dw2``, ``dws13``,
        ``dws2`` (plus the intermediates ``dy_perm``, ``dgate``, ``dlogit``,
        ``dx_perm``, ``dx_shared``); returns ``dx``.  The selection and the
        bias are those of the forward; the bias gets no gradient.
        ``events`` (four torch.cuda.Event) are recorded on ``stream`` around
        the expert Dgrad call and around the expert Wgrad call.

        FP8 kind: the expert Dgrad and Wgrad GEMMs run in FP8 on the
        forward's codes (moe_experts_backward_input_fp8,
        moe_experts_backward_weights_fp8); at most one shared expert."""
        c = self.cfg
        if c.dtype not in ("bf16", "fp8"):
            raise ValueError("the backward pass is implemented for the bf16 and fp8 kinds")
        if not hasattr(self, "bws"):
            self._grad_buffers()
        if c.dtype == "fp8":
            moe_combine_backward(c, dout, self.y_perm, self.row_of_slot, self.topk_w,
                                 self.dy_perm, self.dgate, stream=stream)
            if events is not None:
                events[0].record(stream)
            moe_experts_backward_input_fp8(
                c, self.x_perm, self.x_perm_s, self.x_q, self.x_q_s, self.offsets, self.w13,
                self.w13_s, self.w13t, self.w13t_s, self.w2t, self.w2t_s, self.ws13, self.ws13_s,
                self.ws13t, self.ws13t_s, self.ws2t, self.ws2t_s, self.dy_perm, dout,
                self.dx_perm, self.dx_shared, self.bws,
                ab_kept=getattr(self, "_ab_kept", False), stream=stream)
            self._ab_kept = False  # a later backward without a new forward recomputes it
            if events is not None:
                events[1].record(stream)
            moe_route_backward(c, x, self.router_w, affinity, self.topk_idx, self.dgate,
                               self.row_of_slot, self.token_of_row, self.offsets, self.dx_perm,
                               self.dx_shared, self.dlogit, self.dx, self.drouter_w, self.bws,
                               stream=stream)
            if weights:
                if events is not None:
                    events[2].record(stream)
                moe_experts_backward_weights_fp8(
                    c, self.x_perm, self.x_perm_s, self.x_q, self.x_q_s, self.offsets,
                    self.dy_perm, dout, self.dw13, self.dw2, self.dws13, self.dws2, self.bws,
                    stream=stream)
                if events is not None:
                    events[3].record(stream)
            return self.dx
        if self.gather:
            # the gathering forward never wrote the permuted rows
            moe_permute(c, x, self.token_of_row, self.x_perm, stream=stream)
        moe_combine_backward(c, dout, self.y_perm, self.row_of_slot, self.topk_w, self.dy_perm,
                             self.dgate, stream=stream)
        if events is not None:
            events[0].record(stream)
        moe_experts_backward_input(c, self.x_perm, x, self.offsets, self.w13, self.w2, self.ws13,
                                   self.ws2, self.dy_perm, dout, self.dx_perm, self.dx_shared,
                                   self.bws, ab_kept=getattr(self, "_ab_kept", False),
                                   stream=stream)
        self._ab_kept = False  # consumed: [da | db] now lies over it
        if events is not None:
            events[1].record(stream)
        moe_route_backward(c, x, self.router_w, affinity, self.topk_idx, self.dgate,
                           self.row_of_slot, self.token_of_row, self.offsets, self.dx_perm,
                           self.dx_shared, self.dlogit, self.dx, self.drouter_w, self.bws,
                           stream=stream)
        if weights:
            if events is not None:
                events[2].record(stream)
            moe_experts_backward_weights(c, self.x_perm, x, self.offsets, self.dy_perm, dout,
                                         self.dw13, self.dw2, self.dws13, self.dws2, self.bws,
                                         stream=stream)
            if events is not None:
                events[3].record(stream)
        return self.dx
