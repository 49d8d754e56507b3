"""fp64 oracle of the FP8 variant of the DeepSeekMoE layer forward
(test infrastructure only).

Source: "DeepSeek-V3 Technical Report": mixed-precision framework paragraph
(GEMMs in FP8, MoE gating kept in higher precision), fine-grained
quantisation paragraph (activations dispatched in FP8, 1 x 128 tiles;
weights in 128 x 128 blocks) and Appendix B.2.

Readings: the router and the combine run exactly as in the bf16 layer; the
token rows are quantised once per token before dispatch; the SwiGLU output
h is rounded to fp32 and re-quantised in 1 x 128 tiles along the
intermediate dimension before the down projection; expert weights are
quantised from their bf16 values per expert.  Sums are fp64.
"""

from __future__ import annotations

import numpy as np

from .fp8 import quantize_act_1x128, quantize_weight_128x128, fp8_linear
from .moe_oracle import (sigmoid_affinity, select_experts, gating_weights,
                         segment_layout, silu, combine)


def fp8_swiglu_ffn(qx, sx, w13, w2):
    """One expert FFN with FP8 operands: gate/up and down projections on
    block-quantised weights; h quantised in 1 x 128 tiles between them."""
    qw13, sw13 = quantize_weight_128x128(w13)
    qw2, sw2 = quantize_weight_128x128(w2)
    inter = np.asarray(w13).shape[0] // 2
    ab = fp8_linear(qx, sx, qw13, sw13)
    h = silu(ab[:, :inter]) * ab[:, inter:]
    qh, sh = quantize_act_1x128(h.astype(np.float32))
    return fp8_linear(qh, sh, qw2, sw2)


def moe_layer_forward_fp8(x, router_w, bias, w13, w2, ws13, ws2, *, n_groups,
                          topk_groups, k, route_scale=1.0, group_score_topn=2,
                          affinity32=None):
    """FP8 forward of one DeepSeekMoE layer.

    Arguments as in ``moe_layer_forward``; the weights are the bf16 master
    weights, quantised here.  Returns the output and the routing, plus the
    activation codes/scales of x so that a device's quantiser can be
    compared bit for bit."""
    x64 = np.asarray(x, dtype=np.float64)
    T, d = x64.shape
    E = np.asarray(router_w).shape[0]
    s64 = sigmoid_affinity(x64, router_w)
    s_sel = s64.astype(np.float32) if affinity32 is None else np.asarray(affinity32, np.float32)
    idx = select_experts(s_sel, bias, n_groups, topk_groups, k, group_score_topn)
    gates = gating_weights(s_sel, idx, route_scale)
    counts, offsets, row_of_slot, token_of_row = segment_layout(idx, E)
    qx, sx = quantize_act_1x128(x64.astype(np.float32))
    y_perm = np.zeros((T * k, d), dtype=np.float64)
    for e in range(E):
        lo, hi = int(offsets[e]), int(offsets[e + 1])
        if hi > lo:
            rows = token_of_row[lo:hi]
            y_perm[lo:hi] = fp8_swiglu_ffn(qx[rows], sx[rows], w13[e], w2[e])
    y_shared = None
    n_shared = 0 if ws13 is None else len(ws13)
    if n_shared:
        y_shared = np.zeros((T, d), dtype=np.float64)
        for s in range(n_shared):
            y_shared += fp8_swiglu_ffn(qx, sx, ws13[s], ws2[s])
    out = combine(y_shared, y_perm, row_of_slot, gates)
    return {"affinity": s64, "topk_idx": idx, "topk_w": gates,
            "counts": counts, "offsets": offsets, "row_of_slot": row_of_slot,
            "token_of_row": token_of_row, "x_q": qx, "x_scale": sx,
            "y_perm": y_perm, "y_shared": y_shared, "out": out}


def moe_layer_tokens_fp8(x_rows, idx_rows, gates_rows, w13, w2, ws13, ws2):
    """FP8 layer output for a few tokens whose routing is already known."""
    x64 = np.asarray(x_rows, dtype=np.float64)
    n, d = x64.shape
    qx, sx = quantize_act_1x128(x64.astype(np.float32))
    out = np.zeros((n, d), dtype=np.float64)
    n_shared = 0 if ws13 is None else len(ws13)
    for s in range(n_shared):
        out += fp8_swiglu_ffn(qx, sx, ws13[s], ws2[s])
    idx_rows = np.asarray(idx_rows)
    for e in sorted(set(int(v) for v in idx_rows.reshape(-1))):
        rows, cols = np.nonzero(idx_rows == e)
        y = fp8_swiglu_ffn(qx[rows], sx[rows], w13[e], w2[e])
        out[rows] += np.asarray(gates_rows, np.float64)[rows, cols][:, None] * y
    return out
