"""fp64 oracle of the FP8 expert backward (test infrastructure only): the
Dgrad and Wgrad GEMMs of the mixed precision framework in FP8.

Source: "DeepSeek-V3 Technical Report", mixed precision framework paragraph
(Figure 6): Fprop, Dgrad and Wgrad of every linear run in FP8 with BF16 /
FP32 outputs; fine-grained quantisation paragraph: activations in 1 x N_c
tiles, weights in N_c x N_c blocks (N_c = 128), fp32 scales; activations
cached in FP8 for the backward.

The pages do not say along which dimension a backward operand's tiles run.
Reading used here (listed with the other readings of the design notes):
a scale can only be factored out of a dot product if it is constant along
the contraction, so every activation-like operand is tiled along its GEMM's
contraction dimension:
  * Dgrad (dh = dy W2, dx = [da | db] W13): the gradient rows are quantised
    in 1 x 128 tiles along their columns (the contraction over d or 2I); the
    weights keep their forward 128 x 128 blocks, which a square block allows
    in either orientation.
  * Wgrad (dW2 = dy^T h, dW13 = [da | db]^T u): the contraction is over the
    token rows of a segment, so both operands are quantised in 128 x 1 tiles
    (128 consecutive rows of one column); a segment's last tile holds the
    rows that are left.
  * a, b are the FP8 forward's products (dequantised sums in fp64), h =
    silu(a) b and da, db are formed in fp64; results are fp64.
Scales follow the forward's rule: fl32(amax / 448), 1 for an all-zero tile;
codes E4M3(fl32(v / scale)), nearest-even, saturating.
"""

from __future__ import annotations

import numpy as np

from .fp8 import (N_C, dequantize_act_1x128, dequantize_weight_128x128, fp8_linear,
                  quantize_act_1x128, quantize_weight_128x128)
from .moe_oracle import silu


def quantize_act_128x1(x):
    """Quantise activations [rows, K] in 128 x 1 tiles (128 consecutive rows
    of one column).  Returns (q, scale): q fp64 grid values [rows, K]; scale
    float32 [ceil(rows/128), K].  A ragged last tile is scaled over the rows
    it has (the missing rows count as zeros, which do not change amax)."""
    x32 = np.asarray(x, dtype=np.float32)
    rows, K = x32.shape
    nb = (rows + N_C - 1) // N_C
    padded = np.zeros((nb * N_C, K), dtype=np.float32)
    padded[:rows] = x32
    # a 128 x 1 tile of x is a 1 x 128 tile of x^T
    qt, st = quantize_act_1x128(padded.T)
    return qt.T[:rows].copy(), st.T.copy()


def dequantize_act_128x1(q, scale):
    """q * scale per 128 x 1 tile, in fp64."""
    q = np.asarray(q, np.float64)
    s = np.repeat(np.asarray(scale, np.float64), N_C, axis=0)
    return q * s[:q.shape[0]]


def fp8_dgrad(qg, sg, qw, sw):
    """dX = dequant(g) @ dequant(w) in fp64: g [n, K] in 1 x 128 tiles along
    K, w [K, N] in its 128 x 128 blocks (the forward's weight, contracted
    over its rows)."""
    return dequantize_act_1x128(qg, sg) @ dequantize_weight_128x128(qw, sw)


def fp8_wgrad(qa, sa, qb, sb):
    """dW = dequant(a)^T @ dequant(b) in fp64: a [n, M] and b [n, N] both in
    128 x 1 tiles along the n token rows they are contracted over."""
    return dequantize_act_128x1(qa, sa).T @ dequantize_act_128x1(qb, sb)


def fp8_swiglu_ffn_backward(qx, sx, w13, w2, dy):
    """Gradients of one FP8 SwiGLU expert on the rows whose forward codes
    are ``qx``, ``sx`` (1 x 128 tiles), given ``dy`` [n, d].  ``w13``
    [2I, d] and ``w2`` [d, I] are the bf16 master weights (quantised here in
    128 x 128 blocks, as the forward does).  Returns a dict with ``du``
    [n, d], ``dw13`` [2I, d], ``dw2`` [d, I] and the fp64 intermediates."""
    qw13, sw13 = quantize_weight_128x128(w13)
    qw2, sw2 = quantize_weight_128x128(w2)
    inter = np.asarray(w13).shape[0] // 2
    ab = fp8_linear(qx, sx, qw13, sw13)
    a, b = ab[:, :inter], ab[:, inter:]
    sig = 1.0 / (1.0 + np.exp(-np.clip(a, -700.0, 700.0)))
    h = silu(a) * b
    # Dgrad of the down projection: dh = dy W2
    qg, sg = quantize_act_1x128(np.asarray(dy, np.float64).astype(np.float32))
    dh = fp8_dgrad(qg, sg, qw2, sw2)
    da = dh * b * (sig * (1.0 + a * (1.0 - sig)))
    db = dh * silu(a)
    dab = np.concatenate([da, db], axis=1)
    # Dgrad of the gate/up projection: du = [da | db] W13
    qd, sd = quantize_act_1x128(dab.astype(np.float32))
    du = fp8_dgrad(qd, sd, qw13, sw13)
    # Wgrad: dW2 = dy^T h, dW13 = [da | db]^T u over the rows
    qy, sy = quantize_act_128x1(np.asarray(dy, np.float64).astype(np.float32))
    qh, sh = quantize_act_128x1(h.astype(np.float32))
    dw2 = fp8_wgrad(qy, sy, qh, sh)
    u = dequantize_act_1x128(qx, sx)
    qdt, sdt = quantize_act_128x1(dab.astype(np.float32))
    qu, su = quantize_act_128x1(u.astype(np.float32))
    dw13 = fp8_wgrad(qdt, sdt, qu, su)
    return {"du": du, "dw13": dw13, "dw2": dw2, "a": a, "b": b, "h": h, "dh": dh,
            "da": da, "db": db}
