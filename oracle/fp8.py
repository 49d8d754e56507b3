"""FP8 E4M3 fine-grained quantisation, written out from its definition
(test infrastructure only).

Source: "DeepSeek-V3 Technical Report", fine-grained quantisation paragraph
and Appendix B.2 (block-wise quantisation): activations are grouped in
1 x N_c tiles, weights in N_c x N_c blocks, N_c = 128, each group with its
own scale; the increased-precision accumulation paragraph keeps the sums
in FP32 and applies the scales there.

The page gives no scale formula.  The reading used here:
  scale = fl32(amax / 448)  (scale = 1 when the group is all zeros),
  code  = E4M3(fl32(v / scale)) with round-to-nearest-even and saturation
          to +-448 (the "satfinite" convention of the E4M3FN format),
  value = code * scale.
Scales are plain fp32 numbers (not powers of two).

E4M3FN: 1 sign bit, 4 exponent bits (bias 7), 3 mantissa bits; no
infinities; the largest finite magnitude is 1.75 * 2^8 = 448; the smallest
normal is 2^-6; subnormals are m/8 * 2^-6.
"""

from __future__ import annotations

import numpy as np

E4M3_MAX = 448.0
N_C = 128


def e4m3_round(v):
    """Round fp64 values to the nearest E4M3FN value (ties to even),
    saturating to +-448.  Returns fp64 values on the E4M3 grid."""
    v = np.asarray(v, dtype=np.float64)
    a = np.abs(v)
    _, ex = np.frexp(a)                      # a = m * 2^ex, 0.5 <= m < 1
    e = np.maximum(ex - 1, -6)               # exponent of the leading bit
    quantum = np.ldexp(1.0, e - 3)           # spacing of 3 mantissa bits
    q = np.rint(a / quantum) * quantum       # np.rint rounds half to even
    q = np.where(a == 0, 0.0, q)
    q = np.minimum(q, E4M3_MAX)
    return np.copysign(q, v)


def e4m3_decode(codes):
    """Value of each 8-bit E4M3FN code (0x7F / 0xFF decode to NaN)."""
    c = np.asarray(codes, dtype=np.int64) & 0xFF
    sign = np.where(c & 0x80, -1.0, 1.0)
    exp = (c >> 3) & 0xF
    man = c & 0x7
    val = np.where(exp == 0,
                   np.ldexp(man / 8.0, -6),
                   np.ldexp(1.0 + man / 8.0, exp - 7))
    val = np.where((exp == 0xF) & (man == 0x7), np.nan, val)
    return sign * val


def e4m3_encode(v):
    """8-bit E4M3FN code of values already on the grid (see e4m3_round)."""
    v = np.asarray(v, dtype=np.float64)
    a = np.abs(v)
    _, ex = np.frexp(a)
    e = ex - 1
    normal = (a >= 2.0 ** -6)
    exp_field = np.where(normal, e + 7, 0)
    man = np.where(normal, np.rint((a / np.ldexp(1.0, e) - 1.0) * 8.0),
                   np.rint(a / 2.0 ** -9))
    code = (exp_field.astype(np.int64) << 3) | man.astype(np.int64)
    code = np.where(a == 0, 0, code)
    return (code | np.where(np.signbit(v), 0x80, 0)).astype(np.uint8)


def _scale_of(amax32):
    """fl32(amax / 448), or 1 for an all-zero group."""
    amax32 = np.asarray(amax32, dtype=np.float32)
    s = (amax32 / np.float32(E4M3_MAX)).astype(np.float32)
    return np.where(amax32 == 0, np.float32(1.0), s).astype(np.float32)


def _quantize_group(vals32, scale32):
    """E4M3(fl32(v / scale)) as fp64 grid values."""
    ratio = (np.asarray(vals32, np.float32) / np.float32(scale32)).astype(np.float32)
    return e4m3_round(ratio.astype(np.float64))


def quantize_act_1x128(x):
    """Quantise activations [rows, K] in 1 x 128 tiles along K.

    Returns (q, scale): q fp64 grid values [rows, K]; scale float32
    [rows, K/128].  Values are first taken as float32."""
    x32 = np.asarray(x, dtype=np.float32)
    rows, K = x32.shape
    assert K % N_C == 0
    q = np.zeros((rows, K), dtype=np.float64)
    scale = np.zeros((rows, K // N_C), dtype=np.float32)
    for r in range(rows):
        for kb in range(K // N_C):
            tile = x32[r, kb * N_C:(kb + 1) * N_C]
            sc = _scale_of(np.max(np.abs(tile)))
            scale[r, kb] = sc
            q[r, kb * N_C:(kb + 1) * N_C] = _quantize_group(tile, sc)
    return q, scale


def quantize_weight_128x128(w):
    """Quantise a weight matrix [N, K] in 128 x 128 blocks.

    Returns (q, scale): q fp64 grid values [N, K]; scale float32
    [ceil(N/128), K/128].  A ragged last row-block is scaled over the rows
    it has."""
    w32 = np.asarray(w, dtype=np.float32)
    N, K = w32.shape
    assert K % N_C == 0
    nb = (N + N_C - 1) // N_C
    q = np.zeros((N, K), dtype=np.float64)
    scale = np.zeros((nb, K // N_C), dtype=np.float32)
    for i in range(nb):
        for kb in range(K // N_C):
            blk = w32[i * N_C:(i + 1) * N_C, kb * N_C:(kb + 1) * N_C]
            sc = _scale_of(np.max(np.abs(blk)))
            scale[i, kb] = sc
            q[i * N_C:(i + 1) * N_C, kb * N_C:(kb + 1) * N_C] = _quantize_group(blk, sc)
    return q, scale


def dequantize_act_1x128(q, scale):
    """q * scale per 1 x 128 tile, in fp64."""
    return np.asarray(q, np.float64) * np.repeat(np.asarray(scale, np.float64), N_C, axis=1)


def dequantize_weight_128x128(q, scale):
    """q * scale per 128 x 128 block, in fp64."""
    q = np.asarray(q, np.float64)
    s = np.repeat(np.repeat(np.asarray(scale, np.float64), N_C, axis=0), N_C, axis=1)
    return q * s[:q.shape[0], :q.shape[1]]


def fp8_linear(qa, sa, qw, sw):
    """y = dequant(a) @ dequant(w)^T in fp64.

    The device sums each 128-wide K block in the tensor core, scales the
    partial by sa * sw and accumulates in fp32 (increased-precision
    accumulation paragraph); in fp64 that is the same sum up to rounding, so
    the plain definition is the dequantised product."""
    return dequantize_act_1x128(qa, sa) @ dequantize_weight_128x128(qw, sw).T
