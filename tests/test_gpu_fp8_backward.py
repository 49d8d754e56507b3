"""Parity of the FP8 backward (moe_experts_backward_input_fp8 and
moe_experts_backward_weights_fp8, through the C ABI) with the FP8 backward
oracle.

Mixed precision framework paragraph (Dgrad in FP8); fine-grained
quantisation paragraph: the gradients are quantised in 1 x 128 tiles along
the contraction of their GEMM and the weights keep their forward 128 x 128
blocks.  The device and the oracle quantise dy from the same bf16 values
(codes equal).  [a | b] and dh are rounded to bf16 on the device (relative
2^-9 each) and kept in fp64 by the oracle, so some E4M3 codes of
q([da | db]) fall on the other side of a rounding midpoint; each such code
moves its term by one E4M3 step (2^-3 of its size).  With a fraction p of
the 2I terms of a row flipped, the row's relative error is about
sqrt(p) 2^-3: 2.8% at p = 5%.  The whole tensor must stay within the FP8
bound 3e-2 (relative Frobenius); each row within 6e-2, twice that, for the
rows in the tail of that distribution.

Wgrad: both operands are quantised in 128 x 1 tiles along the segment's
rows.  dy and u (the dequantised forward codes) give equal codes on both
sides; h and [da | db] come from the bf16 [a | b] and dh on the device, so
some of their codes flip as above.  A row of dW sums over the segment's
rows; in a short segment one term can carry most of it, and a flip of that
code moves the row by up to one E4M3 step (2^-3 of the term), so a row
bound does not fit.  Each element is held instead to the bound that follows
from the operands: dW = A^T B with B's codes exact and A's free to move one
E4M3 step each (their tile scale by a relative 2^-7) gives
  |dW_dev - dW_ref| <= (ulp(A) + 2^-7 |A|)^T |B| + 2^-8 |dW_ref|
(the last term: bf16 output and fp32 sums).  That bound assumes every
code moves, all the same way, so it sits far above the usual error; each
expert's gradient as a whole must also stay within the FP8 bound 3e-2
(relative Frobenius)."""

import numpy as np
import pytest
import torch

import oracle
import mixture_experts_layer_82_b300 as moe
from moe_synth import CONFIGS, make_grad, make_layer, shape_with
from oracle.fp8 import dequantize_act_1x128
from oracle.moe_fp8_backward import (dequantize_act_128x1, fp8_swiglu_ffn_backward,
                                     quantize_act_128x1)
from helpers import assert_close, host, rel_frobenius

pytestmark = pytest.mark.gpu

DEV = "cuda"
TOL_FP8 = 3e-2
ROW_TOL_FP8_BWD = 6e-2

SHAPES = [
    # small widths, 16 experts with ragged segments, a shared expert
    shape_with(CONFIGS["v3_fp8"], T=300, d=512, E=16, n_groups=8, topk_groups=4, k=4, inter=256,
               router="gaussian", outlier_channels=5),
    # the V3 hidden and intermediate sizes on few tokens
    shape_with(CONFIGS["v3_fp8"], T=64, E=16, n_groups=8, topk_groups=4, k=4, router="gaussian"),
    # no shared expert; I not a multiple of 256 (the last N tile half outside)
    shape_with(CONFIGS["v3_fp8"], T=200, d=640, E=8, n_groups=4, topk_groups=2, k=2, n_shared=0,
               inter=384, route_scale=1.0, router="gaussian", outlier_channels=7),
    # segments averaging 256 rows (several M tiles per expert, ragged
    # tails), with a shared expert
    shape_with(CONFIGS["v3_fp8"], T=1024, d=512, E=8, n_groups=4, topk_groups=2, k=2, inter=256,
               route_scale=1.0, router="gaussian", outlier_channels=5),
]


def _run(shape, never=(), keep=True):
    """Forward then backward of the FP8 layer; the experts in ``never`` get
    a bias that keeps every token away from them (empty segments).  ``keep``:
    the training forward keeps [a | b] (moe_experts_grouped_train_fp8);
    otherwise the Dgrad recomputes it from the codes."""
    L = make_layer(shape, DEV)
    cfg = moe.LayerCfg.from_shape(shape)
    bias = L["bias"].clone()
    for e in never:
        bias[e] = -1e4
    layer = moe.MoELayer(cfg, L["router_w"], bias, L["w13"], L["w2"],
                         L["ws13"] if shape.n_shared else None,
                         L["ws2"] if shape.n_shared else None)
    aff = torch.empty(shape.T, shape.E, dtype=torch.float32, device=DEV)
    layer.forward(L["x"], affinity_out=aff, update_bias=False, keep=keep)
    dout = make_grad(shape, DEV)
    dx = layer.backward(L["x"], dout, aff)
    assert moe.moe_get_device_error() == 0
    return L, layer, dout, dx


def _codes(t):
    return t.float().cpu().numpy().astype(np.float64)


@pytest.mark.parametrize("shape", SHAPES,
                         ids=lambda s: f"T{s.T}-d{s.d}-E{s.E}-I{s.inter}-Ns{s.n_shared}")
def test_fp8_dgrad_matches_oracle(shape):
    L, layer, dout, dx = _run(shape)
    off = host(layer.offsets)
    qx, sx = _codes(layer.x_perm), host(layer.x_perm_s).astype(np.float64)
    dy = host(layer.dy_perm).astype(np.float64)
    got = host(layer.dx_perm)
    ref = np.zeros_like(got, dtype=np.float64)
    for e in range(shape.E):
        lo, hi = int(off[e]), int(off[e + 1])
        if hi > lo:
            ref[lo:hi] = fp8_swiglu_ffn_backward(qx[lo:hi], sx[lo:hi], host(L["w13"][e]),
                                                 host(L["w2"][e]), dy[lo:hi])["du"]
    assert_close(got, ref, TOL_FP8, "dx_perm", row_tol=ROW_TOL_FP8_BWD)
    if shape.n_shared:
        r = fp8_swiglu_ffn_backward(_codes(layer.x_q), host(layer.x_q_s).astype(np.float64),
                                    host(L["ws13"][0]), host(L["ws2"][0]),
                                    host(dout).astype(np.float64))
        assert_close(host(layer.dx_shared), r["du"], TOL_FP8, "dx_shared", row_tol=ROW_TOL_FP8_BWD)
    assert np.all(np.isfinite(host(dx)))


def _e4m3_ulp(q):
    """One E4M3 step at each grid value q (the unscaled code): 2^(e - 3)
    in the binade [2^e, 2^(e+1)) of a normal value, 2^-9 below 2^-6."""
    a = np.abs(q)
    e = np.floor(np.log2(np.maximum(a, 2.0 ** -6)))
    return np.where(a >= 2.0 ** -6, 2.0 ** (e - 3), 2.0 ** -9)


def _moved(x):
    """(ulp(A) + 2^-7 |A|) per element of A, quantised in 128 x 1 tiles the
    way the oracle quantises it."""
    q, sc = quantize_act_128x1(np.asarray(x, np.float64).astype(np.float32))
    step = np.repeat(np.asarray(sc, np.float64), 128, axis=0)[:len(q)]
    return _e4m3_ulp(q) * step + 2.0 ** -7 * np.abs(dequantize_act_128x1(q, sc))


def _exact(x):
    """|B| as the Wgrad sees it (its 128 x 1 quantisation, dequantised)."""
    q, sc = quantize_act_128x1(np.asarray(x, np.float64).astype(np.float32))
    return np.abs(dequantize_act_128x1(q, sc))


def _check_wgrad(got, r, qx, sx, dy, what):
    """dW2 = dy^T h (h's codes may move) and dW13 = [da | db]^T u ([da | db]
    moves) of one expert against the oracle's ``r``: each element within
    its bound, the whole within 3e-2."""
    dab = np.concatenate([r["da"], r["db"]], axis=1)
    b2 = (_moved(r["h"]).T @ _exact(dy)).T + 2.0 ** -8 * np.abs(r["dw2"])
    b13 = _moved(dab).T @ _exact(dequantize_act_1x128(qx, sx)) + 2.0 ** -8 * np.abs(r["dw13"])
    for g, ref, b, name in ((got[0], r["dw2"], b2, "dw2"), (got[1], r["dw13"], b13, "dw13")):
        excess = np.abs(g - ref) - b
        worst = np.unravel_index(int(np.argmax(excess)), excess.shape)
        assert excess[worst] <= 0, (what, name, worst, float(g[worst]), float(ref[worst]),
                                    float(b[worst]))
        assert rel_frobenius(g, ref) < TOL_FP8, (what, name, rel_frobenius(g, ref))


def _check_experts(L, layer, experts, off):
    """Every expert in ``experts`` checked element by element; returns the
    stacked device and oracle gradients for the Frobenius bound."""
    d, I2 = L["w13"].shape[2], L["w13"].shape[1]
    g13, g2, r13, r2 = [], [], [], []
    for e in experts:
        lo, hi = int(off[e]), int(off[e + 1])
        got = (host(layer.dw2[e]), host(layer.dw13[e]))
        if hi == lo:
            assert not got[0].any() and not got[1].any(), ("expert without rows", e)
            continue
        qx, sx = _codes(layer.x_perm[lo:hi]), host(layer.x_perm_s[lo:hi]).astype(np.float64)
        dy = host(layer.dy_perm[lo:hi]).astype(np.float64)
        r = fp8_swiglu_ffn_backward(qx, sx, host(L["w13"][e]), host(L["w2"][e]), dy)
        _check_wgrad(got, r, qx, sx, dy, f"expert {e}")
        # the same expert's input gradient (Dgrad) on its rows
        assert_close(host(layer.dx_perm[lo:hi]), r["du"], TOL_FP8, f"dx_perm of expert {e}",
                     row_tol=ROW_TOL_FP8_BWD)
        g2.append(got[0]); g13.append(got[1]); r2.append(r["dw2"]); r13.append(r["dw13"])
    return [np.concatenate(v) for v in (g2, r2, g13, r13)]


@pytest.mark.parametrize("shape", SHAPES,
                         ids=lambda s: f"T{s.T}-d{s.d}-E{s.E}-I{s.inter}-Ns{s.n_shared}")
def test_fp8_wgrad_matches_oracle(shape):
    never = (3,)
    L, layer, dout, dx = _run(shape, never)
    off = host(layer.offsets)
    assert off[4] == off[3]
    g2, r2, g13, r13 = _check_experts(L, layer, range(shape.E), off)
    assert rel_frobenius(g2, r2) < TOL_FP8 and rel_frobenius(g13, r13) < TOL_FP8
    if shape.n_shared:
        qx, sx = _codes(layer.x_q), host(layer.x_q_s).astype(np.float64)
        dy = host(dout).astype(np.float64)
        r = fp8_swiglu_ffn_backward(qx, sx, host(L["ws13"][0]), host(L["ws2"][0]), dy)
        got = (host(layer.dws2[0]), host(layer.dws13[0]))
        _check_wgrad(got, r, qx, sx, dy, "shared expert")
        assert rel_frobenius(got[0], r["dw2"]) < TOL_FP8
        assert rel_frobenius(got[1], r["dw13"]) < TOL_FP8


def test_fp8_wgrad_full_size_on_sampled_experts():
    """The FP8 layer at its full size (T = 8192, d = 7168, 256 experts, one
    shared): the oracle recomputes the weight and input gradients of four
    experts, the most loaded, one whose rows fit one 128-row tile, one with
    a ragged last tile over several tiles, and the last expert."""
    shape = CONFIGS["v3_fp8"]
    L, layer, dout, dx = _run(shape)
    off = host(layer.offsets)
    counts = np.diff(off)
    pick = [int(np.argmax(counts)), shape.E - 1]
    one = np.nonzero((counts >= 1) & (counts <= 128))[0]
    ragged = np.nonzero((counts > 128) & (counts % 128 != 0))[0]
    pick += [int(one[0])] if len(one) else []
    pick += [int(ragged[0])] if len(ragged) else []
    g2, r2, g13, r13 = _check_experts(L, layer, sorted(set(pick)), off)
    assert rel_frobenius(g2, r2) < TOL_FP8 and rel_frobenius(g13, r13) < TOL_FP8
    assert np.all(np.isfinite(host(layer.dws2)))


def test_fp8_backward_is_deterministic():
    shape = SHAPES[0]
    L, layer, dout, dx = _run(shape)
    a = layer.dx_perm.clone()
    w13, w2, ws13 = layer.dw13.clone(), layer.dw2.clone(), layer.dws13.clone()
    aff = torch.empty(shape.T, shape.E, dtype=torch.float32, device=DEV)
    layer.forward(L["x"], affinity_out=aff, update_bias=False)
    layer.backward(L["x"], dout, aff)
    assert torch.equal(a.view(torch.int16), layer.dx_perm.view(torch.int16))
    for u, v in ((w13, layer.dw13), (w2, layer.dw2), (ws13, layer.dws13)):
        assert torch.equal(u.view(torch.int16), v.view(torch.int16))
    assert moe.moe_get_device_error() == 0


@pytest.mark.parametrize("shape", [SHAPES[0], SHAPES[2], SHAPES[3]],
                         ids=lambda s: f"T{s.T}-d{s.d}-E{s.E}-I{s.inter}-Ns{s.n_shared}")
def test_fp8_kept_ab_matches_recomputed(shape):
    """The training forward's [a | b] (the gate/up promotion's fp32 sums,
    rounded to bf16) against the Dgrad's recompute from the same codes (the
    same per-128-K promotion in the plain GEMM): the backward's outputs
    agree far inside the FP8 bound."""
    L, kept, dout, _ = _run(shape, keep=True)
    got = [host(t).copy() for t in (kept.dx_perm, kept.dw13, kept.dw2)]
    _, again, _, _ = _run(shape, keep=False)
    for g, r, name in zip(got, (again.dx_perm, again.dw13, again.dw2), ("dx_perm", "dw13", "dw2")):
        assert rel_frobenius(g, host(r)) < 2e-3, (name, rel_frobenius(g, host(r)))


def test_fp8_128x1_quantiser_is_exact():
    """moe_quantize_act_fp8_128x1 (the quantiser of Wgrad's operands) against
    the oracle's 128 x 1 tiles, codes and scales bit for bit: a ragged last
    tile, an all-zero column, outlier rows, and a column whose scale is 1
    holding values exactly on E4M3 rounding midpoints and one bf16 step
    either side (the quotients the reciprocal path hands to the exact
    division)."""
    rng = np.random.default_rng(12)
    rows, cols = 300, 384
    x = rng.standard_normal((rows, cols)) * np.exp(rng.standard_normal(cols))[None, :]
    x[rng.integers(0, rows, 6)] *= 40.0
    x[:, 5] = 0.0
    # column 7: amax 448 in every tile (scale 1), then midpoints of E4M3 steps
    grid = np.array([1.0, 1.125, 1.25, 1.375, 1.5, 1.625, 1.75, 1.875, 2.0])
    mids = np.concatenate([(grid[:-1] + grid[1:]) / 2 * 2.0 ** e for e in range(-6, 8)])
    mb = torch.tensor(mids, dtype=torch.float32).bfloat16()  # exact: 5 significant bits
    step = [(mb.view(torch.int16) + k).view(torch.bfloat16).float().numpy() for k in (-1, 1)]
    col = np.resize(np.concatenate([mids, step[0], step[1]]), rows)
    col[::128] = 448.0
    x[:, 7] = col
    xb = torch.tensor(x, dtype=torch.float32).bfloat16()
    xf = xb.float().numpy()
    P = (rows + 127) // 128 * 128
    q = torch.empty(P, cols, dtype=torch.float8_e4m3fn, device=DEV)
    sc = torch.empty(P // 128, cols, dtype=torch.float32, device=DEV)
    moe.moe_quantize_act_fp8_128x1(xb.to(DEV), q, sc)
    assert moe.moe_get_device_error() == 0
    rq, rs = quantize_act_128x1(xf)
    assert np.array_equal(host(sc), np.asarray(rs, np.float32)), "scales"
    got = q.float().cpu().numpy().astype(np.float64)
    assert np.array_equal(got[:rows], rq), "codes"
    assert not got[rows:].any(), "padding rows"


def test_fp8_weight_transpose_is_exact():
    """The transposed copies hold the forward's codes and block scales,
    transposed: nothing is quantised again."""
    rng = np.random.default_rng(6)
    w = torch.tensor(rng.standard_normal((3, 384, 256)) * 0.02, dtype=torch.bfloat16, device=DEV)
    q = torch.empty(3, 384, 256, dtype=torch.float8_e4m3fn, device=DEV)
    s = torch.empty(3, 3, 2, dtype=torch.float32, device=DEV)
    moe.moe_quantize_weights_fp8(w, q, s)
    qt = torch.empty(3, 256, 384, dtype=torch.float8_e4m3fn, device=DEV)
    st = torch.empty(3, 2, 3, dtype=torch.float32, device=DEV)
    moe.moe_transpose_weights_fp8(q, s, qt, st)
    assert torch.equal(qt.view(torch.uint8), q.view(torch.uint8).transpose(1, 2))
    assert torch.equal(st, s.transpose(1, 2))
    assert moe.moe_get_device_error() == 0
