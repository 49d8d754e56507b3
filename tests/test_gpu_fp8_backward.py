"""Parity of the FP8 backward for input (moe_experts_backward_input_fp8,
through the C ABI) with the FP8 backward oracle.

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
rows in the tail of that distribution."""

import numpy as np
import pytest
import torch

import oracle
import mixture_experts_layer_82_b300 as moe
from moe_synth import CONFIGS, make_grad, make_layer, shape_with
from oracle.moe_fp8_backward import fp8_swiglu_ffn_backward
from helpers import assert_close, host

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
]


def _run(shape):
    L = make_layer(shape, DEV)
    cfg = moe.LayerCfg.from_shape(shape)
    layer = moe.MoELayer(cfg, L["router_w"], L["bias"].clone(), L["w13"], L["w2"],
                         L["ws13"] if shape.n_shared else None,
                         L["ws2"] if shape.n_shared else None)
    aff = torch.empty(shape.T, shape.E, dtype=torch.float32, device=DEV)
    layer.forward(L["x"], affinity_out=aff, update_bias=False)
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


def test_fp8_dgrad_is_deterministic():
    shape = SHAPES[0]
    L, layer, dout, dx = _run(shape)
    a = layer.dx_perm.clone()
    aff = torch.empty(shape.T, shape.E, dtype=torch.float32, device=DEV)
    layer.forward(L["x"], affinity_out=aff, update_bias=False)
    layer.backward(L["x"], dout, aff)
    assert torch.equal(a.view(torch.int16), layer.dx_perm.view(torch.int16))
    assert moe.moe_get_device_error() == 0


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
