"""Parity of the FP8 E4M3 path (through the C ABI) with the FP8 CPU oracle.

The oracle quantises x per 1 x 128 tile and the bf16 master weights per
128 x 128 block with the same fp32 formula, dequantises, multiplies in fp64
and re-quantises h between the two projections.  The activation codes and
scales must match bit for bit; the layer output (and each expert output) must
match within a relative Frobenius error of 3e-2."""

import numpy as np
import pytest
import torch

import oracle
import mixture_experts_layer_82_b300 as moe
from moe_synth import CONFIGS, make_layer, shape_with
from helpers import assert_close, host, ExpertView, tail_sample

pytestmark = pytest.mark.gpu

DEV = "cuda"
TOL_FP8 = 3e-2

# Reduced FP8 layers the oracle finishes in seconds; every one spans several
# M and N tiles with ragged segment tails.
SHAPES = [
    # V3 hidden and intermediate sizes, 16 experts, outlier channels
    shape_with(CONFIGS["v3_fp8"], T=96, E=16, n_groups=8, topk_groups=4, k=4,
               router="gaussian"),
    # d % 256 == 128 (the last down tile is half outside d), two shared experts
    shape_with(CONFIGS["v3_fp8"], T=301, d=640, E=8, n_groups=4, topk_groups=2, k=2,
               n_shared=2, inter=384, route_scale=1.0, router="gaussian", outlier_channels=7),
    # no shared expert, many small segments
    shape_with(CONFIGS["v3_fp8"], T=150, d=512, E=32, n_groups=8, topk_groups=4, k=6,
               n_shared=0, inter=256, router="gaussian", outlier_channels=5),
    # one token
    shape_with(CONFIGS["v3_fp8"], T=1, d=1024, E=16, n_groups=4, topk_groups=2, k=3,
               inter=512, router="gaussian", outlier_channels=10),
    # the mid-size layer's widths in FP8, whole batch: 384 rows per expert on
    # average, so a persistent CTA cycles its TMEM partials over several M
    # tiles of one expert and most segments end in a ragged tile inside a
    # multi-tile expert; two shared experts; 1% outlier channels
    shape_with(CONFIGS["v3_fp8"], T=4096, d=2048, E=64, n_groups=8, topk_groups=4, k=6,
               n_shared=2, inter=1408, route_scale=1.0, router="gaussian",
               outlier_channels=20),
    # segments averaging 256 rows: several M tiles per expert with ragged
    # tails; d % 256 == 128 and I % 256 == 128 (the last N tile of each GEMM
    # half outside), one shared expert
    shape_with(CONFIGS["v3_fp8"], T=1024, d=640, E=8, n_groups=4, topk_groups=2, k=2,
               n_shared=1, inter=384, route_scale=1.0, router="gaussian", outlier_channels=7),
]


def _fp8_layer(shape, L=None):
    L = L or make_layer(shape, DEV)
    cfg = moe.LayerCfg.from_shape(shape)
    layer = moe.MoELayer(cfg, L["router_w"], L["bias"].clone(), L["w13"], L["w2"],
                         L["ws13"] if shape.n_shared else None,
                         L["ws2"] if shape.n_shared else None)
    return L, cfg, layer


def _codes(t):
    """E4M3 tensor -> fp64 grid values on the host."""
    return t.float().cpu().numpy().astype(np.float64)


@pytest.mark.parametrize("shape", [shape_with(CONFIGS["v3_fp8"], T=300), SHAPES[1]],
                         ids=lambda s: f"T{s.T}-d{s.d}")
def test_fp8_dispatch_bitwise(shape):
    """Quantise-then-dispatch: x codes and 1 x 128 scales equal the oracle's
    bit for bit, and every permuted row is its token's codes and scales."""
    L, cfg, layer = _fp8_layer(shape)
    layer.forward(L["x"], update_bias=False)
    assert moe.moe_get_device_error() == 0
    q, s = oracle.quantize_act_1x128(host(L["x"]))
    assert np.array_equal(host(layer.x_q_s).view(np.uint32), s.view(np.uint32))
    assert np.array_equal(_codes(layer.x_q), q)
    tor = torch.tensor(host(layer.token_of_row).astype(np.int64), device=DEV)
    assert torch.equal(layer.x_perm.view(torch.uint8), layer.x_q.view(torch.uint8)[tor])
    assert torch.equal(layer.x_perm_s, layer.x_q_s[tor])


@pytest.mark.parametrize("shape", SHAPES,
                         ids=lambda s: f"T{s.T}-d{s.d}-E{s.E}-I{s.inter}-Ns{s.n_shared}")
def test_fp8_layer_matches_oracle(shape):
    L, cfg, layer = _fp8_layer(shape)
    aff = torch.empty(shape.T, shape.E, dtype=torch.float32, device=DEV)
    out = layer.forward(L["x"], affinity_out=aff, update_bias=False)
    assert moe.moe_get_device_error() == 0
    ws13 = ExpertView(L["ws13"]) if shape.n_shared else None
    ws2 = ExpertView(L["ws2"]) if shape.n_shared else None
    r = oracle.moe_layer_forward_fp8(host(L["x"]), host(L["router_w"]), host(L["bias"]),
                                     ExpertView(L["w13"]), ExpertView(L["w2"]), ws13, ws2,
                                     n_groups=shape.n_groups, topk_groups=shape.topk_groups,
                                     k=shape.k, route_scale=shape.route_scale,
                                     affinity32=host(aff))
    assert np.array_equal(host(layer.topk_idx), r["topk_idx"])
    assert np.array_equal(host(layer.offsets), r["offsets"])
    assert_close(host(layer.y_perm), r["y_perm"], TOL_FP8)
    if shape.n_shared:
        assert_close(host(layer.y_shared), r["y_shared"], TOL_FP8)
    assert_close(host(out), r["out"], TOL_FP8)


def test_fp8_full_size_layer_on_sampled_tokens():
    """The FP8 layer at its full size (T = 8192, d = 7168, 256 experts), in
    the launch configuration the benchmark times; the oracle recomputes 64
    tokens, quantising the master weights itself.  The sample holds the
    tokens of the ragged last tile of the most loaded expert and the last
    rows of one-tile and few-tile experts; each token's row is checked on
    its own."""
    shape = CONFIGS["v3_fp8"]
    L, cfg, layer = _fp8_layer(shape)
    out = layer.forward(L["x"], update_bias=False)
    assert moe.moe_get_device_error() == 0
    o = host(out)
    assert np.all(np.isfinite(o))
    rows = tail_sample(host(layer.offsets), host(layer.token_of_row), shape.T, 64)
    assert len(rows) >= 64
    idx = host(layer.topk_idx)[rows]
    g = host(layer.topk_w)[rows].astype(np.float64)
    ref = oracle.moe_layer_tokens_fp8(host(L["x"][torch.tensor(rows, device=DEV)]), idx, g,
                                      ExpertView(L["w13"]), ExpertView(L["w2"]),
                                      ExpertView(L["ws13"]), ExpertView(L["ws2"]))
    assert_close(o[rows], ref, TOL_FP8)


def test_fp8_layer_is_deterministic():
    shape = SHAPES[0]
    L, cfg, layer = _fp8_layer(shape)
    a = layer.forward(L["x"], update_bias=False).clone()
    ya = layer.y_perm.clone()
    b = layer.forward(L["x"], update_bias=False)
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    assert torch.equal(ya.view(torch.int16), layer.y_perm.view(torch.int16))
    assert moe.moe_get_device_error() == 0
