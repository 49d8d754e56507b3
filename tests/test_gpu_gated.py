"""The gate multiply folded into the down projection (moe_experts_grouped_gated)
with the combine reduced to a plain ordered sum (moe_combine with no gates),
through the C ABI, against the oracle: every gated row is g * FFN(u) for the
copy it holds, and the layer output is the oracle's gate-weighted sum."""

import numpy as np
import pytest
import torch

import oracle
import mixture_experts_layer_82_b300 as moe
from moe_synth import CONFIGS, make_layer, shape_with
from helpers import assert_close, host, ExpertView, tail_sample

pytestmark = pytest.mark.gpu

DEV = "cuda"
TOL = {"fp32": 1e-5, "bf16": 1e-2, "fp8": 3e-2}


def _layer(shape):
    L = make_layer(shape, DEV)
    cfg = moe.LayerCfg.from_shape(shape)
    layer = moe.MoELayer(cfg, L["router_w"], L["bias"].clone(), L["w13"], L["w2"],
                         L["ws13"] if shape.n_shared else None,
                         L["ws2"] if shape.n_shared else None)
    return L, layer


@pytest.mark.parametrize("shape", [
    CONFIGS["tiny_fp32"],
    shape_with(CONFIGS["mid_bf16"], T=1000),
    shape_with(CONFIGS["mid_bf16"], T=333, n_shared=0),
    shape_with(CONFIGS["v3_fp8"], T=96, E=16, n_groups=8, topk_groups=4, k=4, router="gaussian"),
], ids=lambda s: f"{s.dtype}-T{s.T}-Ns{s.n_shared}")
def test_gated_layer_matches_oracle(shape):
    L, layer = _layer(shape)
    aff = torch.empty(shape.T, shape.E, dtype=torch.float32, device=DEV)
    out = layer.forward(L["x"], affinity_out=aff, update_bias=False, gated=True).clone()
    assert moe.moe_get_device_error() == 0
    ws13 = ExpertView(L["ws13"]) if shape.n_shared else None
    ws2 = ExpertView(L["ws2"]) if shape.n_shared else None
    ins = [host(L[k]) for k in ("x", "router_w", "bias")]
    kw = dict(n_groups=shape.n_groups, topk_groups=shape.topk_groups, k=shape.k,
              route_scale=shape.route_scale, affinity32=host(aff))
    if shape.dtype == "fp8":
        r = oracle.moe_layer_forward_fp8(*ins, ExpertView(L["w13"]), ExpertView(L["w2"]), ws13,
                                         ws2, **kw)
    else:
        r = oracle.moe_layer_forward(*ins, ExpertView(L["w13"]), ExpertView(L["w2"]), ws13, ws2,
                                     **kw)
    assert np.array_equal(host(layer.topk_idx), r["topk_idx"])
    gr = oracle.gate_of_row(r["row_of_slot"], r["topk_w"])
    assert_close(host(layer.y_perm), gr[:, None] * r["y_perm"], TOL[shape.dtype])
    assert_close(host(out), r["out"], TOL[shape.dtype])
    # the ungated forward of the same batch: same output within the kind's
    # rounding (the gate is applied before, not after, the bf16 rounding)
    ref = layer.forward(L["x"], update_bias=False)
    assert_close(host(out), host(ref), TOL[shape.dtype])


def test_gated_full_size_layer_on_sampled_tokens():
    """The V3 bf16 layer at full size with gated rows; 64 sampled tokens
    (ragged tails of the busiest expert and of one-tile experts included)
    recomputed by the oracle."""
    shape = CONFIGS["v3_bf16"]
    L, layer = _layer(shape)
    out = layer.forward(L["x"], update_bias=False, gated=True)
    assert moe.moe_get_device_error() == 0
    o = host(out)
    rows = tail_sample(host(layer.offsets), host(layer.token_of_row), shape.T, 64)
    ref = oracle.moe_layer_tokens(host(L["x"][torch.tensor(rows, device=DEV)]),
                                  host(layer.topk_idx)[rows],
                                  host(layer.topk_w)[rows].astype(np.float64),
                                  ExpertView(L["w13"]), ExpertView(L["w2"]),
                                  ExpertView(L["ws13"]), ExpertView(L["ws2"]))
    assert_close(o[rows], ref, TOL["bf16"])


def test_gated_layer_is_deterministic():
    shape = shape_with(CONFIGS["mid_bf16"], T=700)
    L, layer = _layer(shape)
    a = layer.forward(L["x"], update_bias=False, gated=True).clone()
    b = layer.forward(L["x"], update_bias=False, gated=True)
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    assert moe.moe_get_device_error() == 0
