"""moe_experts_grouped_gather: the permute folded into the gate/up GEMM
(routed A rows read from x by token_of_row).  The A operand holds the same
bf16 values as with a permuted copy, so every output must equal the
permute + moe_experts_grouped path bit for bit; one case is also checked
against the CPU oracle directly."""

import numpy as np
import pytest
import torch

import oracle
import mixture_experts_layer_82_b300 as moe
from moe_synth import CONFIGS, make_layer, shape_with
from helpers import rel_frobenius, assert_close, host, ExpertView

pytestmark = pytest.mark.gpu
DEV = "cuda"

SHAPES = [
    shape_with(CONFIGS["mid_bf16"], T=1000),
    shape_with(CONFIGS["mid_bf16"], T=333, n_shared=0),
    shape_with(CONFIGS["mid_bf16"], T=1),
    CONFIGS["v3_bf16"],
]


def _layer(shape, L):
    cfg = moe.LayerCfg.from_shape(shape)
    return moe.MoELayer(cfg, L["router_w"], L["bias"].clone(), L["w13"], L["w2"],
                        L["ws13"] if shape.n_shared else None,
                        L["ws2"] if shape.n_shared else None)


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: f"{s.name}-T{s.T}-Ns{s.n_shared}")
def test_gather_equals_permute_path_bitwise(shape):
    L = make_layer(shape, DEV)
    layer = _layer(shape, L)
    out_p = layer.forward(L["x"], update_bias=False, gather=False).clone()
    y_p = layer.y_perm.clone()
    ys_p = layer.y_shared.clone() if shape.n_shared else None
    layer.y_perm.fill_(7.0)  # the gathering call must write every row again
    out_g = layer.forward(L["x"], update_bias=False, gather=True)
    assert moe.moe_get_device_error() == 0
    assert torch.equal(layer.y_perm.view(torch.int16), y_p.view(torch.int16))
    if shape.n_shared:
        assert torch.equal(layer.y_shared.view(torch.int16), ys_p.view(torch.int16))
    assert torch.equal(out_g.view(torch.int16), out_p.view(torch.int16))


def test_gather_layer_matches_oracle():
    shape = shape_with(CONFIGS["mid_bf16"], T=517)
    L = make_layer(shape, DEV)
    layer = _layer(shape, L)
    aff = torch.empty(shape.T, shape.E, dtype=torch.float32, device=DEV)
    out = layer.forward(L["x"], affinity_out=aff, update_bias=False, gather=True)
    assert moe.moe_get_device_error() == 0
    r = oracle.moe_layer_forward(host(L["x"]), host(L["router_w"]), host(L["bias"]),
                                 ExpertView(L["w13"]), ExpertView(L["w2"]),
                                 ExpertView(L["ws13"]), ExpertView(L["ws2"]),
                                 n_groups=shape.n_groups, topk_groups=shape.topk_groups,
                                 k=shape.k, route_scale=shape.route_scale, affinity32=host(aff))
    assert np.array_equal(host(layer.topk_idx), r["topk_idx"])
    assert_close(host(out), r["out"], 1e-2)


def test_gather_rejects_other_kinds():
    shape = shape_with(CONFIGS["v3_fp8"], T=64, E=16, n_groups=4, topk_groups=2, k=2,
                       router="gaussian", outlier_channels=0)
    L = make_layer(shape, DEV)
    layer = _layer(shape, L)
    layer.forward(L["x"], update_bias=False)
    with pytest.raises(moe.MoeError) as e:
        moe.moe_experts_grouped_gather(layer.cfg, L["x"], layer.token_of_row, layer.offsets,
                                       layer.w13, layer.w2, layer.ws13, layer.ws2, layer.y_perm,
                                       layer.y_shared, layer.ws)
    assert e.value.status == 2  # MOE_ERR_SHAPE
