"""moe_balance_stat (the sequence-wise balance statistic) against the CPU
oracle.  As for routing, the oracle works from the device's fp32 affinities
and makes its own expert selection from them."""

import numpy as np
import pytest
import torch

import oracle
import mixture_experts_layer_82_b300 as moe
from moe_synth import CONFIGS, make_layer, shape_with
from helpers import host

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _route(shape, L=None, s32=None):
    cfg = moe.LayerCfg.from_shape(shape)
    T, E, K = shape.T, shape.E, shape.k
    i32 = dict(dtype=torch.int32, device=DEV)
    out = [torch.empty(T, K, **i32), torch.empty(T, K, dtype=torch.float32, device=DEV),
           torch.empty(E, **i32), torch.empty(E + 1, **i32), torch.empty(T, K, **i32),
           torch.empty(T * K, **i32)]
    ws = torch.empty(moe.moe_workspace_bytes(cfg), dtype=torch.uint8, device=DEV)
    bias = torch.zeros(E, dtype=torch.float32, device=DEV)
    if s32 is None:
        aff = torch.empty(T, E, dtype=torch.float32, device=DEV)
        moe.moe_route(cfg, L["x"], L["router_w"], bias, *out, ws, affinity_out=aff)
    else:
        aff = torch.tensor(s32, device=DEV)
        moe.moe_route(cfg, None, None, bias, *out, ws, affinity_in=aff)
    return cfg, aff, out[0]


def _check(shape, cfg, aff, idx, seq_len, alpha=1e-4):
    n = shape.T // seq_len
    f = torch.empty(n, shape.E, dtype=torch.float32, device=DEV)
    p = torch.empty_like(f)
    loss = torch.empty(n, dtype=torch.float32, device=DEV)
    ws = torch.empty(moe.moe_workspace_bytes(cfg), dtype=torch.uint8, device=DEV)
    moe.moe_balance_stat(cfg, aff, idx, seq_len, f, p, loss, ws, alpha=alpha)
    assert moe.moe_get_device_error() == 0
    s32 = host(aff)
    oidx = oracle.select_experts(s32, np.zeros(shape.E, np.float32), shape.n_groups,
                                 shape.topk_groups, shape.k, shape.group_score_topn)
    assert np.array_equal(host(idx), oidx)
    fo, po, lo = oracle.sequence_balance(s32, oidx, seq_len, alpha)
    np.testing.assert_allclose(host(f), fo, rtol=1e-6, atol=0)
    np.testing.assert_allclose(host(p), po, rtol=1e-4, atol=1e-9)
    np.testing.assert_allclose(host(loss), lo, rtol=1e-4, atol=0)


@pytest.mark.parametrize("name,seq_len", [("mid_bf16", 1024), ("v3_bf16", 8192),
                                          ("v3_bf16", 4096)])
def test_balance_stat_matches_oracle(name, seq_len):
    shape = CONFIGS[name]
    L = make_layer(shape, DEV, weights=False)
    cfg, aff, idx = _route(shape, L)
    _check(shape, cfg, aff, idx, seq_len)


def test_balance_stat_ragged_experts():
    """E = 24 (the last 32-expert chunk is partial), K = 3, three sequences."""
    shape = shape_with(CONFIGS["mid_bf16"], T=300, E=24, n_groups=4, topk_groups=2, k=3)
    rng = np.random.default_rng(5)
    s = rng.random((shape.T, shape.E)).astype(np.float32)
    cfg, aff, idx = _route(shape, s32=s)
    _check(shape, cfg, aff, idx, 100, alpha=3e-3)


def test_balance_stat_rejects_bad_sequence_length():
    shape = shape_with(CONFIGS["mid_bf16"], T=300, E=24, n_groups=4, topk_groups=2, k=3)
    cfg = moe.LayerCfg.from_shape(shape)
    aff = torch.rand(shape.T, shape.E, device=DEV)
    idx = torch.zeros(shape.T, shape.k, dtype=torch.int32, device=DEV)
    f = torch.empty(3, shape.E, device=DEV)
    with pytest.raises(moe.MoeError) as e:
        ws = torch.empty(moe.moe_workspace_bytes(cfg), dtype=torch.uint8, device=DEV)
        moe.moe_balance_stat(cfg, aff, idx, 7, f, f.clone(), torch.empty(3, device=DEV), ws)
    assert e.value.status == 1  # MOE_ERR_INVALID_ARG
