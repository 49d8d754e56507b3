"""Parity of the CUDA path (through the C ABI) with the CPU oracle.

Routing (indices, loads, offsets, permuted rows) must match bit for bit given
the device's own fp32 affinities; floating-point outputs must match within
a relative Frobenius error of 1e-2 (bf16 kind) or 1e-5 (fp32 kind)."""

import numpy as np
import pytest
import torch

import oracle
import mixture_experts_layer_82_b300 as moe
from moe_synth import CONFIGS, make_layer, shape_with
from helpers import rel_frobenius, assert_close, host, ExpertView, tail_sample

pytestmark = pytest.mark.gpu

DEV = "cuda"
TOL = {"fp32": 1e-5, "bf16": 1e-2}


def _layer(shape, L=None):
    L = L or make_layer(shape, DEV)
    cfg = moe.LayerCfg.from_shape(shape)
    layer = moe.MoELayer(cfg, L["router_w"], L["bias"].clone(), L["w13"], L["w2"],
                         L["ws13"] if shape.n_shared else None,
                         L["ws2"] if shape.n_shared else None)
    return L, cfg, layer


def _check_routing(shape, layer, s32, bias):
    idx = oracle.select_experts(s32, bias, shape.n_groups, shape.topk_groups, shape.k,
                                shape.group_score_topn)
    assert np.array_equal(host(layer.topk_idx), idx)
    counts, offsets, ros, tor = oracle.segment_layout(idx, shape.E)
    assert np.array_equal(host(layer.counts), counts)
    assert np.array_equal(host(layer.offsets), offsets)
    assert np.array_equal(host(layer.row_of_slot), ros)
    assert np.array_equal(host(layer.token_of_row), tor)
    g = oracle.gating_weights(s32, idx, shape.route_scale)
    np.testing.assert_allclose(host(layer.topk_w), g, rtol=1e-6, atol=1e-7)
    return idx


# ----------------------------------------------------------------- routing

@pytest.mark.parametrize("name", ["tiny_fp32", "mid_bf16", "v3_bf16", "v3_decode"])
def test_routing_bit_exact(name):
    shape = CONFIGS[name]
    L = make_layer(shape, DEV, weights=False)
    cfg = moe.LayerCfg.from_shape(shape)
    T, E, K = shape.T, shape.E, shape.k
    aff = torch.empty(T, E, dtype=torch.float32, device=DEV)
    i32 = dict(dtype=torch.int32, device=DEV)
    out = dict(topk_idx=torch.empty(T, K, **i32),
               topk_w=torch.empty(T, K, dtype=torch.float32, device=DEV),
               counts=torch.empty(E, **i32), offsets=torch.empty(E + 1, **i32),
               row_of_slot=torch.empty(T, K, **i32), token_of_row=torch.empty(T * K, **i32))
    ws = torch.empty(moe.moe_workspace_bytes(cfg), dtype=torch.uint8, device=DEV)
    moe.moe_route(cfg, L["x"], L["router_w"], L["bias"], ws=ws, affinity_out=aff, **out)
    assert moe.moe_get_device_error() == 0

    class R:  # attribute access like MoELayer
        pass
    r = R()
    for k, v in out.items():
        setattr(r, k, v)
    s32 = host(aff)
    _check_routing(shape, r, s32, host(L["bias"]))
    s64 = oracle.sigmoid_affinity(host(L["x"]), host(L["router_w"]))
    assert np.max(np.abs(s64 - s32)) < 1e-5


def _route_with_affinity(shape, s32, bias):
    cfg = moe.LayerCfg.from_shape(shape)
    T, E, K = shape.T, shape.E, shape.k
    i32 = dict(dtype=torch.int32, device=DEV)

    class R:
        pass
    r = R()
    r.topk_idx = torch.empty(T, K, **i32)
    r.topk_w = torch.empty(T, K, dtype=torch.float32, device=DEV)
    r.counts = torch.empty(E, **i32)
    r.offsets = torch.empty(E + 1, **i32)
    r.row_of_slot = torch.empty(T, K, **i32)
    r.token_of_row = torch.empty(T * K, **i32)
    ws = torch.empty(moe.moe_workspace_bytes(cfg), dtype=torch.uint8, device=DEV)
    moe.moe_route(cfg, None, None, torch.tensor(bias, device=DEV), r.topk_idx, r.topk_w,
                  r.counts, r.offsets, r.row_of_slot, r.token_of_row, ws,
                  affinity_in=torch.tensor(s32, device=DEV))
    assert moe.moe_get_device_error() == 0
    return r


@pytest.mark.parametrize("T,E,G,keep,K,topn,seed", [
    (1000, 256, 8, 4, 8, 2, 0), (77, 16, 4, 2, 2, 2, 1), (33, 64, 8, 4, 6, 2, 2),
    (1, 256, 8, 4, 8, 2, 3), (300, 32, 1, 1, 4, 3, 4), (129, 1024, 32, 5, 32, 2, 5),
    (64, 8, 8, 8, 8, 1, 6),
])
def test_routing_ties_and_edges(T, E, G, keep, K, topn, seed):
    """Saturated sigmoids (exact 1.0f), repeated values and zero bias make
    ties everywhere; ragged T, one token, one group and E = K cover the edges."""
    rng = np.random.default_rng(seed)
    s = rng.random((T, E)).astype(np.float32)
    s[rng.random((T, E)) < 0.3] = np.float32(1.0)
    s[:, 1::4] = s[:, 0::4][:, : s[:, 1::4].shape[1]]
    b = np.where(rng.random(E) < 0.5, 0.0, (rng.random(E) - 0.5) * 0.1).astype(np.float32)
    shape = shape_with(CONFIGS["mid_bf16"], T=T, E=E, n_groups=G, topk_groups=keep, k=K,
                       group_score_topn=topn)
    r = _route_with_affinity(shape, s, b)
    _check_routing(shape, r, s, b)


def test_routing_hot_expert_gets_every_token():
    """Every token picks expert 0 (largest loads possible; all other segments
    hold what is left) and several experts stay empty."""
    T, E = 4100, 64
    rng = np.random.default_rng(9)
    s = (rng.random((T, E)) * 0.5).astype(np.float32)
    s[:, 0] = 1.0
    s[:, 1:8] = 0.9
    shape = shape_with(CONFIGS["mid_bf16"], T=T)
    r = _route_with_affinity(shape, s, np.zeros(E, np.float32))
    idx = _check_routing(shape, r, s, np.zeros(E, np.float32))
    assert host(r.counts)[0] == T


# ----------------------------------------------------------- permute/combine

@pytest.mark.parametrize("name", ["mid_bf16", "v3_bf16", "tiny_fp32"])
def test_permute_exact(name):
    shape = CONFIGS[name]
    L, cfg, layer = _layer(shape)
    layer.forward(L["x"], update_bias=False)
    assert moe.moe_get_device_error() == 0
    tor = host(layer.token_of_row).astype(np.int64)
    xp = layer.x_perm.view(torch.int16 if shape.dtype == "bf16" else torch.int32)
    xx = L["x"].view(torch.int16 if shape.dtype == "bf16" else torch.int32)
    assert torch.equal(xp, xx[torch.tensor(tor, device=DEV)])


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
def test_combine_matches_oracle(dtype):
    T, K, d, E = 517, 6, 2048, 64
    rng = np.random.default_rng(3)
    idx = np.stack([rng.choice(E, K, replace=False) for _ in range(T)]).astype(np.int32)
    _, _, ros, _ = oracle.segment_layout(idx, E)
    g = rng.random((T, K)).astype(np.float32)
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    yp = torch.randn(T * K, d, device=DEV).to(tdt)
    ys = torch.randn(T, d, device=DEV).to(tdt)
    out = torch.empty(T, d, device=DEV, dtype=tdt)
    cfg = moe.LayerCfg(T, d, E, 8, 4, K, 1, 128, dtype=dtype)
    moe.moe_combine(cfg, yp, ys, torch.tensor(ros.astype(np.int32), device=DEV),
                    torch.tensor(g, device=DEV), out)
    ref = oracle.combine(host(ys), host(yp), ros, g.astype(np.float64))
    assert_close(host(out), ref, (4e-3 if dtype == "bf16" else 1e-6))
    # no shared expert
    cfg0 = moe.LayerCfg(T, d, E, 8, 4, K, 0, 128, dtype=dtype)
    moe.moe_combine(cfg0, yp, None, torch.tensor(ros.astype(np.int32), device=DEV),
                    torch.tensor(g, device=DEV), out)
    ref0 = oracle.combine(None, host(yp), ros, g.astype(np.float64))
    assert_close(host(out), ref0, (4e-3 if dtype == "bf16" else 1e-6))


# ----------------------------------------------------------------- layer

def _oracle_layer(shape, L, s32):
    ins = [host(L[k]) for k in ("x", "router_w", "bias")]
    ws13 = ExpertView(L["ws13"]) if shape.n_shared else None
    ws2 = ExpertView(L["ws2"]) if shape.n_shared else None
    return oracle.moe_layer_forward(*ins, ExpertView(L["w13"]), ExpertView(L["w2"]), ws13, ws2,
                                    n_groups=shape.n_groups, topk_groups=shape.topk_groups,
                                    k=shape.k, route_scale=shape.route_scale, affinity32=s32)


@pytest.mark.parametrize("shape", [
    CONFIGS["tiny_fp32"],
    shape_with(CONFIGS["tiny_fp32"], T=45, n_shared=0),
    shape_with(CONFIGS["mid_bf16"], T=256),
    shape_with(CONFIGS["mid_bf16"], T=1000),
    shape_with(CONFIGS["mid_bf16"], T=333, n_shared=0),
    CONFIGS["mid_bf16"],
], ids=lambda s: f"{s.name}-T{s.T}-Ns{s.n_shared}")
def test_layer_matches_oracle(shape):
    L, cfg, layer = _layer(shape)
    aff = torch.empty(shape.T, shape.E, dtype=torch.float32, device=DEV)
    out = layer.forward(L["x"], affinity_out=aff, update_bias=False)
    assert moe.moe_get_device_error() == 0
    s32 = host(aff)
    r = _oracle_layer(shape, L, s32)
    assert np.array_equal(host(layer.topk_idx), r["topk_idx"])
    tol = TOL[shape.dtype]
    assert_close(host(layer.y_perm), r["y_perm"], tol)
    if shape.n_shared:
        assert_close(host(layer.y_shared), r["y_shared"], tol)
    assert_close(host(out), r["out"], tol)


@pytest.mark.parametrize("name,n_sample", [("v3_bf16", 64), ("v3_decode", 128)])
def test_full_size_layer_on_sampled_tokens(name, n_sample):
    """The whole layer at its full size, in the launch configuration the
    benchmark times; the oracle recomputes a sample of tokens one by one
    (every token of the decode batch).  The sample holds the tokens of the
    ragged last tile of the most loaded expert and the last rows of
    one-tile and few-tile experts; every token's row is checked on its own."""
    shape = CONFIGS[name]
    L, cfg, layer = _layer(shape)
    out = layer.forward(L["x"], update_bias=False)
    assert moe.moe_get_device_error() == 0
    o = host(out)
    assert np.all(np.isfinite(o))
    rows = tail_sample(host(layer.offsets), host(layer.token_of_row), shape.T, n_sample)
    assert len(rows) >= min(n_sample, shape.T)
    idx = host(layer.topk_idx)[rows]
    g = host(layer.topk_w)[rows].astype(np.float64)
    ref = oracle.moe_layer_tokens(host(L["x"][torch.tensor(rows, device=DEV)]), idx, g,
                                  ExpertView(L["w13"]), ExpertView(L["w2"]),
                                  ExpertView(L["ws13"]), ExpertView(L["ws2"]))
    assert_close(o[rows], ref, TOL["bf16"])


def test_layer_is_deterministic():
    shape = CONFIGS["v3_bf16"]
    L, cfg, layer = _layer(shape)
    a = layer.forward(L["x"], update_bias=False).clone()
    ya = layer.y_perm.clone()
    b = layer.forward(L["x"], update_bias=False)
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    assert torch.equal(ya.view(torch.int16), layer.y_perm.view(torch.int16))
    assert moe.moe_get_device_error() == 0


# ------------------------------------------------------------ bias update

@pytest.mark.parametrize("name,steps", [("mid_bf16", 50), ("tiny_fp32", 50), ("v3_bf16", 6)])
def test_bias_trajectory_bitwise(name, steps):
    """Route + sign-rule update, step after step on the same batch; the oracle
    follows its own bias from the device's fp32 affinities and must stay
    bitwise equal."""
    shape = CONFIGS[name]
    L = make_layer(shape, DEV, weights=False)
    cfg = moe.LayerCfg.from_shape(shape)
    T, E, K = shape.T, shape.E, shape.k
    aff = torch.empty(T, E, dtype=torch.float32, device=DEV)
    i32 = dict(dtype=torch.int32, device=DEV)
    bufs = [torch.empty(T, K, **i32), torch.empty(T, K, dtype=torch.float32, device=DEV),
            torch.empty(E, **i32), torch.empty(E + 1, **i32), torch.empty(T, K, **i32),
            torch.empty(T * K, **i32)]
    ws = torch.empty(moe.moe_workspace_bytes(cfg), dtype=torch.uint8, device=DEV)
    bias = L["bias"].clone()
    moe.moe_route(cfg, L["x"], L["router_w"], bias, *bufs, ws, affinity_out=aff)
    s32 = host(aff)
    b_or = host(L["bias"]).copy()
    spread0 = None
    for step in range(steps):
        if step:
            moe.moe_route(cfg, None, None, bias, *bufs, ws, affinity_in=aff)
        moe.moe_bias_update(cfg, bufs[2], bias)
        idx = oracle.select_experts(s32, b_or, shape.n_groups, shape.topk_groups, K)
        c = oracle.expert_load(idx, E)
        assert np.array_equal(host(bufs[2]), c), step
        if spread0 is None:
            spread0 = oracle.load_spread(c)
        b_or = oracle.bias_update(b_or, c, T, K, shape.gamma)
        assert np.array_equal(host(bias).view(np.uint32), b_or.view(np.uint32)), step
    assert moe.moe_get_device_error() == 0


# ------------------------------------------------------------------- FP8

def test_quantize_weights_fp8_bitwise():
    rng = np.random.default_rng(4)
    w = torch.tensor(rng.standard_normal((3, 300, 256)) * 0.02, dtype=torch.bfloat16,
                     device=DEV)
    w[1, :128, :128] = 0          # an all-zero block
    w[2, 5, 7] = 3.0              # an outlier
    q = torch.empty(3, 300, 256, dtype=torch.float8_e4m3fn, device=DEV)
    s = torch.empty(3, 3, 2, dtype=torch.float32, device=DEV)
    moe.moe_quantize_weights_fp8(w, q, s)
    for m in range(3):
        oq, os_ = oracle.quantize_weight_128x128(host(w[m]))
        assert np.array_equal(host(s[m]).view(np.uint32), os_.view(np.uint32))
        assert np.array_equal(q[m].float().cpu().numpy().astype(np.float64), oq)


def test_forward_into_a_given_output_buffer():
    """forward(x, out=buf) writes the same bits into buf as into the layer's
    own output buffer (the end-to-end benchmark double-buffers outputs)."""
    shape = shape_with(CONFIGS["mid_bf16"], T=300)
    L, cfg, layer = _layer(shape)
    a = layer.forward(L["x"], update_bias=False).clone()
    buf = torch.full_like(a, 3.0)
    b = layer.forward(L["x"], update_bias=False, out=buf)
    assert b.data_ptr() == buf.data_ptr()
    assert torch.equal(buf.view(torch.int16), a.view(torch.int16))
    assert moe.moe_get_device_error() == 0


@pytest.mark.parametrize("shape", [
    # the ABI's maximum of routed experts: 1024 experts in 32 groups, most
    # segments empty or a few rows long
    shape_with(CONFIGS["mid_bf16"], T=300, d=256, E=1024, n_groups=32, topk_groups=8, k=8,
               n_shared=1, inter=128),
    # d % 256 == 128 (the last down tile is half outside d), two shared experts
    shape_with(CONFIGS["mid_bf16"], T=301, d=640, E=8, n_groups=4, topk_groups=2, k=2,
               n_shared=2, inter=384),
    # the smallest bf16 sizes: d = I = 128, no shared expert
    shape_with(CONFIGS["mid_bf16"], T=130, d=128, E=16, n_groups=4, topk_groups=2, k=4,
               n_shared=0, inter=128),
    # at least 128 rows per expert on average, so the GEMMs run as pair MMAs:
    # the same half-outside last down tile and two shared experts, segments
    # with whole 256-row pair tiles and a ragged second half, and half tiles
    shape_with(CONFIGS["mid_bf16"], T=1024, d=640, E=8, n_groups=4, topk_groups=2, k=2,
               n_shared=2, inter=384),
    # pair MMAs at d = I = 128, one expert per token: half tiles whose second
    # CTA holds some of the rows, none of them, or a full tile's ragged half
    shape_with(CONFIGS["mid_bf16"], T=1400, d=128, E=4, n_groups=2, topk_groups=1, k=1,
               n_shared=0, inter=128),
], ids=lambda s: f"T{s.T}-E{s.E}-d{s.d}-I{s.inter}-Ns{s.n_shared}")
def test_layer_edge_shapes(shape):
    L, cfg, layer = _layer(shape)
    aff = torch.empty(shape.T, shape.E, dtype=torch.float32, device=DEV)
    out = layer.forward(L["x"], affinity_out=aff, update_bias=False)
    assert moe.moe_get_device_error() == 0
    r = _oracle_layer(shape, L, host(aff))
    assert np.array_equal(host(layer.topk_idx), r["topk_idx"])
    assert np.array_equal(host(layer.offsets), r["offsets"])
    assert_close(host(layer.y_perm), r["y_perm"], TOL["bf16"])
    if shape.n_shared:
        assert_close(host(layer.y_shared), r["y_shared"], TOL["bf16"])
    assert_close(host(out), r["out"], TOL["bf16"])
