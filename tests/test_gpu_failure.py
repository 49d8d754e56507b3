"""Failure detection without a GPU fault: a device wait that runs out and an
index out of range are reported through the error word, nothing traps, and
the device stays usable afterwards."""

import pytest
import torch

import mixture_experts_layer_82_b300 as moe
from moe_synth import CONFIGS, make_layer, shape_with

pytestmark = pytest.mark.gpu
DEV = "cuda"
MOE_ERR_TIMEOUT, MOE_ERR_DEVICE = 5, 6


def _route_ok(shape):
    L = make_layer(shape, DEV, weights=False)
    cfg = moe.LayerCfg.from_shape(shape)
    T, E, K = shape.T, shape.E, shape.k
    i32 = dict(dtype=torch.int32, device=DEV)
    bufs = [torch.empty(T, K, **i32), torch.empty(T, K, dtype=torch.float32, device=DEV),
            torch.empty(E, **i32), torch.empty(E + 1, **i32), torch.empty(T, K, **i32),
            torch.empty(T * K, **i32)]
    ws = torch.empty(moe.moe_workspace_bytes(cfg), dtype=torch.uint8, device=DEV)
    moe.moe_route(cfg, L["x"], L["router_w"], L["bias"], *bufs, ws)
    assert moe.moe_get_device_error() == 0
    assert int(bufs[2].sum()) == T * K
    return L, cfg, bufs


def test_wait_that_runs_out_is_reported():
    assert moe.moe_get_device_error() == 0
    moe.moe_selftest_wait(20_000_000)  # 20 ms
    assert moe.moe_get_device_error() == MOE_ERR_TIMEOUT
    assert moe.moe_get_device_error() == 0  # read and cleared
    _route_ok(shape_with(CONFIGS["mid_bf16"], T=200))


def test_selftest_rejects_bad_limits():
    for bad in (0, -5, 10 ** 11):
        with pytest.raises(moe.MoeError):
            moe.moe_selftest_wait(bad)


def test_index_out_of_range_is_reported_and_skipped():
    shape = shape_with(CONFIGS["mid_bf16"], T=200)
    L, cfg, bufs = _route_ok(shape)
    tor = bufs[5].clone()
    tor[7] = shape.T        # one row points past the last token
    x_perm = torch.zeros(shape.T * shape.k, shape.d, dtype=torch.bfloat16, device=DEV)
    moe.moe_permute(cfg, L["x"], tor, x_perm)
    assert moe.moe_get_device_error() == MOE_ERR_DEVICE
    assert torch.count_nonzero(x_perm[7]) == 0   # the bad row was skipped
    ok = bufs[5][8].item()
    assert torch.equal(x_perm[8], L["x"][ok])    # the others were copied
    _route_ok(shape)


@pytest.mark.parametrize("kind", ["fp32", "bf16", "fp8"])
def test_bad_segment_offsets_are_reported_and_skipped(kind):
    """moe_experts_grouped with offsets that are not a valid segment layout:
    offsets[E] past T * K (the last expert's segment would leave y_perm) and
    a negative offsets[3] (experts 2 and 3 run backwards / start before row
    0).  The call must report MOE_ERR_DEVICE, treat those experts as empty,
    write nothing outside its buffers (guard rows around y_perm and guard
    bytes after the workspace stay intact) and give every valid expert the
    rows it gets from the valid offsets."""
    base = {"fp32": CONFIGS["tiny_fp32"], "bf16": CONFIGS["mid_bf16"],
            "fp8": CONFIGS["v3_fp8"]}[kind]
    shape = shape_with(base, T=200) if kind != "fp8" else shape_with(
        base, T=96, d=512, E=16, n_groups=8, topk_groups=4, k=4, inter=256,
        router="gaussian", outlier_channels=5)
    L = make_layer(shape, DEV)
    cfg = moe.LayerCfg.from_shape(shape)
    layer = moe.MoELayer(cfg, L["router_w"], L["bias"].clone(), L["w13"], L["w2"],
                         L["ws13"], L["ws2"])
    layer.forward(L["x"], update_bias=False)
    assert moe.moe_get_device_error() == 0
    T, E, K, d = shape.T, shape.E, shape.k, shape.d
    ref = layer.y_perm.clone()
    good = layer.offsets.clone()
    bad = good.clone()
    bad[E] = T * K + 128
    bad[3] = -5
    G = 256  # guard rows before and after y_perm
    buf = torch.full((G + T * K + G, d), 7.0, dtype=ref.dtype, device=DEV)
    y_perm = buf[G:G + T * K]
    nws = layer.ws.numel()
    ws_big = torch.full((nws + 4096,), 0x5A, dtype=torch.uint8, device=DEV)
    y_shared = torch.empty_like(layer.y_shared)
    shared_in = layer.x_q if kind == "fp8" else L["x"]
    moe.moe_experts_grouped(cfg, layer.x_perm, shared_in, bad, layer.w13, layer.w2, layer.ws13,
                            layer.ws2, y_perm, y_shared, ws_big[:nws],
                            x_perm_scales=layer.x_perm_s, x_scales=layer.x_q_s,
                            w13_scales=layer.w13_s, w2_scales=layer.w2_s,
                            ws13_scales=layer.ws13_s, ws2_scales=layer.ws2_s)
    assert moe.moe_get_device_error() == MOE_ERR_DEVICE
    assert torch.all(buf[:G] == 7.0) and torch.all(buf[G + T * K:] == 7.0)
    assert torch.all(ws_big[nws:] == 0x5A)
    off = good.cpu().tolist()
    for e in range(E):
        if e in (2, 3, E - 1):
            continue
        lo, hi = off[e], off[e + 1]
        assert torch.equal(y_perm[lo:hi], ref[lo:hi]), e
    assert torch.equal(y_shared, layer.y_shared)
    _route_ok(shape_with(CONFIGS["mid_bf16"], T=200))
