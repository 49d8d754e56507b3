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
