"""moe_route_static_scratch: routing for callers that cannot allocate device
memory (for instance a plugin inside a serving engine that has reserved all
device memory for its own pool and offers no allocator).  Its scratch is a
fixed array inside the library, so it takes no workspace; its results must
equal those of moe_route, which uses a caller-provided workspace.

The file is named to be collected last, so that a run that stops at the
first failure has already run every other test.  It must pass both alone in
a fresh process (the first call on the device looks up the array's address)
and after the other tests."""

import ctypes

import pytest
import torch

import mixture_experts_layer_82_b300 as moe
from moe_synth import CONFIGS, make_layer, shape_with

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _outputs(shape):
    T, E, K = shape.T, shape.E, shape.k
    i32 = dict(dtype=torch.int32, device=DEV)
    return dict(topk_idx=torch.full((T, K), -1, **i32),
                topk_w=torch.full((T, K), -1.0, dtype=torch.float32, device=DEV),
                counts=torch.full((E,), -1, **i32), offsets=torch.full((E + 1,), -1, **i32),
                row_of_slot=torch.full((T, K), -1, **i32),
                token_of_row=torch.full((T * K,), -1, **i32))


def _same(a, b):
    for k in ("topk_idx", "counts", "offsets", "row_of_slot", "token_of_row"):
        assert torch.equal(a[k], b[k]), k
    # same kernels on the same inputs: the gates agree to the last bit, far
    # inside the 1e-6 relative tolerance the routing tests use
    torch.testing.assert_close(a["topk_w"], b["topk_w"], rtol=1e-6, atol=0)


@pytest.mark.parametrize("shape", [CONFIGS["v3_bf16"], CONFIGS["tiny_fp32"],
                                   shape_with(CONFIGS["mid_bf16"], T=1001)],
                         ids=lambda s: f"{s.name}-T{s.T}")
def test_static_scratch_route_matches_moe_route_on_two_calls(shape):
    L = make_layer(shape, DEV, weights=False)
    cfg = moe.LayerCfg.from_shape(shape)
    ws = torch.empty(moe.moe_workspace_bytes(cfg), dtype=torch.uint8, device=DEV)
    bias2 = L["bias"] + torch.linspace(-0.05, 0.05, shape.E, device=DEV)
    for call, bias in enumerate((L["bias"], bias2)):
        ref, got = _outputs(shape), _outputs(shape)
        moe.moe_route(cfg, L["x"], L["router_w"], bias, ws=ws, **ref)
        # first call: affinities in the static scratch; second: kept by the caller
        aff = None if call == 0 else torch.empty(shape.T, shape.E, device=DEV)
        moe.moe_route_static_scratch(cfg, L["x"], L["router_w"], bias, affinity_out=aff, **got)
        torch.cuda.synchronize()
        assert moe.moe_get_device_error() == 0
        _same(ref, got)


def test_static_scratch_rejects_shapes_beyond_its_size():
    shape = shape_with(CONFIGS["v3_bf16"], T=65536)   # 64 MiB of affinities
    cfg = moe.LayerCfg.from_shape(shape)
    lib = moe.library()
    p = [0x100000 * (i + 1) for i in range(11)]       # checked, never dereferenced
    p[3] = p[4] = None                                # no affinity_in / affinity_out
    status = lib.moe_route_static_scratch(ctypes.byref(cfg.c()), *p, None)
    assert status == 7  # MOE_ERR_WORKSPACE, nothing launched
