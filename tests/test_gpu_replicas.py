"""The layer's data-parallel load exchange on one GPU: with a process group
of one replica the all-reduced loads are the local loads, so the bias
update must equal the ungrouped one bit for bit (the exchange itself is
checked with two CPU ranks in test_multiprocess.py)."""

import socket

import pytest
import torch
import torch.distributed as dist

import mixture_experts_layer_82_b300 as moe
from moe_synth import CONFIGS, make_layer, shape_with

pytestmark = pytest.mark.gpu


def _port():
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_forward_with_a_one_replica_load_group():
    shape = shape_with(CONFIGS["mid_bf16"], T=300)
    L = make_layer(shape, "cuda")
    cfg = moe.LayerCfg.from_shape(shape)
    mk = lambda: moe.MoELayer(cfg, L["router_w"], L["bias"].clone(), L["w13"], L["w2"],
                              L["ws13"], L["ws2"])
    a, b = mk(), mk()
    a.forward(L["x"])
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{_port()}", rank=0,
                            world_size=1)
    try:
        b.forward(L["x"], load_group=dist.group.WORLD)
    finally:
        dist.destroy_process_group()
    assert moe.moe_get_device_error() == 0
    assert torch.equal(a.counts, b.counts)
    assert torch.equal(a.bias.view(torch.int32), b.bias.view(torch.int32))
    assert torch.equal(a.out.view(torch.int16), b.out.view(torch.int16))


def test_load_group_on_a_stream_that_is_not_current():
    """forward(stream=s, load_group=g) with s not torch's current stream: the
    all-reduce of the loads must run in s's order (after the routing that
    writes them, before the bias update that reads them).  Two steps on
    different batches, so stale loads of the first step would show in the
    second."""
    shape = shape_with(CONFIGS["mid_bf16"], T=300)
    L = make_layer(shape, "cuda")
    x2 = torch.flip(L["x"], dims=[0]).contiguous() * 1.5
    cfg = moe.LayerCfg.from_shape(shape)
    mk = lambda: moe.MoELayer(cfg, L["router_w"], L["bias"].clone(), L["w13"], L["w2"],
                              L["ws13"], L["ws2"])
    a, b = mk(), mk()
    for x in (L["x"], x2):
        a.forward(x)
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{_port()}", rank=0,
                            world_size=1)
    try:
        for x in (L["x"], x2):
            b.forward(x, stream=s, load_group=dist.group.WORLD)
        s.synchronize()
    finally:
        dist.destroy_process_group()
    assert moe.moe_get_device_error() == 0
    assert torch.equal(a.counts, b.counts)
    assert torch.equal(a.bias.view(torch.int32), b.bias.view(torch.int32))
    assert torch.equal(a.out.view(torch.int16), b.out.view(torch.int16))
