"""Parity of the backward pass (bf16 kind, through the C ABI) with the fp64
backward oracle.

The forward runs first on the GPU; the oracle routes from the GPU's own fp32
affinities, so both sides hold the same selection.  Floating-point outputs
are compared by relative Frobenius error.  Tolerances: every gradient that
passes through bf16 storage (dy_perm, [da | db], h, dx_perm, dx, dW) sees a
chain of about four bf16 roundings (unit roundoff 2^-8; a uniformly
rounded tensor has relative Frobenius error about 2^-8 / sqrt(3) = 2.3e-3),
so 2e-2 leaves a margin of about four; dgate, dlogit and drouter_w are fp32
dot products of stored bf16 values, compared at 1e-4."""

import numpy as np
import pytest
import torch

import oracle
import mixture_experts_layer_82_b300 as moe
from moe_synth import CONFIGS, make_grad, make_layer, shape_with
from helpers import ExpertView, assert_close, host, rel_frobenius

pytestmark = pytest.mark.gpu

DEV = "cuda"
TOL_BF16 = 2e-2
TOL_F32 = 1e-4


def _layer(shape):
    L = make_layer(shape, DEV)
    cfg = moe.LayerCfg.from_shape(shape)
    layer = moe.MoELayer(cfg, L["router_w"], L["bias"].clone(), L["w13"], L["w2"],
                         L["ws13"] if shape.n_shared else None,
                         L["ws2"] if shape.n_shared else None)
    return L, layer


def _run(shape, L, layer, keep=True):
    """Training forward (keeping the gate/up products unless ``keep`` is
    False) and backward."""
    aff = torch.empty(shape.T, shape.E, dtype=torch.float32, device=DEV)
    layer.forward(L["x"], affinity_out=aff, update_bias=False, keep=keep)
    dout = make_grad(shape, DEV)
    layer.backward(L["x"], dout, aff)
    assert moe.moe_get_device_error() == 0
    return aff, dout


SHAPES = [
    # several M, N and K tiles, ragged segments, one shared expert, rho = 2.5
    shape_with(CONFIGS["mid_bf16"], T=300, d=256, E=16, n_groups=4, topk_groups=2, k=4,
               n_shared=1, inter=256, route_scale=2.5),
    # N tiles half outside I (384) and d (640), two shared experts
    shape_with(CONFIGS["mid_bf16"], T=301, d=640, E=8, n_groups=4, topk_groups=2, k=2,
               n_shared=2, inter=384),
    # no shared expert, many empty and one-row segments
    shape_with(CONFIGS["mid_bf16"], T=40, d=128, E=64, n_groups=8, topk_groups=4, k=6,
               n_shared=0, inter=128),
    # the mid-size workload's own widths on fewer tokens
    shape_with(CONFIGS["mid_bf16"], T=256),
    # 256 rows per expert: the forward (keeping [a | b]) and the recompute run
    # as pair MMAs; N tiles half outside I and d, two shared experts
    shape_with(CONFIGS["mid_bf16"], T=1024, d=640, E=8, n_groups=4, topk_groups=2, k=2,
               n_shared=2, inter=384),
]


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: f"T{s.T}-d{s.d}-E{s.E}-I{s.inter}-Ns{s.n_shared}")
def test_backward_matches_oracle(shape):
    L, layer = _layer(shape)
    aff, dout = _run(shape, L, layer)
    s32 = host(aff)
    ws13 = ExpertView(L["ws13"]) if shape.n_shared else None
    ws2 = ExpertView(L["ws2"]) if shape.n_shared else None
    fwd = oracle.moe_layer_forward(host(L["x"]), host(L["router_w"]), host(L["bias"]),
                                   ExpertView(L["w13"]), ExpertView(L["w2"]), ws13, ws2,
                                   n_groups=shape.n_groups, topk_groups=shape.topk_groups,
                                   k=shape.k, route_scale=shape.route_scale, affinity32=s32)
    assert np.array_equal(host(layer.topk_idx), fwd["topk_idx"])
    r = oracle.moe_layer_backward(host(L["x"]), host(L["router_w"]), ExpertView(L["w13"]),
                                  ExpertView(L["w2"]), ws13, ws2, fwd, host(dout),
                                  route_scale=shape.route_scale, affinity32=s32,
                                  y_perm=host(layer.y_perm))
    assert_close(host(layer.dgate), r["dgate"], TOL_F32)
    assert_close(host(layer.dlogit), r["dlogit"], TOL_F32)
    assert_close(host(layer.dy_perm), r["dy_perm"], TOL_BF16)
    assert_close(host(layer.dx_perm), r["dx_perm"], TOL_BF16)
    assert_close(host(layer.dx), r["dx"], TOL_BF16)
    assert_close(host(layer.drouter_w), r["drouter_w"], TOL_BF16)
    assert_close(host(layer.dw13), r["dw13"], TOL_BF16)
    assert_close(host(layer.dw2), r["dw2"], TOL_BF16)
    counts = host(layer.counts)
    assert np.all(host(layer.dw13)[counts == 0] == 0) and np.all(host(layer.dw2)[counts == 0] == 0)
    if shape.n_shared:
        assert_close(host(layer.dx_shared), r["dx_shared"], TOL_BF16)
        assert_close(host(layer.dws13), r["dws13"], TOL_BF16)
        assert_close(host(layer.dws2), r["dws2"], TOL_BF16)


def test_backward_is_deterministic():
    shape = SHAPES[0]
    L, layer = _layer(shape)
    aff, dout = _run(shape, L, layer)
    names = ("dx", "drouter_w", "dw13", "dw2", "dws13", "dws2", "dgate", "dlogit")
    first = {k: getattr(layer, k).clone() for k in names}
    _run(shape, L, layer)
    for k, v in first.items():
        bits = torch.int16 if v.dtype == torch.bfloat16 else torch.int32
        assert torch.equal(getattr(layer, k).view(bits), v.view(bits)), k


@pytest.mark.parametrize("shape", [SHAPES[1], SHAPES[4]], ids=["multicast", "pair"])
def test_kept_gate_up_products_match_recomputed(shape):
    """moe_experts_grouped_train keeps [a | b] from the forward's gate/up
    epilogue; the backward that uses them matches the one that recomputes
    them, and the training forward's own outputs equal the plain forward's
    bit for bit (both GEMM kernels: fewer and more than 128 rows per
    expert)."""
    L, layer = _layer(shape)
    _run(shape, L, layer, keep=False)
    ref = {k: getattr(layer, k).clone() for k in
           ("y_perm", "y_shared", "dx", "drouter_w", "dw13", "dw2", "dws13", "dws2")}
    _run(shape, L, layer, keep=True)
    for k in ("y_perm", "y_shared"):
        assert torch.equal(getattr(layer, k), ref[k]), k
    for k in ("dx", "drouter_w", "dw13", "dw2", "dws13", "dws2"):
        assert_close(host(getattr(layer, k)), host(ref[k]), 1e-3, k)


def test_gathering_forward_gives_the_same_backward():
    shape = SHAPES[1]
    L, layer = _layer(shape)
    aff, dout = _run(shape, L, layer, keep=False)
    ref = {k: getattr(layer, k).clone() for k in ("dx", "drouter_w", "dw13", "dw2")}
    layer.gather = True
    aff2 = torch.empty_like(aff)
    layer.forward(L["x"], affinity_out=aff2, update_bias=False)
    layer.backward(L["x"], dout, aff2)
    assert moe.moe_get_device_error() == 0
    for k, v in ref.items():
        assert torch.equal(getattr(layer, k), v), k


def _sample_units(inter, n, seed):
    return np.sort(np.random.default_rng(seed).choice(inter, size=n, replace=False))


def test_full_size_backward_on_samples():
    """The V3 shape (T = 8192, d = 7168, 256 experts, top-8, I = 2048):
    selected gradients against the oracle.  Restricting an expert to a
    subset of its hidden units gives exactly those columns of dW2 and rows
    of dW1, dW3 (each hidden unit's gradient involves only its own weights),
    so the oracle evaluates only the sampled units."""
    shape = CONFIGS["v3_bf16"]
    L, layer = _layer(shape)
    aff, dout = _run(shape, L, layer)
    T, d, E, K, I = shape.T, shape.d, shape.E, shape.k, shape.inter
    s32 = host(aff)
    idx = host(layer.topk_idx).astype(np.int64)
    ros = host(layer.row_of_slot).astype(np.int64)
    tor = host(layer.token_of_row).astype(np.int64)
    off = host(layer.offsets).astype(np.int64)
    gates = host(layer.topk_w)
    x = host(L["x"])
    go = host(dout)

    # gates -> logits on every token, from the device's dgate
    _, dl = oracle.gate_backward(s32, idx, shape.route_scale, host(layer.dgate))
    assert_close(host(layer.dlogit), dl, TOL_F32)
    # router weights on every expert
    dr = oracle.router_weight_grad(x, idx, host(layer.dlogit), E)
    assert_close(host(layer.drouter_w), dr, TOL_F32)

    # combine backward on sampled tokens
    rng = np.random.default_rng(5)
    toks = np.sort(rng.choice(T, size=32, replace=False))
    yrows = {int(r): host(layer.y_perm[int(r)]) for r in ros[toks].reshape(-1)}
    ros_s = ros[toks]
    dy_s, dg_s = oracle.combine_backward(go[toks], yrows, ros_s, gates[toks])
    assert_close(host(layer.dgate)[toks], dg_s, TOL_F32)
    got = np.stack([[host(layer.dy_perm[int(r)]) for r in row] for row in ros_s])
    assert_close(got, dy_s, TOL_BF16)

    # routed experts: the lightest non-empty, the median and the heaviest
    counts = np.diff(off)
    order = np.argsort(counts, kind="stable")
    nonempty = order[counts[order] > 0]
    for e in (int(nonempty[0]), int(nonempty[len(nonempty) // 2]), int(nonempty[-1])):
        lo, hi = int(off[e]), int(off[e + 1])
        u = x[tor[lo:hi]]
        dy = host(layer.dy_perm[lo:hi])
        w13 = host(L["w13"][e])
        w2 = host(L["w2"][e])
        units = _sample_units(I, 8, e)
        r = oracle.swiglu_ffn_backward(u, w13[units], w13[I + units], w2[:, units], dy)
        assert_close(host(layer.dw2[e])[:, units], r["dw2"], TOL_BF16, e)
        assert_close(host(layer.dw13[e])[units], r["dw1"], TOL_BF16, e)
        assert_close(host(layer.dw13[e])[I + units], r["dw3"], TOL_BF16, e)
        if hi - lo <= 256:  # the whole FFN for the input gradient of a short segment
            full = oracle.swiglu_ffn_backward(u, w13[:I], w13[I:], w2, dy)
            assert_close(host(layer.dx_perm[lo:hi]), full["du"], TOL_BF16, e)

    # shared expert: sampled hidden units over all tokens, input gradient of
    # sampled tokens
    w13 = host(L["ws13"][0])
    w2 = host(L["ws2"][0])
    units = _sample_units(I, 8, 99)
    r = oracle.swiglu_ffn_backward(x, w13[units], w13[I + units], w2[:, units], go)
    assert_close(host(layer.dws2[0])[:, units], r["dw2"], TOL_BF16)
    assert_close(host(layer.dws13[0])[units], r["dw1"], TOL_BF16)
    assert_close(host(layer.dws13[0])[I + units], r["dw3"], TOL_BF16)
    full = oracle.swiglu_ffn_backward(x[toks], w13[:I], w13[I:], w2, go[toks])
    assert_close(host(layer.dx_shared)[toks], full["du"], TOL_BF16)

    # the input gradient of sampled tokens from the device's expert parts
    dxp = {int(r): host(layer.dx_perm[int(r)]) for r in ros_s.reshape(-1)}
    dx_s = oracle.input_grad(host(layer.dx_shared)[toks], dxp, ros_s, idx[toks],
                             host(layer.dlogit)[toks], host(L["router_w"]))
    assert_close(host(layer.dx)[toks], dx_s, TOL_BF16)
