"""Pins of the backward oracle against facts that do not come from its own
derivation: central finite differences of the (separately pinned) forward
oracle with the top-K selection held fixed, the scale invariance of
normalised gates, and the vanishing router gradient when one expert is
selected."""

import numpy as np
import pytest

import oracle
from moe_synth import CONFIGS, make_layer, shape_with

TINY = shape_with(CONFIGS["tiny_fp32"], T=6, d=16, E=8, n_groups=4, topk_groups=2, k=3,
                  n_shared=2, inter=8, route_scale=2.5, seed=11)


def _np(t):
    return None if t is None else t.double().numpy()


def _setup(shape):
    L = make_layer(shape)
    P = {k: _np(v) for k, v in L.items()}
    fwd = oracle.moe_layer_forward(P["x"], P["router_w"], P["bias"], P["w13"], P["w2"],
                                   P["ws13"] if shape.n_shared else None,
                                   P["ws2"] if shape.n_shared else None,
                                   n_groups=shape.n_groups, topk_groups=shape.topk_groups,
                                   k=shape.k, route_scale=shape.route_scale)
    rng = np.random.default_rng(shape.seed + 1)
    dout = rng.standard_normal((shape.T, shape.d))
    return P, fwd, dout


def _loss(P, idx, dout, rho, n_shared):
    """sum(dout * layer output) with the selection ``idx`` fixed, built only
    from forward-oracle pieces; affinities in fp64 (no fp32 rounding, so
    that finite differences see a smooth function)."""
    s = oracle.sigmoid_affinity(P["x"], P["router_w"])
    gates = oracle.gating_weights(s, idx, rho)
    _, offsets, ros, tor = oracle.segment_layout(idx, P["router_w"].shape[0])
    xp = oracle.permute_rows(P["x"], tor)
    inter = P["w13"].shape[1] // 2
    yp = np.zeros((xp.shape[0], P["x"].shape[1]))
    for e in range(P["router_w"].shape[0]):
        lo, hi = int(offsets[e]), int(offsets[e + 1])
        if hi > lo:
            w = P["w13"][e]
            yp[lo:hi] = oracle.swiglu_ffn(xp[lo:hi], w[:inter], w[inter:], P["w2"][e])
    ys = None
    if n_shared:
        ys = sum(oracle.swiglu_ffn(P["x"], P["ws13"][s][:inter], P["ws13"][s][inter:], P["ws2"][s])
                 for s in range(n_shared))
    return float((dout * oracle.combine(ys, yp, ros, gates)).sum())


def _backward(P, fwd, dout, shape):
    # gates from the fp64 affinities, as in _loss
    return oracle.moe_layer_backward(P["x"], P["router_w"], P["w13"], P["w2"],
                                     P["ws13"] if shape.n_shared else None,
                                     P["ws2"] if shape.n_shared else None,
                                     dict(fwd, topk_w=oracle.gating_weights(
                                         fwd["affinity"], fwd["topk_idx"], shape.route_scale)),
                                     dout, route_scale=shape.route_scale,
                                     affinity32=None)


@pytest.mark.parametrize("name,grad", [("x", "dx"), ("router_w", "drouter_w"), ("w13", "dw13"),
                                       ("w2", "dw2"), ("ws13", "dws13"), ("ws2", "dws2")])
def test_gradients_match_central_differences(name, grad):
    shape = TINY
    P, fwd, dout = _setup(shape)
    # the backward under test takes its gates from fp64 affinities here
    bwd = oracle.moe_layer_backward(P["x"], P["router_w"], P["w13"], P["w2"], P["ws13"], P["ws2"],
                                    dict(fwd, topk_w=oracle.gating_weights(
                                        fwd["affinity"], fwd["topk_idx"], shape.route_scale)),
                                    dout, route_scale=shape.route_scale,
                                    affinity32=fwd["affinity"])
    idx = fwd["topk_idx"]
    rng = np.random.default_rng(7)
    arr = P[name]
    flat = arr.reshape(-1)
    picks = rng.choice(flat.size, size=min(60, flat.size), replace=False)
    eps = 1e-6
    for i in picks:
        keep = flat[i]
        flat[i] = keep + eps
        lp = _loss(P, idx, dout, shape.route_scale, shape.n_shared)
        flat[i] = keep - eps
        lm = _loss(P, idx, dout, shape.route_scale, shape.n_shared)
        flat[i] = keep
        fd = (lp - lm) / (2 * eps)
        an = bwd[grad].reshape(-1)[i]
        assert abs(fd - an) <= 1e-6 * max(1.0, abs(fd)), (name, i, fd, an)


def test_dgate_and_dy_perm_against_differences_of_the_gates():
    shape = TINY
    P, fwd, dout = _setup(shape)
    bwd = _backward(P, fwd, dout, shape)
    # d(sum dout * out)/d g[t, j] is the dot product of dout[t] with the
    # routed row: perturb one gate of the combine directly
    ros, yp = fwd["row_of_slot"], fwd["y_perm"]
    gates = oracle.gating_weights(fwd["affinity"], fwd["topk_idx"], shape.route_scale)
    for t in range(shape.T):
        for j in range(shape.k):
            g2 = gates.copy()
            g2[t, j] += 1.0  # the combine is linear in every gate
            diff = (dout * (oracle.combine(None, yp, ros, g2) - oracle.combine(None, yp, ros, gates))).sum()
            assert abs(diff - bwd["dgate"][t, j]) < 1e-12 * max(1.0, abs(diff))
            np.testing.assert_allclose(bwd["dy_perm"][ros[t, j]], gates[t, j] * dout[t], rtol=1e-15)


def test_normalised_gates_are_scale_invariant():
    # g = rho s / sum(s) does not change when all selected s are scaled,
    # so sum_j dL/ds_j s_j = 0 for every token
    rng = np.random.default_rng(3)
    T, E, K = 20, 12, 4
    s = rng.uniform(0.05, 0.95, size=(T, E))
    idx = np.stack([rng.choice(E, size=K, replace=False) for _ in range(T)])
    dg = rng.standard_normal((T, K))
    ds, dl = oracle.gate_backward(s, idx, 2.5, dg)
    sel = np.take_along_axis(s, idx, axis=1)
    assert np.abs((ds * sel).sum(axis=1)).max() < 1e-12
    np.testing.assert_allclose(dl, ds * sel * (1 - sel), rtol=1e-15)


def test_one_selected_expert_gives_no_router_gradient():
    # K = 1: the normalised gate is the constant rho whatever the affinity
    shape = shape_with(TINY, k=1, n_groups=1, topk_groups=1)
    P, fwd, dout = _setup(shape)
    bwd = _backward(P, fwd, dout, shape)
    assert np.abs(bwd["dlogit"]).max() < 1e-15
    assert np.abs(bwd["drouter_w"]).max() < 1e-15


def test_swiglu_backward_closed_form_point():
    # one row, one hidden unit: a = 0 gives silu(0) = 0 and silu'(0) = 1/2
    u = np.array([[1.0, 0.0]])
    w1 = np.array([[0.0, 3.0]])      # a = 0
    w3 = np.array([[2.0, 0.0]])      # b = 2
    w2 = np.array([[1.0], [0.0]])    # y = [h, 0]
    r = oracle.swiglu_ffn_backward(u, w1, w3, w2, np.array([[1.0, 5.0]]))
    assert r["h"][0, 0] == 0.0
    assert r["dh"][0, 0] == 1.0
    assert r["da"][0, 0] == 1.0      # dh * b * 1/2
    assert r["db"][0, 0] == 0.0
    np.testing.assert_allclose(r["du"], [[0.0, 3.0]])   # da * w1
    np.testing.assert_allclose(r["dw1"], [[1.0, 0.0]])  # da * u
    assert np.all(r["dw2"] == 0.0)                       # h = 0
