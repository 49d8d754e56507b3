"""Pins of the CPU oracle against facts that do not come from the oracle:
hand-derived examples, brute force on tiny inputs, closed forms,
invariants, and library routines for special cases."""

import itertools
import math
import os

import numpy as np
import pytest
import scipy.special
import torch

import oracle
from oracle import moe_fp8
from moe_synth import CONFIGS, make_layer, shape_with

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _read_kv(name):
    out = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, *vals = line.split()
            out[key] = vals
    return out


# ----------------------------------------------------------------- affinity

def test_affinity_closed_forms():
    # u . e = 0 -> 1/2 ; u . e = ln 3 -> 3/4 ; u . e = -ln 3 -> 1/4
    u = np.array([[1.0, 0.0]])
    e = np.array([[0.0, 1.0], [math.log(3.0), 0.0], [-math.log(3.0), 5.0]])
    s = oracle.sigmoid_affinity(u, e)
    assert s[0, 0] == 0.5
    assert abs(s[0, 1] - 0.75) < 1e-15
    assert abs(s[0, 2] - 0.25) < 1e-15


def test_affinity_matches_library_and_symmetry():
    rng = np.random.default_rng(0)
    u = rng.standard_normal((7, 5))
    e = rng.standard_normal((3, 5))
    s = oracle.sigmoid_affinity(u, e)
    np.testing.assert_allclose(s, scipy.special.expit(u @ e.T), rtol=1e-14)
    np.testing.assert_allclose(s + oracle.sigmoid_affinity(-u, e), 1.0, atol=1e-15)


# ---------------------------------------------------------------- selection

def test_routing_hand_example():
    g = _read_kv("routing_hand_example.txt")
    s = np.array([[float(v) for v in g["s"]]], dtype=np.float32)
    b = np.array([float(v) for v in g["b"]], dtype=np.float32)
    idx = oracle.select_experts(s, b, int(g["groups"][0]), int(g["keep_groups"][0]),
                                int(g["K"][0]))
    assert idx[0].tolist() == [int(v) for v in g["expect_idx"]]
    gates = oracle.gating_weights(s, idx)
    den = float(g["expect_gate_den"][0])
    np.testing.assert_allclose(gates[0], [float(v) / den for v in g["expect_gate_num"]],
                               rtol=1e-15)


def _dominates(a, b, val):
    """Expert/group a ranks above b: larger value, or equal and lower index."""
    return val[a] > val[b] or (val[a] == val[b] and a < b)


def _brute_force_select(biased, n_groups, keep, k, topn):
    """Selection by enumeration: the kept group set is the unique subset whose
    every member dominates every non-member under the group score; the
    expert set likewise inside the kept groups.  The group score is the
    largest fp32 sum over the allowed subsets of topn members."""
    E = biased.shape[0]
    per = E // n_groups
    topn = min(topn, per)
    gscore = np.zeros(n_groups, dtype=np.float32)
    for g in range(n_groups):
        members = range(g * per, (g + 1) * per)
        best = None
        for sub in itertools.combinations(members, topn):
            vals = sorted((biased[i] for i in sub), reverse=True)
            acc = np.float32(0)
            for v in vals:
                acc = np.float32(acc + v)
            best = acc if best is None or acc > best else best
        gscore[g] = best
    chosen = None
    for sub in itertools.combinations(range(n_groups), keep):
        rest = [g for g in range(n_groups) if g not in sub]
        if all(_dominates(a, b, gscore) for a in sub for b in rest):
            assert chosen is None
            chosen = sub
    cand = [i for g in chosen for i in range(g * per, (g + 1) * per)]
    pick = None
    for sub in itertools.combinations(cand, k):
        rest = [i for i in cand if i not in sub]
        if all(_dominates(a, b, biased) for a in sub for b in rest):
            assert pick is None
            pick = sub
    # listing order: pairwise dominance
    return sorted(pick, key=lambda i: (-float(biased[i]), i))


@pytest.mark.parametrize("E,G,keep,k,seed,ties", [
    (16, 4, 2, 2, 0, False), (16, 4, 2, 2, 1, True), (8, 2, 1, 3, 2, True),
    (12, 3, 2, 4, 3, False), (12, 4, 3, 5, 4, True), (6, 1, 1, 2, 5, True),
    (8, 8, 3, 3, 6, True), (16, 4, 2, 2, 7, True),
])
def test_selection_brute_force(E, G, keep, k, seed, ties):
    rng = np.random.default_rng(seed)
    T = 24
    s = rng.random((T, E)).astype(np.float32)
    b = (rng.random(E).astype(np.float32) - 0.5) * 0.2
    if ties:
        # saturated sigmoids: many exact 1.0f and repeated values
        s[rng.random((T, E)) < 0.4] = np.float32(1.0)
        s[:, ::3] = s[:, 1::3][:, : s[:, ::3].shape[1]] if E % 3 == 0 else s[:, ::3]
        b[:] = np.where(rng.random(E) < 0.5, 0.0, b)
    idx = oracle.select_experts(s, b, G, keep, k)
    biased = oracle.biased_scores(s, b)
    for t in range(T):
        assert idx[t].tolist() == _brute_force_select(biased[t], G, keep, k, 2)


def test_group_score_is_best_pair_sum():
    rng = np.random.default_rng(11)
    biased = rng.standard_normal((5, 32)).astype(np.float32)
    gs = oracle.group_scores(biased, 4, 2)
    for t in range(5):
        for g in range(4):
            vals = biased[t, g * 8:(g + 1) * 8]
            best = max(np.float32(vals[i] + vals[j]) for i in range(8) for j in range(8) if i != j)
            assert gs[t, g] == best


def test_selection_respects_group_limit_and_bias_only_for_choice():
    shape = CONFIGS["tiny_fp32"]
    L = make_layer(shape, "cpu", weights=False)
    s = oracle.sigmoid_affinity(L["x"].numpy(), L["router_w"].numpy()).astype(np.float32)
    b = L["bias"].numpy()
    idx = oracle.select_experts(s, b, shape.n_groups, shape.topk_groups, shape.k)
    per = shape.E // shape.n_groups
    for t in range(shape.T):
        assert len(set(idx[t].tolist())) == shape.k
        assert len(set((idx[t] // per).tolist())) <= shape.topk_groups
    g = oracle.gating_weights(s, idx, 1.0)
    s64 = s.astype(np.float64)
    sel = s64[np.arange(shape.T)[:, None], idx]
    np.testing.assert_allclose(g, sel / sel.sum(1, keepdims=True), rtol=1e-12)


@pytest.mark.parametrize("rho", [1.0, 2.5])
def test_gates_sum_to_route_scale(rho):
    rng = np.random.default_rng(3)
    s = rng.random((50, 16)).astype(np.float32)
    idx = oracle.select_experts(s, np.zeros(16, np.float32), 4, 2, 3)
    g = oracle.gating_weights(s, idx, rho)
    assert np.all(g >= 0)
    np.testing.assert_allclose(g.sum(1), rho, rtol=1e-12)


# ---------------------------------------------------------- permute/combine

def test_segment_layout_invariants():
    rng = np.random.default_rng(5)
    T, E, k = 40, 12, 3
    idx = np.stack([rng.choice(E, k, replace=False) for _ in range(T)]).astype(np.int32)
    counts, offsets, ros, tor = oracle.segment_layout(idx, E)
    assert counts.sum() == T * k
    assert offsets[0] == 0 and np.all(np.diff(offsets) == counts)
    assert sorted(ros.reshape(-1).tolist()) == list(range(T * k))
    for t in range(T):
        for j in range(k):
            r = ros[t, j]
            assert tor[r] == t
            assert offsets[idx[t, j]] <= r < offsets[idx[t, j] + 1]
    for e in range(E):
        seg = tor[offsets[e]:offsets[e + 1]]
        assert np.all(np.diff(seg) > 0)  # ascending token order


def test_permute_combine_identity():
    rng = np.random.default_rng(6)
    T, E, k, d = 30, 8, 3, 5
    x = rng.standard_normal((T, d))
    idx = np.stack([rng.choice(E, k, replace=False) for _ in range(T)]).astype(np.int32)
    _, _, ros, tor = oracle.segment_layout(idx, E)
    xp = oracle.permute_rows(x, tor)
    for t in range(T):
        for j in range(k):
            assert np.array_equal(xp[ros[t, j]], x[t])
    out = oracle.combine(None, xp, ros, np.ones((T, k)))
    assert np.array_equal(out, k * x)


# ------------------------------------------------------------------ experts

def test_silu_closed_forms_and_library():
    assert oracle.silu(0.0) == 0.0
    assert abs(oracle.silu(math.log(3.0)) - 0.75 * math.log(3.0)) < 1e-15
    a = np.linspace(-9, 9, 101)
    np.testing.assert_allclose(oracle.silu(a) - oracle.silu(-a), a, atol=1e-14)
    np.testing.assert_allclose(oracle.silu(a),
                               torch.nn.functional.silu(torch.tensor(a)).numpy(), rtol=1e-14)


def test_swiglu_selection_weights_closed_form():
    # d = 3, I = 2: W1 picks (x1, x0), W3 picks (x0, x2), W2 sends h0 -> out0
    # and h1 -> out2.  out = [silu(x1) x0, 0, silu(x0) x2].  A transposed or
    # swapped operand breaks either the shapes or the mapping.
    x = np.array([[0.7, -1.3, 2.0]])
    w1 = np.array([[0, 1, 0], [1, 0, 0]], float)
    w3 = np.array([[1, 0, 0], [0, 0, 1]], float)
    w2 = np.array([[1, 0], [0, 0], [0, 1]], float)
    y = oracle.swiglu_ffn(x, w1, w3, w2)
    sl = lambda a: a / (1 + math.exp(-a))
    np.testing.assert_allclose(y[0], [sl(-1.3) * 0.7, 0.0, sl(0.7) * 2.0], rtol=1e-15)


def _dense_case(E, n_shared, seed=0):
    rng = np.random.default_rng(seed)
    T, d, inter = 9, 12, 6
    x = rng.standard_normal((T, d))
    rw = rng.standard_normal((E, d)) * 0.3
    w13 = rng.standard_normal((E, 2 * inter, d)) * 0.2
    w2 = rng.standard_normal((E, d, inter)) * 0.2
    ws13 = np.repeat(w13[:1], n_shared, axis=0)
    ws2 = np.repeat(w2[:1], n_shared, axis=0)
    return x, rw, w13, w2, ws13, ws2, inter


def test_dense_reduction_one_expert():
    x, rw, w13, w2, _, _, inter = _dense_case(1, 0)
    r = oracle.moe_layer_forward(x, rw, np.zeros(1, np.float32), w13, w2, None, None,
                                 n_groups=1, topk_groups=1, k=1)
    assert np.all(r["topk_w"] == 1.0)
    dense = oracle.swiglu_ffn(x, w13[0, :inter], w13[0, inter:], w2[0])
    np.testing.assert_allclose(r["out"], dense, rtol=1e-13, atol=1e-15)
    # with the same weights also as one shared expert the output doubles
    x, rw, w13, w2, ws13, ws2, _ = _dense_case(1, 1)
    r2 = oracle.moe_layer_forward(x, rw, np.zeros(1, np.float32), w13, w2, ws13, ws2,
                                  n_groups=1, topk_groups=1, k=1)
    np.testing.assert_allclose(r2["out"], 2 * dense, rtol=1e-13, atol=1e-15)


def test_layer_is_linear_in_down_projection_and_gates():
    shape = shape_with(CONFIGS["tiny_fp32"], T=16)
    L = make_layer(shape, "cpu")
    args = dict(n_groups=shape.n_groups, topk_groups=shape.topk_groups, k=shape.k)
    r1 = oracle.moe_layer_forward(L["x"].numpy(), L["router_w"].numpy(), L["bias"].numpy(),
                                  L["w13"].numpy(), L["w2"].numpy(), L["ws13"].numpy(),
                                  L["ws2"].numpy(), route_scale=1.0, **args)
    r2 = oracle.moe_layer_forward(L["x"].numpy(), L["router_w"].numpy(), L["bias"].numpy(),
                                  L["w13"].numpy(), 3 * L["w2"].numpy().astype(np.float64),
                                  L["ws13"].numpy(), 3 * L["ws2"].numpy().astype(np.float64),
                                  route_scale=1.0, **args)
    np.testing.assert_allclose(r2["out"], 3 * r1["out"], rtol=1e-12, atol=1e-14)
    r3 = oracle.moe_layer_forward(L["x"].numpy(), L["router_w"].numpy(), L["bias"].numpy(),
                                  L["w13"].numpy(), L["w2"].numpy(), None, None,
                                  route_scale=2.0, **args)
    np.testing.assert_allclose(r3["out"], 2 * (r1["out"] - r1["y_shared"]), rtol=1e-12,
                               atol=1e-14)
    # the bias never enters the gate values, only the choice
    np.testing.assert_allclose(r1["topk_w"].sum(1), 1.0, rtol=1e-12)


# ------------------------------------------------------------- bias update

def test_bias_update_hand_example():
    g = _read_kv("routing_hand_example.txt")
    counts = np.array([int(v) for v in g["counts"]])
    b0 = np.array([float(v) for v in g["bias_before"]], np.float32)
    b1 = oracle.bias_update(b0, counts, int(g["tokens"][0]), int(g["K"][0]),
                            float(g["gamma"][0]))
    assert b1.tolist() == [float(v) for v in g["bias_after"]]


def test_bias_update_moves_by_exactly_gamma():
    rng = np.random.default_rng(8)
    E, T, k, gamma = 64, 100, 6, 1e-3
    b = (rng.random(E).astype(np.float32) - 0.5)
    counts = rng.integers(0, 20, E)
    counts[0] = T * k // E if (T * k) % E == 0 else counts[0]
    b1 = oracle.bias_update(b, counts, T, k, gamma)
    g32 = np.float32(gamma)
    mean = T * k / E
    for i in range(E):
        if counts[i] > mean:
            assert b1[i] == np.float32(b[i] - g32) and b1[i] < b[i]
        else:
            assert b1[i] == np.float32(b[i] + g32) and b1[i] > b[i]
    # sign is opposite to (load - mean)
    assert np.all(np.sign(b1 - b) == np.where(counts * E > T * k, -1, 1))


def test_bias_trajectory_piecewise_multiples_of_gamma():
    gamma = 2.0 ** -10  # exact in fp32 so the trajectory is exact
    b = np.zeros(4, np.float32)
    loads = [np.array([9, 1, 3, 3]), np.array([9, 1, 3, 3]), np.array([2, 8, 3, 3])]
    for c in loads:
        b = oracle.bias_update(b, c, 8, 2, gamma)
    assert b.tolist() == [-gamma, gamma, 3 * gamma, 3 * gamma]


# --------------------------------------------------------------------- FP8

def _all_finite_bf16():
    bits = torch.arange(0, 1 << 16, dtype=torch.int32).to(torch.int16)
    v = bits.view(torch.bfloat16).float()
    return v[torch.isfinite(v)]


def test_e4m3_round_matches_library_cast():
    v = _all_finite_bf16()
    v = v[v.abs() < 464]  # beyond that the library cast gives NaN, not saturation
    ours = oracle.e4m3_round(v.double().numpy())
    ref = v.to(torch.float8_e4m3fn).double().numpy()
    assert np.array_equal(ours, ref)


def test_e4m3_saturates_and_decode_table():
    assert oracle.e4m3_round(1e6) == 448.0 and oracle.e4m3_round(-500.0) == -448.0
    assert oracle.E4M3_MAX == 448.0
    codes = np.arange(256)
    ours = oracle.e4m3_decode(codes)
    ref = torch.tensor(codes, dtype=torch.uint8).view(torch.float8_e4m3fn).double().numpy()
    finite = ~np.isnan(ref)
    assert np.array_equal(np.isnan(ours), np.isnan(ref))
    assert np.array_equal(ours[finite], ref[finite])
    assert np.nanmax(ours) == 448.0 and np.nanmin(np.abs(ours[ours != 0])) == 2.0 ** -9
    # encode inverts decode on every finite code (the two zeros included)
    fin = codes[finite]
    assert np.array_equal(oracle.e4m3_encode(ours[finite]), fin.astype(np.uint8))


def test_fp8_quantisers_scale_and_range():
    rng = np.random.default_rng(9)
    x = (rng.standard_normal((3, 256)) * 5).astype(np.float32)
    x[1, :128] = 0.0
    q, s = oracle.quantize_act_1x128(x)
    assert s.shape == (3, 2) and s.dtype == np.float32
    assert s[1, 0] == 1.0 and np.all(q[1, :128] == 0)
    for r in range(3):
        for kb in range(2):
            tile = x[r, kb * 128:(kb + 1) * 128]
            amax = np.max(np.abs(tile))
            if amax:
                assert s[r, kb] == np.float32(amax / np.float32(448))
                assert np.max(np.abs(q[r, kb * 128:(kb + 1) * 128])) >= 416  # near the top code
    assert np.all(np.abs(q) <= 448)
    deq = oracle.dequantize_act_1x128(q, s)
    assert np.max(np.abs(deq - x) / (np.abs(x) + 1e-30) * (np.abs(x) > 0.1 * np.abs(x).max())) < 2 ** -3
    w = (rng.standard_normal((200, 256)) * 0.02).astype(np.float32)
    qw, sw = oracle.quantize_weight_128x128(w)
    assert sw.shape == (2, 2)
    assert sw[1, 1] == np.float32(np.max(np.abs(w[128:, 128:])) / np.float32(448))


def test_fp8_linear_exact_on_grid_with_unit_scales():
    rng = np.random.default_rng(10)
    a = oracle.e4m3_round(rng.standard_normal((5, 256)) * 3)
    w = oracle.e4m3_round(rng.standard_normal((130, 256)) * 3)
    sa = np.ones((5, 2), np.float32)
    sw = np.ones((2, 2), np.float32)
    y = oracle.fp8_linear(a, sa, w, sw)
    exact = np.array([[sum(int(round(a[i, j] * 512)) * int(round(w[n, j] * 512))
                           for j in range(256)) for n in range(130)] for i in range(5)],
                     dtype=object)
    assert np.array_equal(y * (512 * 512), exact.astype(np.float64))


def test_fp8_linear_block_scale_invariance():
    rng = np.random.default_rng(12)
    a = oracle.e4m3_round(rng.standard_normal((4, 256)))
    w = oracle.e4m3_round(rng.standard_normal((128, 256)))
    sa = rng.random((4, 2)).astype(np.float32) + 0.5
    sw = rng.random((1, 2)).astype(np.float32) + 0.5
    y = oracle.fp8_linear(a, sa, w, sw)
    # moving a power of two between a K block's codes and its scale is a no-op
    a2, sa2 = a.copy(), sa.copy()
    a2[:, 128:] /= 4
    sa2[:, 1] *= 4
    np.testing.assert_allclose(oracle.fp8_linear(a2, sa2, w, sw), y, rtol=1e-14)
    # a K block scale multiplies only that block's contribution
    sw3 = sw.copy()
    sw3[0, 0] *= 2
    part0 = (a[:, :128] * sa[:, :1]) @ (w[:, :128] * sw[0, 0]).T
    np.testing.assert_allclose(oracle.fp8_linear(a, sa, w, sw3), y + part0, rtol=1e-12)


def test_fp8_layer_close_to_bf16_layer():
    shape = shape_with(CONFIGS["tiny_fp32"], T=24)
    L = make_layer(shape, "cpu")
    args = dict(n_groups=shape.n_groups, topk_groups=shape.topk_groups, k=shape.k)
    ins = [L[k].numpy() for k in ("x", "router_w", "bias", "w13", "w2", "ws13", "ws2")]
    r = oracle.moe_layer_forward(*ins, **args)
    r8 = moe_fp8.moe_layer_forward_fp8(*ins, **args)
    assert np.array_equal(r["topk_idx"], r8["topk_idx"])
    err = np.linalg.norm(r8["out"] - r["out"]) / np.linalg.norm(r["out"])
    # E4M3 keeps 3 mantissa bits: an RMS relative rounding error of about
    # 2.5% per quantised operand.  Four quantised operands on the path
    # (x, W13, h, W2) give roughly 5-6% against the unquantised layer.
    assert 0.01 < err < 0.1


# ------------------------------------------------------------ page values

def test_v3_workloads_carry_the_pages_hyperparameters():
    g = {k: float(v[0]) for k, v in _read_kv("v3_hyperparameters.txt").items()}
    for name in ("v3_bf16", "v3_fp8", "v3_decode"):
        c = CONFIGS[name]
        assert c.d == g["hidden_dim"] and c.n_shared == g["shared_experts"]
        assert c.E == g["routed_experts"] and c.inter == g["expert_intermediate"]
        assert c.k == g["active_routed_experts"] and c.topk_groups == g["max_nodes_per_token"]
        assert c.gamma == g["bias_update_speed"]
        assert c.d % int(g["fp8_group_size"]) == 0


def test_fp8_ffn_reduces_to_dense_ffn_on_grid_inputs():
    # Inputs already on the E4M3 grid with every group's amax = 448 make all
    # scales exactly 1 and the quantisers the identity on x and W; the FP8
    # FFN then differs from the plain SwiGLU FFN only by the re-quantisation
    # of h between the two projections.
    rng = np.random.default_rng(13)
    d, inter, n = 256, 128, 6
    def grid(shape):
        v = oracle.e4m3_round(rng.standard_normal(shape) * 60)
        return v
    x = grid((n, d)); x[:, 0] = 448.0; x[:, 128] = -448.0
    w13 = grid((2 * inter, d)) / 1.0
    w13[0, 0] = w13[0, 128] = w13[128, 0] = w13[128, 128] = 448.0
    w2 = grid((d, inter)); w2[0, 0] = w2[128, 0] = 448.0
    qx, sx = oracle.quantize_act_1x128(x)
    assert np.all(sx == 1.0) and np.array_equal(qx, x)
    y = moe_fp8.fp8_swiglu_ffn(qx, sx, w13, w2)
    h = oracle.silu(x @ w13[:inter].T) * (x @ w13[inter:].T)
    qh, sh = oracle.quantize_act_1x128(h.astype(np.float32))
    np.testing.assert_allclose(y, oracle.dequantize_act_1x128(qh, sh) @ w2.T, rtol=1e-12)
    assert np.linalg.norm(y - h @ w2.T) > 0  # the h quantisation is really there


def test_sampled_tokens_match_whole_layer():
    shape = shape_with(CONFIGS["tiny_fp32"], T=20)
    L = make_layer(shape, "cpu")
    ins = [L[k].numpy() for k in ("x", "router_w", "bias", "w13", "w2", "ws13", "ws2")]
    r = oracle.moe_layer_forward(*ins, n_groups=shape.n_groups,
                                 topk_groups=shape.topk_groups, k=shape.k)
    rows = [0, 7, 19]
    y = oracle.moe_layer_tokens(ins[0][rows], r["topk_idx"][rows], r["topk_w"][rows],
                                ins[3], ins[4], ins[5], ins[6])
    np.testing.assert_allclose(y, r["out"][rows], rtol=1e-12, atol=1e-14)


# ------------------------------------------------- sequence-wise balance statistic

def test_sequence_balance_invariants():
    """sum_i f_i = E for every sequence; equal affinities give P_i = 1/E and
    so L = alpha whatever the routing; alpha scales the loss linearly."""
    rng = np.random.default_rng(11)
    T, E, K, L = 96, 16, 3, 24
    s = rng.random((T, E)) + 0.05
    idx = np.stack([rng.choice(E, K, replace=False) for _ in range(T)])
    f, P, loss = oracle.sequence_balance(s, idx, L, alpha=1e-4)
    np.testing.assert_allclose(f.sum(axis=1), E, rtol=0, atol=1e-12)
    np.testing.assert_allclose(P.sum(axis=1), 1.0, rtol=0, atol=1e-12)
    f2, P2, loss2 = oracle.sequence_balance(np.full((T, E), 0.37), idx, L, alpha=1e-4)
    np.testing.assert_allclose(P2, 1.0 / E, rtol=1e-14)
    np.testing.assert_allclose(loss2, 1e-4, rtol=1e-12)
    _, _, loss3 = oracle.sequence_balance(s, idx, L, alpha=3e-3)
    np.testing.assert_allclose(loss3, loss * 30, rtol=1e-12)


def test_sequence_balance_hand_example():
    """Two tokens, E = 4, K = 1, one sequence.  Token 0 chooses expert 2 with
    s = [1, 1, 2, 0]; token 1 chooses expert 2 with s = [0, 0, 1, 1].
    f = 4 / (1 * 2) * [0, 0, 2, 0] = [0, 0, 4, 0];
    P = ([.25, .25, .5, 0] + [0, 0, .5, .5]) / 2 = [.125, .125, .5, .25];
    L = alpha * 4 * 0.5 = 2 alpha."""
    s = np.array([[1.0, 1.0, 2.0, 0.0], [0.0, 0.0, 1.0, 1.0]])
    idx = np.array([[2], [2]])
    f, P, loss = oracle.sequence_balance(s, idx, 2, alpha=1e-4)
    np.testing.assert_array_equal(f[0], [0, 0, 4, 0])
    np.testing.assert_allclose(P[0], [0.125, 0.125, 0.5, 0.25], rtol=0, atol=1e-15)
    np.testing.assert_allclose(loss, [2e-4], rtol=1e-13)


def test_sequence_balance_splits_sequences():
    """Sequences are independent: the statistic of a batch of two sequences
    is the statistic of each sequence alone."""
    rng = np.random.default_rng(12)
    T, E, K = 40, 8, 2
    s = rng.random((T, E))
    idx = np.stack([rng.choice(E, K, replace=False) for _ in range(T)])
    f, P, loss = oracle.sequence_balance(s, idx, 20)
    fa, Pa, la = oracle.sequence_balance(s[:20], idx[:20], 20)
    fb, Pb, lb = oracle.sequence_balance(s[20:], idx[20:], 20)
    np.testing.assert_array_equal(f, np.concatenate([fa, fb]))
    np.testing.assert_array_equal(loss, np.concatenate([la, lb]))


def test_fp8_sampled_tokens_match_whole_fp8_layer():
    """The FP8 oracle's few-token form (the checker of the full-size FP8
    layer) against the rows of its whole-layer form, on a tiny FP8 layer with
    16 experts, top-3 and a shared expert: the per-token 1 x 128 tiles, the
    per-expert weight blocks, the gate column of each slot and the shared
    expert must all line up, so the rows agree to fp64 rounding."""
    from oracle import moe_fp8
    shape = shape_with(CONFIGS["v3_fp8"], T=24, d=256, E=16, n_groups=4, topk_groups=2, k=3,
                       inter=128, router="gaussian", outlier_channels=3)
    L = make_layer(shape, "cpu")
    f = lambda t: t.float().numpy()
    ins = [f(L[k]) for k in ("x", "router_w", "bias", "w13", "w2", "ws13", "ws2")]
    r = moe_fp8.moe_layer_forward_fp8(*ins, n_groups=shape.n_groups,
                                      topk_groups=shape.topk_groups, k=shape.k,
                                      route_scale=shape.route_scale)
    assert len(set(r["topk_idx"].reshape(-1).tolist())) >= 8   # many experts in play
    rows = [0, 5, 11, 23]
    y = moe_fp8.moe_layer_tokens_fp8(ins[0][rows], r["topk_idx"][rows], r["topk_w"][rows],
                                     ins[3], ins[4], ins[5], ins[6])
    np.testing.assert_allclose(y, r["out"][rows], rtol=1e-12, atol=1e-12)
    # a slot's gate belongs to that slot's expert: swapping two gate columns
    # of a token changes its row
    g = r["topk_w"][rows].copy()
    g[:, [0, 1]] = g[:, [1, 0]]
    y2 = moe_fp8.moe_layer_tokens_fp8(ins[0][rows], r["topk_idx"][rows], g,
                                      ins[3], ins[4], ins[5], ins[6])
    assert np.max(np.abs(y2 - r["out"][rows])) > 1e-3


def test_load_spread_hand_example():
    """Loads [0, 2, 4, 6] over four experts: mean 3, max / mean = 2,
    population standard deviation sqrt((9 + 1 + 1 + 9) / 4) = sqrt(5), so the
    coefficient of variation is sqrt(5) / 3; min 0, max 6.  An even load
    gives max / mean = 1 and CV = 0."""
    s = oracle.load_spread(np.array([0, 2, 4, 6]))
    assert s["max_over_mean"] == 2.0
    assert abs(s["cv"] - np.sqrt(5.0) / 3.0) < 1e-15
    assert (s["min"], s["max"]) == (0, 6)
    e = oracle.load_spread(np.full(8, 5))
    assert (e["max_over_mean"], e["cv"], e["min"], e["max"]) == (1.0, 0.0, 5, 5)
    # the benchmark's host-side report of the same loads (T * K = 12 selections)
    import bench
    b = bench.load_stats([0, 2, 4, 6], T=4, K=3)
    assert b["max_over_mean"] == 2.0 and abs(b["cv"] - np.sqrt(5.0) / 3.0) < 1e-15
    assert (b["min"], b["max"], b["empty_experts"]) == (0, 6, 1)


def test_gate_of_row_makes_the_combine_a_plain_sum():
    """Scaling each permuted row by its slot's gate and then adding rows with
    unit weights is the gate-weighted combine (DeepSeekMoE paragraph), and
    every row receives exactly the gate of the (token, slot) it holds."""
    rng = np.random.default_rng(21)
    T, E, K, d = 37, 12, 3, 16
    idx = np.stack([rng.choice(E, K, replace=False) for _ in range(T)]).astype(np.int32)
    _, _, ros, tor = oracle.segment_layout(idx, E)
    g = rng.random((T, K))
    y = rng.standard_normal((T * K, d))
    ys = rng.standard_normal((T, d))
    gr = oracle.gate_of_row(ros, g)
    assert gr.shape == (T * K,)
    for t in range(T):
        for j in range(K):
            assert gr[ros[t, j]] == g[t, j]
    np.testing.assert_allclose(oracle.combine(ys, gr[:, None] * y, ros, np.ones((T, K))),
                               oracle.combine(ys, y, ros, g), rtol=1e-14, atol=1e-14)
    # a wrong pairing (gates of the next slot) is visible
    bad = oracle.gate_of_row(ros, np.roll(g, 1, axis=1))
    assert np.max(np.abs(bad - gr)) > 1e-3
