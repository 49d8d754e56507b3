"""Pins of the FP8 backward oracle (Dgrad and Wgrad GEMMs in FP8): exact
results on the E4M3 grid with unit scales, the orientation of the 128 x 1
tiles, power-of-two scale equivariance, and closeness to the fp64 backward
(the FP8 expert backward kernels are not built yet; this is the reference
they will be checked against)."""

import numpy as np

import oracle

GRID = np.unique(np.abs(oracle.e4m3_decode(np.arange(256, dtype=np.uint8))))
GRID = GRID[np.isfinite(GRID)]


def _grid_values(rng, shape):
    """Random E4M3 values of magnitude at most 224 (so that a 448 placed in a
    tile is its maximum)."""
    small = GRID[GRID <= 224.0]
    v = rng.choice(small, size=shape) * rng.choice([-1.0, 1.0], size=shape)
    return v.astype(np.float64)


def test_128x1_tiles_run_along_rows():
    rng = np.random.default_rng(0)
    rows, K = 300, 256          # three row tiles, the last one 44 rows
    x = _grid_values(rng, (rows, K))
    for i in range(3):
        x[i * 128, :] = 448.0   # one 448 in every 128 x 1 tile, in three rows only
    q, s = oracle.quantize_act_128x1(x)
    assert s.shape == (3, K)
    assert np.all(s == 1.0)     # a 1 x 128 tiling would give most rows a smaller scale
    assert np.array_equal(q, x)
    assert np.array_equal(oracle.dequantize_act_128x1(q, s), x)


def test_128x1_scales_are_power_of_two_equivariant():
    rng = np.random.default_rng(1)
    x = rng.standard_normal((200, 128)).astype(np.float32)
    q, s = oracle.quantize_act_128x1(x)
    q8, s8 = oracle.quantize_act_128x1(x * np.float32(8.0))
    assert np.array_equal(q, q8)
    assert np.array_equal(s8, s * np.float32(8.0))


def test_dgrad_and_wgrad_exact_on_the_grid():
    rng = np.random.default_rng(2)
    n, K, N = 256, 256, 384
    g = _grid_values(rng, (n, K))
    g[:, ::128] = 448.0                       # every 1 x 128 tile of g holds 448
    w = _grid_values(rng, (K, N))
    for i in range(0, K, 128):
        for j in range(0, N, 128):
            w[i, j] = 448.0                   # every 128 x 128 block holds 448
    qg, sg = oracle.quantize_act_1x128(g)
    qw, sw = oracle.quantize_weight_128x128(w)
    assert np.all(sg == 1.0) and np.all(sw == 1.0)
    assert np.array_equal(oracle.fp8_dgrad(qg, sg, qw, sw), g @ w)

    a = _grid_values(rng, (n, 128))
    b = _grid_values(rng, (n, N))
    a[::128, :] = 448.0                       # every 128 x 1 tile holds 448
    b[::128, :] = 448.0
    qa, sa = oracle.quantize_act_128x1(a)
    qb, sb = oracle.quantize_act_128x1(b)
    assert np.array_equal(oracle.fp8_wgrad(qa, sa, qb, sb), a.T @ b)


def test_expert_backward_close_to_fp64_and_zero_for_zero_gradient():
    rng = np.random.default_rng(3)
    n, d, inter = 150, 256, 128
    x = rng.standard_normal((n, d)).astype(np.float32)
    w13 = (rng.standard_normal((2 * inter, d)) * 0.05).astype(np.float32)
    w2 = (rng.standard_normal((d, inter)) * 0.05).astype(np.float32)
    dy = rng.standard_normal((n, d)).astype(np.float32)
    qx, sx = oracle.quantize_act_1x128(x)
    r8 = oracle.fp8_swiglu_ffn_backward(qx, sx, w13, w2, dy)
    r = oracle.swiglu_ffn_backward(x, w13[:inter], w13[inter:], w2, dy)
    rel = lambda a, b: np.linalg.norm(a - b) / np.linalg.norm(b)
    # E4M3 keeps 3 mantissa bits (relative rounding error up to 1/16 per value)
    assert rel(r8["du"], r["du"]) < 0.1
    assert rel(r8["dw2"], r["dw2"]) < 0.1
    assert rel(r8["dw13"], np.concatenate([r["dw1"], r["dw3"]])) < 0.1
    z = oracle.fp8_swiglu_ffn_backward(qx, sx, w13, w2, np.zeros_like(dy))
    for k in ("du", "dw13", "dw2"):
        assert np.all(z[k] == 0.0)
