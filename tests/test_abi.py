"""The C-ABI library without a GPU: it loads, exports every declared symbol,
and its host-side argument checks answer before any launch."""

import ctypes
import os
import re

import pytest

import mixture_experts_layer_82_b300 as moe
from moe_synth import CONFIGS

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "moe.h")


def _declared():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z0-9_]+)\s*\(", text)))


def test_every_declared_symbol_is_exported():
    names = _declared()
    assert "moe_route" in names and "moe_experts_grouped" in names
    lib = moe.library()
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) == set(moe.EXPORTED)


def _param_counts():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    out = {}
    for name, params in re.findall(r"\b(moe_[a-z0-9_]+)\s*\(([^)]*)\)\s*;", text):
        params = params.strip()
        out[name] = 0 if params in ("", "void") else params.count(",") + 1
    return out


def test_binding_signatures_match_header():
    lib = moe.library()
    counts = _param_counts()
    assert set(counts) == set(moe.EXPORTED)
    for name, n in counts.items():
        argtypes = getattr(lib, name).argtypes
        assert argtypes is not None and len(argtypes) == n, (name, n, argtypes)


def test_cfg_struct_layout():
    # 9 int32 + 2 float + 1 int32, no padding
    assert ctypes.sizeof(moe.MoeCfg) == 48
    assert moe.MoeCfg.route_scale.offset == 36 and moe.MoeCfg.dtype.offset == 44


def test_version_and_status_strings():
    lib = moe.library()
    assert lib.moe_version() >= 100
    for code in range(8):
        assert lib.moe_status_str(code).decode()
    assert lib.moe_status_str(99).decode() == "unknown status"


@pytest.mark.parametrize("name", sorted(CONFIGS))
def test_workloads_pass_the_checks(name):
    cfg = moe.LayerCfg.from_shape(CONFIGS[name])
    if cfg.dtype == "fp8" and moe.moe_check_cfg(cfg) == 2:
        pytest.skip("fp8 kind not enabled")
    assert moe.moe_check_cfg(cfg) == 0
    assert moe.moe_workspace_bytes(cfg) > 0


def _base(**kw):
    c = moe.LayerCfg.from_shape(CONFIGS["mid_bf16"])
    for k, v in kw.items():
        setattr(c, k, v)
    return c


@pytest.mark.parametrize("kw,status", [
    (dict(T=0), 1), (dict(E=63), 1), (dict(topk_groups=9), 1), (dict(k=65), 1),
    (dict(n_groups=64, topk_groups=1, k=2), 1),   # kept groups hold fewer than K experts
    (dict(d=2000), 2), (dict(inter=1400), 2), (dict(T=(1 << 22) + 1), 2),
    (dict(group_score_topn=0), 1), (dict(group_score_topn=9), 2), (dict(n_shared=-1), 1),
    (dict(E=2048, n_groups=32), 2), (dict(k=33, E=128), 2), (dict(route_scale=float("nan")), 1),
])
def test_bad_configs_are_rejected(kw, status):
    assert moe.moe_check_cfg(_base(**kw)) == status
    assert moe.moe_workspace_bytes(_base(**kw)) == 0


def test_fp32_kind_allows_any_multiple_of_four():
    c = _base(dtype="fp32", d=260, inter=100)
    assert moe.moe_check_cfg(c) == 0
    assert moe.moe_check_cfg(_base(dtype="fp32", d=258)) == 2


def _route_raw(cfg, ptrs, ws_bytes=1 << 20):
    lib = moe.library()
    return lib.moe_route(ctypes.byref(cfg.c()), *ptrs, ws_bytes, None)


def test_route_rejects_null_and_misaligned_pointers_without_launching():
    cfg = _base()
    good = [0x10000 * (i + 1) for i in range(12)]  # never dereferenced: checks come first
    ptrs = list(good)
    ptrs[2] = None  # bias
    assert _route_raw(cfg, ptrs) == 1
    ptrs = list(good)
    ptrs[3] = None; ptrs[0] = None  # neither x nor affinity_in
    assert _route_raw(cfg, ptrs) == 1
    ptrs = list(good)
    ptrs[5] += 4  # topk_idx misaligned
    assert _route_raw(cfg, ptrs) == 3
    assert _route_raw(cfg, good, ws_bytes=16) == 7  # workspace too small


def test_other_calls_check_before_launching():
    lib = moe.library()
    cfg = ctypes.byref(_base().c())
    a = 0x100000
    assert lib.moe_permute(cfg, None, a, a, None, None, None, None) == 1
    assert lib.moe_combine(cfg, a, a, a + 8, a, a, None) == 3
    assert lib.moe_bias_update(cfg, None, a, None) == 1
    assert lib.moe_quantize_weights_fp8(a, 1, 128, 100, a, a, None) == 2
    assert lib.moe_quantize_weights_fp8(a, 0, 128, 128, a, a, None) == 1
    args = [None] * 15
    assert lib.moe_experts_grouped(cfg, *args, None, 0, None) == 1
    fp8 = _base(dtype="fp8")
    if moe.moe_check_cfg(fp8) == 0:
        # FP8 without scale pointers
        p = [a] * 15
        p[1] = None
        assert lib.moe_experts_grouped(ctypes.byref(fp8.c()), *p, a, 1 << 40, None) == 1


def test_binding_refuses_host_tensors():
    import torch
    with pytest.raises(ValueError):
        moe.moe_bias_update(_base(), torch.zeros(64, dtype=torch.int32),
                            torch.zeros(64, dtype=torch.float32), stream=0)


def _align256(n):
    return (n + 255) // 256 * 256


def test_backward_workspace_formula_and_kinds():
    c = _base()  # mid-size bf16 layer: T=4096, K=6, N_s=2, I=1408
    tk, T, I, ns = c.T * c.k, c.T, c.inter, c.n_shared
    assert moe.moe_backward_workspace_bytes(c) == (_align256((tk + T * ns) * 3 * I * 2)
                                                   + _align256(tk * 4))
    # the backward exists for the bf16 kind (at most 64 shared experts) and,
    # on the input side, the FP8 kind with at most one shared expert: its
    # expert part holds q(dy), [a | b], dh and q([da | db]) for T*K + T rows
    assert moe.moe_backward_workspace_bytes(_base(dtype="fp32")) == 0
    assert moe.moe_backward_workspace_bytes(_base(dtype="fp8")) == 0   # two shared experts
    f = _base(dtype="fp8", n_shared=1)
    rows, d, E = tk + T, f.d, f.E
    dgrad = (_align256(rows * d) + _align256(rows * (d // 128) * 4) + _align256(rows * 2 * I * 2)
             + _align256(rows * I * 2) + _align256(rows * 2 * I)
             + _align256(rows * (2 * I // 128) * 4))
    # Wgrad: padded segment starts and the rows of every padded tile, then
    # the codes and scales of dy, u, h, [da | db] with every segment padded
    # to 128 rows (routed) and the shared expert's T rows
    P = (tk + 127 * E + 127) // 128 * 128
    Ps = (T + 127) // 128 * 128
    wgrad = _align256((E + 1) * 4) + _align256(P // 128 * 8) + sum(
        _align256(C * P) + _align256(P // 128 * C * 4) + _align256(C * Ps)
        + _align256(Ps // 128 * C * 4) for C in (d, d, I, 2 * I))
    assert moe.moe_backward_workspace_bytes(f) == dgrad + wgrad + _align256(tk * 4)
    assert moe.moe_backward_workspace_bytes(_base(n_shared=65)) == 0
    assert moe.moe_backward_workspace_bytes(_base(d=2000)) == 0


def test_backward_calls_check_before_launching():
    lib = moe.library()
    bf = ctypes.byref(_base().c())
    fp32 = ctypes.byref(_base(dtype="fp32").c())
    a = 0x100000
    ws = moe.moe_backward_workspace_bytes(_base())
    # combine backward: kind, null, alignment
    assert lib.moe_combine_backward(fp32, a, a, a, a, a, a, None) == 2
    assert lib.moe_combine_backward(bf, a, None, a, a, a, a, None) == 1
    assert lib.moe_combine_backward(bf, a, a, a, a, a + 4, a, None) == 3
    # input call: missing shared-expert pointers, small workspace, misaligned
    p = [a] * 11
    q = list(p); q[5] = None  # ws13 with N_s = 2
    assert lib.moe_experts_backward_input(bf, *q, 0, a, ws, None) == 1
    assert lib.moe_experts_backward_input(bf, *p, 0, a, ws - 1, None) == 7
    q = list(p); q[9] = a + 8  # dx_perm misaligned
    assert lib.moe_experts_backward_input(bf, *q, 0, a, ws, None) == 3
    # weights call
    p = [a] * 9
    assert lib.moe_experts_backward_weights(fp32, *p, a, ws, None) == 2
    q = list(p); q[5] = None  # dw13
    assert lib.moe_experts_backward_weights(bf, *q, a, ws, None) == 1
    assert lib.moe_experts_backward_weights(bf, *p, a, 16, None) == 7
    # route backward
    p = [a] * 13
    q = list(p); q[2] = None  # affinity
    assert lib.moe_route_backward(bf, *q, a, ws, None) == 1
    assert lib.moe_route_backward(bf, *p, a, 16, None) == 7
    # training forward: the backward workspace must be large enough
    p = [a] * 10
    big = moe.moe_workspace_bytes(_base())
    assert lib.moe_experts_grouped_train(bf, *p, big, a, ws - 1, None) == 7
    assert lib.moe_experts_grouped_train(fp32, *p, big, a, ws, None) == 2


def test_fp8_backward_calls_check_before_launching():
    """The FP8 training calls: kind and shared-expert limits, NULL and
    misaligned pointers, workspace sizes, the 128 x 1 quantiser's width."""
    lib = moe.library()
    a = 0x100000
    f8 = _base(dtype="fp8", n_shared=1)
    f8c = ctypes.byref(f8.c())
    bf = ctypes.byref(_base().c())
    two = ctypes.byref(_base(dtype="fp8", n_shared=2).c())
    ws = moe.moe_backward_workspace_bytes(f8)
    big = moe.moe_workspace_bytes(f8)
    # training forward keeping [a | b]: kind, N_s <= 1, bws size and alignment
    p = [a] * 16
    assert lib.moe_experts_grouped_train_fp8(bf, *p, big, a, ws, None) == 2
    assert lib.moe_experts_grouped_train_fp8(two, *p, big, a, ws, None) == 2
    assert lib.moe_experts_grouped_train_fp8(f8c, *p, big, None, ws, None) == 1
    assert lib.moe_experts_grouped_train_fp8(f8c, *p, big, a + 8, ws, None) == 3
    assert lib.moe_experts_grouped_train_fp8(f8c, *p, big, a, ws - 1, None) == 7
    # Dgrad: kind, a missing weight transpose, misaligned dy, small workspace
    p = [a] * 21
    assert lib.moe_experts_backward_input_fp8(bf, *p, 0, a, ws, None) == 2
    q = list(p); q[8] = None  # w2t
    assert lib.moe_experts_backward_input_fp8(f8c, *q, 1, a, ws, None) == 1
    q = list(p); q[17] = a + 4  # dy_perm
    assert lib.moe_experts_backward_input_fp8(f8c, *q, 0, a, ws, None) == 3
    assert lib.moe_experts_backward_input_fp8(f8c, *p, 0, a, 16, None) == 7
    # Wgrad: kind, NULL dW2, the shared expert's dWs2, small workspace
    p = [a] * 11
    assert lib.moe_experts_backward_weights_fp8(bf, *p, a, ws, None) == 2
    q = list(p); q[8] = None  # dw2
    assert lib.moe_experts_backward_weights_fp8(f8c, *q, a, ws, None) == 1
    q = list(p); q[10] = None  # dws2 with N_s = 1
    assert lib.moe_experts_backward_weights_fp8(f8c, *q, a, ws, None) == 1
    assert lib.moe_experts_backward_weights_fp8(f8c, *p, a, 16, None) == 7
    # 128 x 1 quantiser: width, NULL, alignment, empty
    assert lib.moe_quantize_act_fp8_128x1(a, 300, 200, a, a, None) == 2
    assert lib.moe_quantize_act_fp8_128x1(None, 300, 256, a, a, None) == 1
    assert lib.moe_quantize_act_fp8_128x1(a, 300, 256, a + 8, a, None) == 3
    assert lib.moe_quantize_act_fp8_128x1(a, 0, 256, a, a, None) == 1


def test_bias_update_takes_the_whole_batch_of_many_replicas():
    """Data-parallel replicas call moe_bias_update with T = world x T (the
    whole batch's mean load).  That T may exceed the 2^22 tokens one routing
    call accepts: the bias update checks only E, K, T and gamma, so such a
    configuration gets past the shape check to the pointer check (NULL
    counts: MOE_ERR_INVALID_ARG, nothing launched)."""
    from mixture_experts_layer_82_b300.replicas import global_cfg

    lib = moe.library()
    a = 0x100000
    cfg = _base()
    for world in (2, 64, 512):
        g = global_cfg(cfg, world)
        g.T = (1 << 22) + 1 if world == 2 else g.T * 600
        assert moe.moe_check_cfg(g) != 0  # routing would refuse this T
        assert lib.moe_bias_update(ctypes.byref(g.c()), None, a, None) == 1
        assert lib.moe_bias_update(ctypes.byref(g.c()), a, a + 4, None) == 3
    bad = _base()
    bad.k = bad.E + 1
    assert lib.moe_bias_update(ctypes.byref(bad.c()), a, a, None) == 1
    bad = _base()
    bad.E = 2048
    bad.n_groups = 1
    bad.topk_groups = 1
    assert lib.moe_bias_update(ctypes.byref(bad.c()), a, a, None) == 2
