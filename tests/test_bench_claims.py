"""The benchmark's launch counts (its `gpu_launches` claim) against the
committed ncu launch lists of the same steps, and its algorithmic FLOP
counts against the layer's definition."""

import os
import re
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import pytest  # noqa: E402

import bench  # noqa: E402
from moe_synth import CONFIGS  # noqa: E402


def _kernel_rows(name):
    """(kernel, launches) rows of a launch list that counts launches per kernel."""
    rows = []
    with open(os.path.join(ROOT, "profiles", name)) as f:
        for line in f:
            m = re.match(r"\| ((?:[^|\\]|\\.)+) \| (\d+) \|", line)
            if m and m.group(1).strip() != "kernel":
                rows.append((m.group(1).strip(), int(m.group(2))))
    return rows


def _step_rows(name):
    """Kernel rows of a launch list of one captured step (kernel | grid | ...)."""
    rows = []
    with open(os.path.join(ROOT, "profiles", name)) as f:
        for line in f:
            m = re.match(r"\| ([^|]+) \| (\([0-9,]+\)) \|", line)
            if m:
                rows.append(m.group(1).strip())
    return rows


@pytest.mark.parametrize("workload", ["v3_bf16", "v3_fp8", "v3_decode"])
def test_forward_launches_match_the_launch_list(workload):
    rows = _step_rows(f"launches_{workload}.md")
    # one row per launch of the captured step
    assert bench.launches_per_step(CONFIGS[workload]) == len(rows)
    assert sum("experts_" in r for r in rows) == 2
    assert sum("combine" in r for r in rows) == 1


def test_training_launches_match_the_launch_list():
    rows = _kernel_rows("launches_v3_bf16_train.md")
    assert all(n == 6 for _, n in rows)   # 6 training steps, one row per position
    assert bench.train_launches(CONFIGS["v3_bf16"]) == len(rows)
    # the gathering forward adds a permute and the recompute in the backward
    # and drops the forward's permute
    assert (bench.train_launches(CONFIGS["v3_bf16"], gather=True)
            == bench.train_launches(CONFIGS["v3_bf16"]) + 1)


def test_fp8_training_launches_match_the_launch_list():
    rows = _step_rows("launches_v3_fp8_train.md")
    assert bench.train_launches(CONFIGS["v3_fp8"]) == len(rows)
    assert sum("wgrad_fp8" in r for r in rows) == 2
    assert sum("quant_rows" in r for r in rows) == 8   # 4 operands x (routed, shared)


def test_algorithmic_flops():
    s = CONFIGS["v3_bf16"]
    rows = s.T * s.k + s.T * s.n_shared
    assert bench.expert_flops(s) == 6.0 * s.d * s.inter * rows
    b = bench.backward_flops(s)
    assert b["dgrad"] == b["wgrad"] == bench.expert_flops(s)
    assert abs(bench.expert_flops(s) / 1e12 - 6.494) < 1e-3   # 6.494 TFLOP per step
