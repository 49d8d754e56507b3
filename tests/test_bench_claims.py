"""The benchmark's launch counts (its `gpu_launches` claim) against the
committed ncu launch lists of the same steps, and its algorithmic FLOP
counts against the layer's definition."""

import os
import re
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from moe_synth import CONFIGS  # noqa: E402


def _kernel_rows(name):
    rows = []
    with open(os.path.join(ROOT, "profiles", name)) as f:
        for line in f:
            m = re.match(r"\| ((?:[^|\\]|\\.)+) \| (\d+) \|", line)
            if m and m.group(1).strip() != "kernel":
                rows.append((m.group(1).strip(), int(m.group(2))))
    return rows


def test_forward_launches_match_the_launch_list():
    rows = _kernel_rows("launches_v3_bf16.md")
    # every kernel of the step appears once per step, 11 steps in the list
    assert all(n == 11 for _, n in rows)
    assert bench.launches_per_step(CONFIGS["v3_bf16"]) == len(rows)


def test_training_launches_match_the_launch_list():
    rows = _kernel_rows("launches_v3_bf16_train.md")
    assert all(n == 6 for _, n in rows)   # 6 training steps, one row per position
    assert bench.train_launches(CONFIGS["v3_bf16"]) == len(rows)
    # the gathering forward adds a permute and the recompute in the backward
    # and drops the forward's permute
    assert (bench.train_launches(CONFIGS["v3_bf16"], gather=True)
            == bench.train_launches(CONFIGS["v3_bf16"]) + 1)


def test_algorithmic_flops():
    s = CONFIGS["v3_bf16"]
    rows = s.T * s.k + s.T * s.n_shared
    assert bench.expert_flops(s) == 6.0 * s.d * s.inter * rows
    b = bench.backward_flops(s)
    assert b["dgrad"] == b["wgrad"] == bench.expert_flops(s)
    assert abs(bench.expert_flops(s) / 1e12 - 6.494) < 1e-3   # 6.494 TFLOP per step
