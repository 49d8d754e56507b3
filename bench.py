"""Benchmark of the DeepSeekMoE layer forward on B300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload v3_bf16|v3_fp8|v3_decode|mid_bf16] [--no-also]

A step is one pass of the whole layer (route -> permute -> grouped expert
GEMMs -> combine -> bias update) over one batch of T tokens, with every
input already resident in device memory.  The default workload is the
DeepSeek-V3-shaped layer in bf16 (T=8192, d=7168, 256 routed experts in 8
groups, top-4 groups, top-8, 1 shared expert, I=2048, route scale 2.5, Zipf
-skewed router); the same run also times the FP8 layer of that shape and
the decode-shaped batch (T=128) and reports them under "also", each with
its own roofline, clock record and end-to-end figure.  With N > 1
(torchrun) every rank runs its own replica on its own batch (weak scaling,
no collective on the data path; the replicas
sum their per-expert loads with one all-reduce of counts[E] per step so that
the bias update sees the whole batch); the time is the maximum over ranks.
Rank 0 prints one JSON line.

``--train`` (bf16 and fp8 kinds) makes a step one training pass instead: the
forward above, then its backward (combine backward, expert Dgrad, router
backward, expert Wgrad), given a fixed dL/dy.  The forward keeps the
gate/up products for the backward.

``--impl reference`` times the CPU oracle (fp64 NumPy) on the host cores on a
bounded sample of the same workload; that is the only other place, besides
the ``cpu_baseline`` leg, where this script runs the oracle.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from moe_synth import CONFIGS, make_layer  # noqa: E402

METRIC = "MoE-layer tokens/s at V3 shape (bf16, FP8); TFLOP/s as % of B300 peak"
METRIC_TRAIN = ("MoE-layer training tokens/s (forward + backward) at V3 shape (bf16); "
                "TFLOP/s as % of B300 peak")
PEAKS_FALLBACK = {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0}
# sources of the expert GEMM kernels of each kind (the bf16 calls dispatch
# between the pair-MMA and the multicast-pair kernels)
KERNEL_SRC = {"bf16": ["mixture_experts_layer_82_b300/csrc/experts_sm100.cu",
                       "mixture_experts_layer_82_b300/csrc/experts_pair.cu"],
              "fp8": ["mixture_experts_layer_82_b300/csrc/experts_fp8.cu"]}


def kernel_src_sha256(dtype):
    """SHA-256 of the kind's kernel sources, concatenated in order."""
    h = hashlib.sha256()
    for f in KERNEL_SRC[dtype]:
        with open(os.path.join(ROOT, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()


# --------------------------------------------------------------- workload

def describe(shape):
    return (f"{shape.name}: T={shape.T}, d={shape.d}, E={shape.E} routed in {shape.n_groups} "
            f"groups (top-{shape.topk_groups} groups), top-{shape.k}, {shape.n_shared} shared, "
            f"I={shape.inter}, route scale {shape.route_scale}, {shape.dtype}, router "
            f"{shape.router}, seed {shape.seed}")


def expert_flops(shape):
    """Algorithmic FLOPs of the expert GEMMs: 3 projections of d x I per
    routed slot and per token for every shared expert (no padding)."""
    return 6.0 * shape.d * shape.inter * (shape.T * shape.k + shape.T * shape.n_shared)


def expert_bytes(shape, counts):
    """Algorithmic DRAM bytes of one moe_experts_grouped call: the weights of
    every expert that received a token (read once), the shared experts, and
    the activations (x_perm and x read, h written and read, y written)."""
    wb = 1 if shape.dtype == "fp8" else (4 if shape.dtype == "fp32" else 2)
    ab = 4 if shape.dtype == "fp32" else 2
    touched = int((np.asarray(counts) > 0).sum())
    weights = 3 * shape.d * shape.inter * wb * (touched + shape.n_shared)
    rows = shape.T * shape.k
    act = (rows * shape.d * (wb if shape.dtype == "fp8" else ab) + shape.T * shape.d * ab
           + 2 * (rows + shape.T * shape.n_shared) * shape.inter * ab
           + (rows + shape.T * (1 if shape.n_shared else 0)) * shape.d * ab)
    return weights + act, touched


def backward_flops(shape):
    """Algorithmic FLOPs of the expert backward: Dgrad (dh = dy W2 and
    dx = [da | db] W13) and Wgrad (dW2 and dW13), 6 d I per row each.  The
    recomputation of [a | b] (4 d I per row; only when the forward did not
    keep it, i.e. with --dispatch gather) is not counted."""
    rows = shape.T * shape.k + shape.T * shape.n_shared
    return {"dgrad": 6.0 * shape.d * shape.inter * rows, "wgrad": 6.0 * shape.d * shape.inter * rows,
            "recompute": 4.0 * shape.d * shape.inter * rows}


def train_launches(shape, gather=False):
    """Kernels of one training step: the forward's, then combine backward,
    two Dgrad and two Wgrad GEMMs, the router backward's two kernels, and,
    when the forward gathered its rows, a permute and the recomputation of
    the gate/up products.  FP8 kind (the forward keeps [a | b]): the Dgrad
    quantises dy (one launch per class: routed, shared), forms dh,
    quantises [da | db] and forms dx (three launches); the Wgrad pads the segment
    starts, writes each of its four operands transposed in 128 x 1 tiles
    (one launch per operand and class) and runs its two GEMMs."""
    if shape.dtype == "fp8":
        cls = 1 + (1 if shape.n_shared else 0)
        return launches_per_step(shape) + 1 + (cls + 3) + 2 + (1 + 4 * cls + 2)
    return launches_per_step(shape, gather) + 1 + 2 + 2 + 2 + (2 if gather else 0)


def layer_flops(shape):
    return expert_flops(shape) + 2.0 * shape.T * shape.d * shape.E


def router_launches(shape):
    """Kernels of the router product: one CUDA-core kernel for the fp32
    kind; for bf16 token rows the centroid split, the tensor-core product
    and, when the 128 x 128 output tiles cannot fill the 148 SMs and d is
    long enough to split, the ordered reduction of the split-K partials."""
    if shape.dtype == "fp32":
        return 1
    tiles = -(-shape.T // 128) * -(-shape.E // 128)
    splits = max(1, min(148 // tiles, (shape.d // 64) // 4))
    if splits > 1:
        per = -(-(shape.d // 64) // splits)
        splits = -(-(shape.d // 64) // per)
    return 2 + (1 if splits > 1 else 0)


def launches_per_step(shape, gather=False):
    """Kernels one layer step launches: router product, select, scan,
    assign; permute (quantise + permute for fp8; none when the gate/up GEMM
    gathers its rows); gate/up and down GEMMs; combine; bias update."""
    permute = 0 if gather else (2 if shape.dtype == "fp8" else 1)
    return router_launches(shape) + 3 + permute + 2 + 1 + 1


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        d["_source"] = "measured"
        return d
    d = dict(PEAKS_FALLBACK)
    d["_source"] = "fallback"
    return d


def kernel_traffic(dtype, workload):
    """DRAM bytes per launch of the expert GEMM pair from the committed ncu
    summary, if the kernel source has not changed since it was taken."""
    summ = os.path.join(ROOT, "profiles", f"experts_{dtype}_{workload}_traffic.json")
    if dtype not in KERNEL_SRC or not os.path.exists(summ):
        return None
    sha = kernel_src_sha256(dtype)
    with open(summ) as f:
        d = json.load(f)
    if d.get("kernel_src_sha256") != sha:
        return None
    return d.get("traffic_bytes_per_launch")


# ----------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi clock / throttle sampling during the timed region."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "100", "-f", self.path],
                stdout=subprocess.DEVNULL, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        pw = [float(r[3]) for r in rows if r[3].replace(".", "").isdigit()]
        # "under load": samples drawing more than half of the maximum power seen
        loaded = [s for s, p in zip(sm, pw) if pw and p > 0.5 * max(pw)] or sm
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in rows for n, v in zip(names, r[5:9]) if v == "Active"})
        return {"sm_mhz": statistics.median(loaded) if loaded else None,
                "sm_max_mhz": float(rows[0][2]) if rows[0][2].replace(".", "").isdigit() else None,
                "reasons": reasons, "samples": len(rows),
                "power_w_max": max(pw) if pw else None}


# ------------------------------------------------------------ distributed

def dist_setup(n_gpus):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    elif torch.cuda.is_available():
        torch.cuda.set_device(0)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(v, world):
    if world == 1:
        return v
    import torch.distributed as dist
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    t = torch.tensor([v], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ------------------------------------------------------------ load balance

def load_stats(counts, T, K):
    """Descriptive statistics of per-expert loads (host side)."""
    c = np.asarray(counts, dtype=np.float64)
    mean = T * K / len(c)
    return {"max_over_mean": float(c.max() / mean), "cv": float(c.std() / mean),
            "min": int(c.min()), "max": int(c.max()), "empty_experts": int((c == 0).sum())}


def load_balance(moe, shape, L, steps):
    """Per-expert load spread on the workload's batch before the first and
    after `steps` sign-rule bias updates (route + bias update per step,
    through the library; the affinities of the fixed batch are computed once
    and passed back in)."""
    cfg = moe.LayerCfg.from_shape(shape)
    T, E, K = shape.T, shape.E, shape.k
    dev = L["x"].device
    i32 = dict(dtype=torch.int32, device=dev)
    bufs = [torch.empty(T, K, **i32), torch.empty(T, K, dtype=torch.float32, device=dev),
            torch.empty(E, **i32), torch.empty(E + 1, **i32), torch.empty(T, K, **i32),
            torch.empty(T * K, **i32)]
    ws = torch.empty(moe.moe_workspace_bytes(cfg), dtype=torch.uint8, device=dev)
    aff = torch.empty(T, E, dtype=torch.float32, device=dev)
    bias = L["bias"].clone()
    # sequence-wise balance statistic of the batch taken as one sequence
    f = torch.empty(1, E, dtype=torch.float32, device=dev)
    p = torch.empty_like(f)
    loss = torch.empty(1, dtype=torch.float32, device=dev)
    moe.moe_route(cfg, L["x"], L["router_w"], bias, *bufs, ws, affinity_out=aff)
    moe.moe_balance_stat(cfg, aff, bufs[0], T, f, p, loss, ws)
    before = load_stats(bufs[2].cpu().numpy(), T, K)
    before["seq_balance_stat"] = float(loss.item())
    for i in range(steps):
        if i:
            moe.moe_route(cfg, None, None, bias, *bufs, ws, affinity_in=aff)
        moe.moe_bias_update(cfg, bufs[2], bias)
    moe.moe_route(cfg, None, None, bias, *bufs, ws, affinity_in=aff)
    after = load_stats(bufs[2].cpu().numpy(), T, K)
    # time the statistic's two kernels (after warm-up)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    for _ in range(3):
        moe.moe_balance_stat(cfg, aff, bufs[0], T, f, p, loss, ws)
    e0.record()
    for _ in range(10):
        moe.moe_balance_stat(cfg, aff, bufs[0], T, f, p, loss, ws)
    e1.record()
    torch.cuda.synchronize()
    after["seq_balance_stat"] = float(loss.item())
    if moe.moe_get_device_error() != 0:
        raise RuntimeError("device error in the load-balance steps")
    return {"bias_steps": steps, "gamma": shape.gamma, "before": before, "after": after,
            "seq_balance": {"alpha": 1e-4, "seq_len": T,
                            "us_per_call": 1e3 * e0.elapsed_time(e1) / 10}}


# ----------------------------------------------------------- CPU baseline

def oracle_sample(shape, L, n_tokens, token0=0):
    """Runs the fp64 oracle end to end (affinity, selection, gates, experts,
    combine) on n_tokens tokens of the workload; returns (seconds, tokens).
    Expert weights are fetched from device memory one expert at a time."""
    import oracle
    from oracle import moe_fp8

    class View:
        def __init__(self, t):
            self.t = t

        def __len__(self):
            return self.t.shape[0]

        def __getitem__(self, e):
            return self.t[e].float().cpu().numpy()

    rows = torch.arange(token0, token0 + n_tokens, device=L["x"].device)
    x = L["x"][rows].float().cpu().numpy()
    rw = L["router_w"].cpu().numpy()
    b = L["bias"].cpu().numpy()
    t0 = time.perf_counter()
    s = oracle.sigmoid_affinity(x, rw)
    idx = oracle.select_experts(s.astype(np.float32), b, shape.n_groups, shape.topk_groups,
                                shape.k, shape.group_score_topn)
    g = oracle.gating_weights(s, idx, shape.route_scale)
    fn = moe_fp8.moe_layer_tokens_fp8 if shape.dtype == "fp8" else oracle.moe_layer_tokens
    fn(x, idx, g, View(L["w13"]), View(L["w2"]), View(L["ws13"]), View(L["ws2"]))
    return time.perf_counter() - t0, n_tokens


def oracle_train_sample(shape, L, n_tokens, token0=0):
    """The fp64 oracle forward + backward on n_tokens tokens of the workload
    taken as a batch of their own (their routing, expert and router
    gradients); returns (seconds, tokens)."""
    import oracle
    from moe_synth import make_grad

    class View:
        def __init__(self, t):
            self.t = t

        def __len__(self):
            return self.t.shape[0]

        def __getitem__(self, e):
            return self.t[e].float().cpu().numpy()

    rows = torch.arange(token0, token0 + n_tokens, device=L["x"].device)
    x = L["x"][rows].float().cpu().numpy()
    go = make_grad(shape, L["x"].device)[rows].float().cpu().numpy()
    rw = L["router_w"].cpu().numpy()
    b = L["bias"].cpu().numpy()
    ws13 = View(L["ws13"]) if shape.n_shared else None
    ws2 = View(L["ws2"]) if shape.n_shared else None
    t0 = time.perf_counter()
    if shape.dtype == "fp8":
        # FP8 forward, then each expert's FP8 Dgrad and Wgrad on its rows
        # (dL/dy of a row = its gate times dL/d(out) of its token); the
        # router's backward is not part of this sample
        from oracle.moe_fp8 import moe_layer_forward_fp8
        from oracle.moe_fp8_backward import fp8_swiglu_ffn_backward
        fwd = moe_layer_forward_fp8(x, rw, b, View(L["w13"]), View(L["w2"]), ws13, ws2,
                                    n_groups=shape.n_groups, topk_groups=shape.topk_groups,
                                    k=shape.k, route_scale=shape.route_scale)
        off, tor = fwd["offsets"], fwd["token_of_row"]
        slot = np.argsort(fwd["row_of_slot"].reshape(-1))
        gate_of_row = fwd["topk_w"].reshape(-1)[slot]
        for e in range(shape.E):
            lo, hi = int(off[e]), int(off[e + 1])
            if hi > lo:
                t = tor[lo:hi]
                fp8_swiglu_ffn_backward(fwd["x_q"][t], fwd["x_scale"][t], View(L["w13"])[e],
                                        View(L["w2"])[e], gate_of_row[lo:hi, None] * go[t])
        for j in range(shape.n_shared):
            fp8_swiglu_ffn_backward(fwd["x_q"], fwd["x_scale"], ws13[j], ws2[j], go)
        return time.perf_counter() - t0, n_tokens
    fwd = oracle.moe_layer_forward(x, rw, b, View(L["w13"]), View(L["w2"]), ws13, ws2,
                                   n_groups=shape.n_groups, topk_groups=shape.topk_groups,
                                   k=shape.k, route_scale=shape.route_scale)
    oracle.moe_layer_backward(x, rw, View(L["w13"]), View(L["w2"]), ws13, ws2, fwd, go,
                              route_scale=shape.route_scale)
    return time.perf_counter() - t0, n_tokens


def blas_threads():
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads", 0) for i in threadpool_info() if i.get("user_api") == "blas"]
        return max(n) if n else 1
    except Exception:
        return len(os.sched_getaffinity(0))


# ------------------------------------------------------------------- arms

def run_reference(args, shape, world, rank):
    """The oracle as it stands, timed on the host cores: each step is a bounded
    sample of the workload (args.ref_tokens tokens end to end)."""
    if rank != 0:
        return 0
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    L = make_layer(shape, dev)
    train = getattr(args, "train", False)
    fn = oracle_train_sample if train else oracle_sample
    for i in range(args.warmup):
        fn(shape, L, args.ref_tokens, token0=i * args.ref_tokens)
    secs, toks = 0.0, 0
    for i in range(args.steps):
        s, n = fn(shape, L, args.ref_tokens,
                  token0=((args.warmup + i) * args.ref_tokens) % (shape.T - args.ref_tokens))
        secs += s
        toks += n
    value = toks / secs
    cores = blas_threads()
    sample = (f"{args.ref_tokens} tokens of the {shape.name} batch per step, end to end "
              f"(affinity, group-limited top-k, gates, shared + routed SwiGLU experts in fp64, "
              f"combine{'; then the whole backward' if train else ''}); expert weights "
              f"fetched from device memory per expert")
    line = {"impl": "reference", "metric": METRIC_TRAIN if train else METRIC,
            "value": value, "unit": "tokens/s",
            "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * secs / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": describe(shape)},
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


ALSO = ("v3_fp8", "v3_decode")  # timed beside the default workload in the same run


def run_ours(args, shape, world, rank, local):
    """The headline line; with the default workload (and no --no-also) the
    FP8 and decode-shaped V3 layers are timed in the same run and reported
    under "also", each with its own roofline, clocks and e2e."""
    line = measure_ours(args, shape, world, rank, local, cpu_baseline=True)
    if args.workload == "v3_bf16" and not args.set and not args.no_also:
        line["also"] = {}
        for name in ALSO:
            sub = measure_ours(args, CONFIGS[name], world, rank, local, cpu_baseline=False)
            for k in ("metric", "n_gpus", "steps", "warmup", "higher_is_better", "scaling",
                      "vs_baseline", "data"):
                sub.pop(k, None)
            line["also"][name] = sub
    if rank == 0:
        print(json.dumps(line), flush=True)
    return 0


def measure_ours(args, shape, world, rank, local, cpu_baseline):
    """Times one workload: device-resident steps (CUDA events), then the same
    steps end to end through host buffers; returns the JSON line's fields."""
    import mixture_experts_layer_82_b300 as moe

    dev = f"cuda:{local}"
    torch.cuda.set_device(local)
    L = make_layer(shape, dev)
    cfg = moe.LayerCfg.from_shape(shape)
    gather = args.dispatch == "gather" and shape.dtype == "bf16"
    layer = moe.MoELayer(cfg, L["router_w"], L["bias"].clone(), L["w13"], L["w2"],
                         L["ws13"] if shape.n_shared else None, L["ws2"] if shape.n_shared else None,
                         gather=gather)
    x = L["x"]
    stream = torch.cuda.current_stream()
    # data-parallel replicas sum their per-expert loads for the bias update
    lg = None
    if world > 1:
        import torch.distributed as dist
        lg = dist.group.WORLD
    gated = args.gated and not gather
    for _ in range(args.warmup):
        layer.forward(x, load_group=lg, gated=gated)
    torch.cuda.synchronize()
    status = moe.moe_get_device_error()
    if status != 0:
        raise RuntimeError(f"device error status {status} after warm-up")

    # ---- device-resident timing
    K = args.steps
    ev_exp = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(K)]
    ev_step = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(K)]
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(local)
    clocks.start()
    barrier(world)
    torch.cuda.synchronize()
    t_start.record(stream)
    for i in range(K):
        ev_step[i][0].record(stream)
        layer.forward(x, expert_events=ev_exp[i], load_group=lg, gated=gated)
        ev_step[i][1].record(stream)
    t_end.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    clk = clocks.stop()
    total_ms = max_over_ranks(t_start.elapsed_time(t_end), world)
    exp_ms = [a.elapsed_time(b) for a, b in ev_exp]
    step_ms = [a.elapsed_time(b) for a, b in ev_step]
    status = moe.moe_get_device_error()
    if status != 0:
        raise RuntimeError(f"device error status {status} in the timed region")

    # ---- end to end through host buffers (pinned), copies inside the region.
    # Every step copies its input x from pinned host memory and reads its
    # output back; the copies are pipelined the way a serving loop runs
    # them: step i+1's input copy (stream h2d) and step i's output copy
    # (stream d2h) overlap the kernels of step i, with double-buffered
    # device inputs and outputs.  The region ends when the last output is
    # on the host.
    x_host = x.cpu().pin_memory()
    out_host = [torch.empty(shape.T, shape.d, dtype=layer.out.dtype).pin_memory() for _ in range(2)]
    x_dev = [torch.empty_like(x) for _ in range(2)]
    out_dev = [torch.empty_like(layer.out) for _ in range(2)]
    h2d_s, d2h_s = torch.cuda.Stream(), torch.cuda.Stream()

    def e2e_run(n):
        ev = lambda: torch.cuda.Event()
        h2d_done = [ev(), ev()]
        comp_done = [ev(), ev()]
        d2h_done = [ev(), ev()]
        used = [False, False]
        # nothing of the run may start before the region's start marker
        start = ev()
        start.record(stream)
        h2d_s.wait_event(start)
        d2h_s.wait_event(start)

        def h2d(i):
            b = i % 2
            if used[b]:
                h2d_s.wait_event(comp_done[b])  # step i-2 has finished reading x_dev[b]
            with torch.cuda.stream(h2d_s):
                x_dev[b].copy_(x_host, non_blocking=True)
            h2d_done[b].record(h2d_s)

        h2d(0)
        for i in range(n):
            b = i % 2
            if i + 1 < n:
                h2d(i + 1)
            stream.wait_event(h2d_done[b])
            if used[b]:
                stream.wait_event(d2h_done[b])  # step i-2's output has been read back
            layer.forward(x_dev[b], out=out_dev[b], load_group=lg, gated=gated)
            comp_done[b].record(stream)
            used[b] = True
            d2h_s.wait_event(comp_done[b])
            with torch.cuda.stream(d2h_s):
                out_host[b].copy_(out_dev[b], non_blocking=True)
            d2h_done[b].record(d2h_s)
        stream.wait_event(d2h_done[(n - 1) % 2])

    e2e_run(2)
    torch.cuda.synchronize()
    barrier(world)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    e2e_run(K)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), world)
    status = moe.moe_get_device_error()
    if status != 0:
        raise RuntimeError(f"device error status {status} in the end-to-end region")

    peaks = load_peaks()
    tokens = world * shape.T * K
    value = tokens / (total_ms * 1e-3)
    exp_mean = statistics.mean(exp_ms)
    achieved = expert_flops(shape) / (exp_mean * 1e-3) / 1e12
    if shape.dtype == "fp8":
        # no measured FP8 figure: the measured bf16 peak times the nominal
        # dense FP8 : bf16 ratio of B300 (4.5 : 2.25 PFLOP/s)
        peak = 2.0 * peaks["bf16_tflops"]
        peak_sust = 2.0 * peaks.get("bf16_tflops_sustained", peaks["bf16_tflops"])
        peak_kind = f"fp8 dense = 2 x bf16 dense burst, {peaks['_source']}"
    else:
        peak = peaks["bf16_tflops"]
        peak_sust = peaks.get("bf16_tflops_sustained", peak)
        peak_kind = f"bf16 dense burst, {peaks['_source']}"
    # this replica's loads (counts hold the summed loads when replicas > 1)
    ebytes, touched = expert_bytes(shape, np.diff(layer.offsets.cpu().numpy()))
    hbm_achieved = ebytes / (exp_mean * 1e-3) / 1e9
    # the bf16 calls run pair MMAs when the segments average >= 128 rows
    kname = (f"experts_{shape.dtype}_kernel" if shape.dtype != "bf16" or args.dispatch == "gather"
             or shape.T * shape.k < 128 * shape.E else "experts_bf16_pair_kernel")
    kernel = f"{kname} (gate/up + down launches of one moe_experts_grouped call)"
    traffic = kernel_traffic(shape.dtype, shape.name)
    if shape.T * shape.k < 16 * shape.E:  # fewer than 16 rows per expert on average
        # decode-sized batch: the expert GEMMs stream the touched weights
        roofline = {"bound": "hbm", "kernel": kernel, "achieved": hbm_achieved,
                    "peak": peaks["hbm_gbs"], "unit": "GB/s",
                    "frac": hbm_achieved / peaks["hbm_gbs"],
                    "peak_kind": f"HBM copy bandwidth, {peaks['_source']}",
                    "algorithmic_bytes": ebytes, "experts_touched": touched,
                    "traffic": traffic, "expert_ms_per_step": exp_mean}
    else:
        roofline = {"bound": "tensor", "kernel": kernel, "achieved": achieved, "peak": peak,
                    "unit": "TFLOP/s", "frac": achieved / peak,
                    "peak_kind": peak_kind, "frac_of_sustained": achieved / peak_sust,
                    "hbm_gbs": hbm_achieved, "hbm_frac": hbm_achieved / peaks["hbm_gbs"],
                    "algorithmic_bytes": ebytes, "traffic": traffic,
                    "expert_ms_per_step": exp_mean}
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": total_ms / K, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": shape.dtype, "data": "synthetic",
        "config": {"workload": describe(shape), "global_batch": world * shape.T,
                   "dispatch": "gather rows inside the gate/up GEMM" if gather
                               else "permute kernel before the expert GEMMs",
                   "combine": "gates folded into the down projection; combine adds rows"
                              if gated else "combine multiplies rows by their gates",
                   "parallelism": f"data-parallel replicas x{world}, one all-reduce of the "
                                  f"per-expert loads per step" if world > 1 else "single GPU",
                   "l2": "inputs larger than L2: every step streams all expert weights "
                         f"({(3 * shape.d * shape.inter * (shape.E + shape.n_shared)) * (1 if shape.dtype == 'fp8' else 2) / 1e9:.1f} GB)"},
        "layer_tflops": layer_flops(shape) * world * K / (total_ms * 1e-3) / 1e12,
        # each step's own events (this rank): the median and the best of the K steps
        "per_step": {"layer_ms_median": statistics.median(step_ms), "layer_ms_best": min(step_ms),
                     "expert_ms_median": statistics.median(exp_ms), "expert_ms_best": min(exp_ms),
                     "frac_at_best_expert_ms": roofline["frac"] * exp_mean / min(exp_ms)},
        "roofline": roofline,
        "e2e": {"value": tokens / (e2e_ms * 1e-3), "unit": "tokens/s",
                "h2d_bytes_per_step": x_host.numel() * x_host.element_size(),
                "d2h_bytes_per_step": out_host[0].numel() * out_host[0].element_size(),
                "copies": "pipelined on two copy streams (double-buffered)"},
        "gpu_launches": (launches_per_step(shape, gather) + (1 if gated else 0)) * K,
        "clocks": clk,
    }
    if shape.bias_steps:
        line["load_balance"] = load_balance(moe, shape, L, shape.bias_steps)
    if cpu_baseline and rank == 0 and world == 1 and not args.no_cpu_baseline:
        secs, n = oracle_sample(shape, L, args.cpu_tokens)
        line["cpu_baseline"] = {
            "value": n / secs, "unit": "tokens/s", "cores": blas_threads(), "kind": "oracle",
            "sample": f"{n} tokens of the same batch end to end through the fp64 oracle "
                      f"({secs:.1f} s)"}
    # release this workload's weights and buffers before the next one
    del layer, L, x, x_host, x_dev, out_dev, out_host
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return line


def run_train(args, shape, world, rank, local):
    """One training step per iteration: forward (with the bias update) and
    the whole backward, inputs and dL/dy resident on the device."""
    import mixture_experts_layer_82_b300 as moe
    from moe_synth import make_grad

    if shape.dtype not in ("bf16", "fp8"):
        raise SystemExit("--train: the backward pass is implemented for the bf16 and fp8 kinds")
    fp8 = shape.dtype == "fp8"
    if fp8 and args.dispatch == "gather":
        raise SystemExit("--train: the gathering forward is implemented for the bf16 kind")
    dev = f"cuda:{local}"
    torch.cuda.set_device(local)
    L = make_layer(shape, dev)
    cfg = moe.LayerCfg.from_shape(shape)
    gather = args.dispatch == "gather"
    layer = moe.MoELayer(cfg, L["router_w"], L["bias"].clone(), L["w13"], L["w2"],
                         L["ws13"] if shape.n_shared else None, L["ws2"] if shape.n_shared else None,
                         gather=gather)
    x = L["x"]
    dout = make_grad(shape, dev)
    aff = torch.empty(shape.T, shape.E, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()

    lg = None
    if world > 1:
        import torch.distributed as dist
        lg = dist.group.WORLD

    def step(xx, gg, ev=None):
        layer.forward(xx, affinity_out=aff, expert_events=None if ev is None else ev[0:2],
                      keep=not gather, load_group=lg)
        return layer.backward(xx, gg, aff, events=None if ev is None else ev[2:6])

    for _ in range(args.warmup):
        step(x, dout)
    torch.cuda.synchronize()
    if moe.moe_get_device_error() != 0:
        raise RuntimeError("device error after warm-up")

    K = args.steps
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(6)] for _ in range(K)]
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(local)
    clocks.start()
    barrier(world)
    torch.cuda.synchronize()
    t_start.record(stream)
    for i in range(K):
        step(x, dout, evs[i])
    t_end.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    clk = clocks.stop()
    total_ms = max_over_ranks(t_start.elapsed_time(t_end), world)
    parts = {"forward experts": [e[0].elapsed_time(e[1]) for e in evs],
             "backward experts, input (Dgrad)": [e[2].elapsed_time(e[3]) for e in evs],
             "backward experts, weights (Wgrad)": [e[4].elapsed_time(e[5]) for e in evs]}
    if moe.moe_get_device_error() != 0:
        raise RuntimeError("device error in the timed region")

    # ---- end to end: x and dL/dy from pinned host memory, dL/dx back, every
    # step, on the compute stream (no overlap)
    x_host = x.cpu().pin_memory()
    g_host = dout.cpu().pin_memory()
    dx_host = torch.empty(shape.T, shape.d, dtype=torch.bfloat16).pin_memory()
    x_dev, g_dev = torch.empty_like(x), torch.empty_like(dout)

    def e2e_step():
        x_dev.copy_(x_host, non_blocking=True)
        g_dev.copy_(g_host, non_blocking=True)
        dx_host.copy_(step(x_dev, g_dev), non_blocking=True)

    e2e_step()
    torch.cuda.synchronize()
    barrier(world)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(K):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), world)
    if moe.moe_get_device_error() != 0:
        raise RuntimeError("device error in the end-to-end region")

    peaks = load_peaks()
    peak = peaks["bf16_tflops"]
    peak_sust = peaks.get("bf16_tflops_sustained", peak)
    peak_kind = f"bf16 dense burst, {peaks['_source']}"
    if fp8:
        # the measured bf16 peak times the nominal dense FP8 : bf16 ratio
        # of B300 (4.5 : 2.25 PFLOP/s)
        peak, peak_sust = 2.0 * peak, 2.0 * peak_sust
        peak_kind = f"fp8 dense = 2 x bf16 dense burst, {peaks['_source']}"
    bf = backward_flops(shape)
    alg = {"forward experts": expert_flops(shape),
           "backward experts, input (Dgrad)": bf["dgrad"],
           "backward experts, weights (Wgrad)": bf["wgrad"]}
    breakdown = {}
    for k, v in parts.items():
        m = statistics.mean(v)
        breakdown[k] = {"ms_per_step": m, "algorithmic_tflop": alg[k] / 1e12,
                        "tflops": alg[k] / (m * 1e-3) / 1e12}
    dom = max(breakdown, key=lambda k: breakdown[k]["ms_per_step"])
    achieved = breakdown[dom]["tflops"]
    tokens = world * shape.T * K
    # expert forward, Dgrad and Wgrad, and the dense router product; the
    # router backward touches only the K selected centroids (4 T K d, small)
    step_flops = expert_flops(shape) + bf["dgrad"] + bf["wgrad"] + 2.0 * shape.T * shape.d * shape.E
    line = {
        "metric": METRIC_TRAIN, "value": tokens / (total_ms * 1e-3), "unit": "tokens/s",
        "n_gpus": world, "steps": K, "warmup": args.warmup, "ms_per_step": total_ms / K,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": shape.dtype,
        "data": "synthetic",
        "config": {"workload": describe(shape), "global_batch": world * shape.T,
                   "step": "forward in FP8 (route, quantise + permute, experts keeping [a|b], "
                           "combine, bias update) + backward (combine, experts Dgrad in FP8, "
                           "router, experts Wgrad in FP8)"
                           if fp8 else
                           "forward (route, permute, experts keeping [a|b], combine, bias update) + "
                           "backward (combine, experts Dgrad, router, experts Wgrad)"
                           if not gather else
                           "forward (route, experts gathering rows, combine, bias update) + backward "
                           "(permute, combine, experts Dgrad with [a|b] recomputed, router, experts Wgrad)",
                   "parallelism": f"data-parallel replicas x{world}, one all-reduce of the "
                                  f"per-expert loads per step" if world > 1 else "single GPU",
                   "l2": "inputs larger than L2: every step streams all expert weights and "
                         "writes all weight gradients"},
        "layer_tflops": step_flops * world * K / (total_ms * 1e-3) / 1e12,
        "roofline": {"bound": "tensor", "kernel": dom, "achieved": achieved, "peak": peak,
                     "unit": "TFLOP/s", "frac": achieved / peak,
                     "peak_kind": peak_kind,
                     "frac_of_sustained": achieved / peak_sust, "traffic": None,
                     "breakdown": breakdown,
                     "recompute_tflop_not_counted": bf["recompute"] / 1e12 if gather else 0.0},
        "e2e": {"value": tokens / (e2e_ms * 1e-3), "unit": "tokens/s",
                "h2d_bytes_per_step": 2 * x_host.numel() * x_host.element_size(),
                "d2h_bytes_per_step": dx_host.numel() * dx_host.element_size(),
                "copies": "x and dL/dy in, dL/dx out, on the compute stream"},
        "gpu_launches": train_launches(shape, gather) * K,
        "clocks": clk,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        secs, n = oracle_train_sample(shape, L, args.cpu_tokens)
        line["cpu_baseline"] = {
            "value": n / secs, "unit": "tokens/s", "cores": blas_threads(), "kind": "oracle",
            "sample": f"{n} tokens of the same batch through the fp64 oracle forward and "
                      f"backward ({secs:.1f} s)"}
    if rank == 0:
        print(json.dumps(line), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="v3_bf16", choices=sorted(CONFIGS))
    ap.add_argument("--cpu-tokens", type=int, default=8)
    ap.add_argument("--ref-tokens", type=int, default=2)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-also", action="store_true",
                    help="with the default workload, time it alone (without the FP8 and "
                         "decode-shaped layers reported under \"also\")")
    ap.add_argument("--dispatch", choices=["permute", "gather"], default="permute",
                    help="bf16 kind: permute x into per-expert rows before the expert GEMMs, "
                         "or gather the rows inside the gate/up GEMM")
    ap.add_argument("--gated", action="store_true",
                    help="fold the gate multiply into the down projection "
                         "(moe_experts_grouped_gated); the combine then only adds rows")
    ap.add_argument("--train", action="store_true",
                    help="time a training step (forward + backward; bf16 kind)")
    ap.add_argument("--set", action="append", default=[], metavar="FIELD=VALUE",
                    help="override a field of the workload's shape (a reduced case for "
                         "profiling, e.g. --set E=32 --set router=gaussian)")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)  # timing rule: at least 3 untimed steps
    shape = CONFIGS[args.workload]
    if args.set:
        from dataclasses import fields
        from moe_synth import shape_with
        types = {f.name: f.type for f in fields(shape)}
        kw = {}
        for item in args.set:
            k, v = item.split("=", 1)
            if k not in types:
                ap.error(f"--set: unknown shape field {k!r}")
            t = types[k] if not isinstance(types[k], str) else {"int": int, "float": float,
                                                                 "str": str}[types[k]]
            kw[k] = t(v)
        shape = shape_with(shape, **kw)
    world, rank, local = dist_setup(args.gpus)
    try:
        if args.impl == "reference":
            return run_reference(args, shape, world, rank)
        if args.train:
            return run_train(args, shape, world, rank, local)
        return run_ours(args, shape, world, rank, local)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    sys.exit(main())
