"""The benchmark's multi-process path (one process per GPU under torchrun),
exercised on the CPU with the gloo backend and two ranks: rendezvous, the
barrier around the timed region, the maximum of the per-rank times, the
reference arm's rule that only rank 0 runs the oracle, and the one exchange
of data-parallel replicas (the per-expert loads summed for the bias
update)."""

import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(world),
                      RANK=str(rank), LOCAL_RANK=str(rank))
    import argparse

    import bench
    from moe_synth import CONFIGS

    w, r, local = bench.dist_setup(world)
    assert (w, r, local) == (world, rank, rank)
    bench.barrier(w)
    # each rank "measured" a different time; every rank must see the largest
    t = bench.max_over_ranks(3.0 + 10.0 * rank, w)
    ref = None
    if rank != 0:
        # the reference arm: ranks other than 0 exit at once, without work
        args = argparse.Namespace(warmup=3, steps=1, ref_tokens=1)
        ref = bench.run_reference(args, CONFIGS["v3_bf16"], w, r)
    bench.barrier(w)
    import torch.distributed as dist
    dist.destroy_process_group()
    with open(os.path.join(out_dir, f"rank{rank}.txt"), "w") as f:
        f.write(f"{t} {ref}")


def test_two_ranks_gloo(tmp_path):
    world = 2
    mp.start_processes(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world,
                       join=True, start_method="spawn")
    got = [open(tmp_path / f"rank{r}.txt").read().split() for r in range(world)]
    assert [float(g[0]) for g in got] == [13.0, 13.0]
    assert got[1][1] == "0"


def test_single_process_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    for k in ("WORLD_SIZE", "RANK", "LOCAL_RANK"):
        os.environ.pop(k, None)
    world, rank, local = bench.dist_setup(1)
    assert (world, rank, local) == (1, 0, 0)
    bench.barrier(world)
    assert bench.max_over_ranks(2.5, world) == 2.5


def _load_rank(rank, world, port, out_dir):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(world),
                      RANK=str(rank), LOCAL_RANK=str(rank))
    import numpy as np
    import torch
    import torch.distributed as dist

    import oracle
    from mixture_experts_layer_82_b300.replicas import global_cfg, global_load
    from mixture_experts_layer_82_b300 import LayerCfg
    from moe_synth import CONFIGS, make_layer, shape_with

    dist.init_process_group("gloo", rank=rank, world_size=world)
    shape = shape_with(CONFIGS["tiny_fp32"], T=48)
    L = make_layer(shape, weights=False)
    x = L["x"].double().numpy()
    s = oracle.sigmoid_affinity(x, L["router_w"].double().numpy()).astype(np.float32)
    b = L["bias"].numpy()
    half = shape.T // world
    mine = slice(rank * half, (rank + 1) * half)
    idx = oracle.select_experts(s[mine], b, shape.n_groups, shape.topk_groups, shape.k)
    counts = torch.from_numpy(oracle.expert_load(idx, shape.E).astype(np.int32))
    n = global_load(counts)
    cfg = global_cfg(LayerCfg.from_shape(shape, T=half), n)
    bias = oracle.bias_update(b, counts.numpy(), cfg.T, cfg.k, cfg.gamma)
    dist.destroy_process_group()
    np.save(os.path.join(out_dir, f"load{rank}.npy"), counts.numpy())
    np.save(os.path.join(out_dir, f"bias{rank}.npy"), bias)


def test_replicas_sum_their_loads_for_the_bias_update(tmp_path):
    import numpy as np

    import oracle
    from moe_synth import CONFIGS, make_layer, shape_with
    world = 2
    mp.start_processes(_load_rank, args=(world, _free_port(), str(tmp_path)), nprocs=world,
                       join=True, start_method="spawn")
    # one process routing the whole batch
    shape = shape_with(CONFIGS["tiny_fp32"], T=48)
    L = make_layer(shape, weights=False)
    s = oracle.sigmoid_affinity(L["x"].double().numpy(),
                                L["router_w"].double().numpy()).astype(np.float32)
    idx = oracle.select_experts(s, L["bias"].numpy(), shape.n_groups, shape.topk_groups, shape.k)
    whole = oracle.expert_load(idx, shape.E)
    ref = oracle.bias_update(L["bias"].numpy(), whole, shape.T, shape.k, shape.gamma)
    for r in range(world):
        assert np.array_equal(np.load(tmp_path / f"load{r}.npy"), whole)
        assert np.array_equal(np.load(tmp_path / f"bias{r}.npy").view(np.uint32), ref.view(np.uint32))
