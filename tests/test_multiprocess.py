"""The benchmark's multi-process path (one process per GPU under torchrun),
exercised on the CPU with the gloo backend and two ranks: rendezvous, the
barrier around the timed region, the maximum of the per-rank times, and the
reference arm's rule that only rank 0 runs the oracle."""

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
