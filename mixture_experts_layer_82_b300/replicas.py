"""Data-parallel replicas of the layer: the one exchange they need.

"DeepSeek-V3 Technical Report", auxiliary-loss-free load balancing
paragraph: at the end of each step the bias of expert i moves by gamma
according to whether i was overloaded over the whole batch.  With the batch
split over data-parallel replicas (one process per GPU, each routing its
own tokens), the whole-batch load is the sum of the replicas' per-expert
loads: one all-reduce of counts[E] (int32, 4 E bytes) per step, after which
every replica applies the same sign rule against the global batch of
world * T tokens, so the replicas' biases stay identical.  Nothing else of
the layer crosses GPUs: tokens, experts' inputs and outputs stay local.
"""

from __future__ import annotations

import copy


def global_load(counts, group=None, stream=None):
    """Sums ``counts`` (the per-expert loads of this replica's batch) over
    the replicas of ``group`` in place; returns the number of replicas.

    ``stream`` (device tensors): the stream the routing that wrote
    ``counts`` was enqueued on (a torch.cuda.Stream or a raw handle; None is
    torch's current stream).  The all-reduce is issued with that stream
    current, so that it reads the loads after the routing and the bias
    update enqueued next on it reads the sums."""
    import torch
    import torch.distributed as dist

    if counts.is_cuda and stream is not None:
        if not isinstance(stream, torch.cuda.Stream):
            stream = torch.cuda.ExternalStream(int(stream), device=counts.device)
        with torch.cuda.stream(stream):
            dist.all_reduce(counts, op=dist.ReduceOp.SUM, group=group)
    else:
        dist.all_reduce(counts, op=dist.ReduceOp.SUM, group=group)
    return dist.get_world_size(group)


def global_cfg(cfg, world):
    """The layer configuration of the whole batch: the same layer over
    world * T tokens (what the bias update's mean load is taken over)."""
    g = copy.copy(cfg)
    g.T = cfg.T * world
    return g
