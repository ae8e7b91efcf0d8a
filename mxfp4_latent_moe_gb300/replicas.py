"""Replica data parallelism for the layer.

The layer has no exchange between tokens: routing, grouping, both expert
GEMMs and the combine of one token read only that token's activations and the
expert weights, of which each GPU holds a full copy. Several GPUs therefore run independent replicas,
one process per GPU, each on its own batch of tokens, with no collective on
the data path. The only cross-rank steps are host-side: a barrier before the
timed region and a max over the ranks' elapsed times after it, so that the
aggregate throughput is the tokens all ranks processed divided by the slowest
rank's time.

Works with any torch.distributed backend (nccl on GPUs, gloo on CPU); with no
process group initialised every function is the single-process identity.
"""
import os

import torch


def dist_env():
    """(rank, world_size, local_rank) from the torchrun environment."""
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def _active():
    return torch.distributed.is_available() and torch.distributed.is_initialized()


def replica_seed(seed, rank):
    """Each replica draws its own batch: seed + rank."""
    return int(seed) + int(rank)


def barrier():
    if _active():
        torch.distributed.barrier()


def max_over_ranks(value, device=None):
    """The largest of the ranks' `value` (a float), on every rank."""
    if not _active():
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def aggregate_rate(units_per_rank, world, steps, max_ms):
    """Whole-job throughput: units all ranks processed / the slowest rank's time."""
    if max_ms <= 0:
        raise ValueError("elapsed time must be positive")
    return world * units_per_rank * steps / (max_ms / 1e3)
