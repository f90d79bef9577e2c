"""Coordination of one-replica-per-GPU runs (one process per GPU).

Attention shards over (batch, key/value head) with no exchange, so a
multi-GPU run is N independent replicas; the only collectives are the ones a
benchmark needs: a barrier around the timed region and the maximum of the
per-rank elapsed times.  `shard` gives the (batch, kv-head) pairs a rank owns
when one problem is split across ranks instead.
"""

import os

import torch


def rank_env():
    """(world_size, rank, local_rank) from the torch.distributed launcher env."""
    return (int(os.environ.get("WORLD_SIZE", "1")), int(os.environ.get("RANK", "0")),
            int(os.environ.get("LOCAL_RANK", "0")))


def init(backend, device=None):
    import torch.distributed as dist
    if device is not None and backend == "nccl":
        dist.init_process_group(backend, device_id=device)
    else:
        dist.init_process_group(backend)


def barrier():
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        dist.barrier()


def max_over_ranks(value, device="cpu"):
    """Largest `value` over all ranks (the value itself when not distributed)."""
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def shard(B, Hkv, rank, world):
    """(b, kv_head) pairs owned by `rank`: contiguous, sizes differ by <= 1.
    A whole query-head group stays on one rank, so dK/dV need no reduction."""
    pairs = [(b, h) for b in range(B) for h in range(Hkv)]
    n = len(pairs)
    lo = rank * n // world
    hi = (rank + 1) * n // world
    return pairs[lo:hi]


def finalize():
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        dist.destroy_process_group()
