"""Multi-process (world size 2, gloo, CPU) checks of the replica
coordination used by bench.py for N > 1 GPUs."""

import os
import socket

import pytest
import torch.multiprocessing as mp

from exact_attention_78_gb300 import replicas


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(world), RANK=str(rank),
                      LOCAL_RANK=str(rank))
    assert replicas.rank_env() == (world, rank, rank)
    replicas.init("gloo")
    replicas.barrier()
    elapsed = 10.0 + rank * 2.5            # each rank "timed" a different duration
    out[rank] = replicas.max_over_ranks(elapsed)
    replicas.barrier()
    replicas.finalize()


def test_max_over_two_gloo_ranks():
    world, port = 2, _free_port()
    out = mp.get_context("spawn").Manager().dict()   # no fork of this multi-threaded process
    mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
    assert out[0] == out[1] == 12.5


@pytest.mark.parametrize("B,Hkv,world", [(2, 16, 2), (64, 8, 3), (1, 1, 2), (4, 16, 8)])
def test_shards_are_disjoint_and_cover(B, Hkv, world):
    seen = []
    for r in range(world):
        s = replicas.shard(B, Hkv, r, world)
        assert abs(len(s) - (B * Hkv) / world) < 1
        seen += s
    assert sorted(seen) == [(b, h) for b in range(B) for h in range(Hkv)]


def test_not_distributed_is_identity():
    assert replicas.max_over_ranks(3.25) == 3.25
    replicas.barrier()
