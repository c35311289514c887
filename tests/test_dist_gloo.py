"""The multi-rank host logic on CPU: world size 2 over gloo (no GPU)."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from dflash2_block_drafter_gb300.dist import aggregate_throughput, shard_blocks


def test_shard_blocks_covers_every_block_once():
    for total in (0, 1, 7, 64, 1000):
        for world in (1, 2, 3, 8):
            seen = []
            for r in range(world):
                lo, n = shard_blocks(total, world, r)
                seen.extend(range(lo, lo + n))
                assert abs(n - total / world) < 1
            assert seen == list(range(total))
    with pytest.raises(ValueError):
        shard_blocks(4, 2, 2)


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        lo, n = shard_blocks(128, world, rank)
        # rank 1 is the slow one: the job's time is its time
        ms = 10.0 if rank == 0 else 25.0
        value, blocks, max_ms = aggregate_throughput(n, ms)
        out[rank] = (lo, n, value, blocks, max_ms)
    finally:
        dist.destroy_process_group()


def test_two_ranks_aggregate_over_gloo():
    world = 2
    port = _free_port()
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_worker, args=(world, port, out), nprocs=world, start_method="spawn", join=True)
    assert out[0][:2] == (0, 64) and out[1][:2] == (64, 64)
    for r in range(world):
        value, blocks, max_ms = out[r][2:]
        assert blocks == 128
        assert max_ms == 25.0
        assert value == pytest.approx(128 / 0.025)


def test_single_process_aggregate():
    value, blocks, max_ms = aggregate_throughput(64, 2.0)
    assert (blocks, max_ms) == (64, 2.0)
    assert value == pytest.approx(32000.0)
