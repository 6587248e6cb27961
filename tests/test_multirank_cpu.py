"""The multi-rank bookkeeping of bench.py on CPU with gloo, world size 2: each rank gets its own
batch of the same shape, the step time is the slowest rank's, and the job throughput counts the
bytes of every rank.  (The attention path itself has no collective: requests shard across GPUs.)"""

import os
import socket

import pytest
import torch
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, out):
    import torch.distributed as dist

    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench

        b = bench.rank_batch(2, rank, scale_batch=0.05)
        fake_ms = 10.0 + 5.0 * rank  # rank 1 is the slow one
        m = bench.max_over_ranks(fake_ms)
        sig = torch.tensor([float(b.kv_len.sum()), float(b.kv_indices[:8].sum())], dtype=torch.float64)
        gathered = [torch.zeros_like(sig) for _ in range(world)]
        dist.all_gather(gathered, sig)
        out[rank] = (m, b.kv_bytes_read(), [g.tolist() for g in gathered], b.batch_size)
    finally:
        dist.destroy_process_group()


def test_two_ranks_shard_batches_and_reduce_time():
    world = 2
    port = _free_port()
    mgr = mp.get_context("spawn").Manager()  # no fork of this (multi-threaded) process
    out = mgr.dict()
    mp.start_processes(_worker, args=(world, port, out), nprocs=world, join=True, start_method="spawn")
    (m0, b0, g0, n0), (m1, b1, g1, n1) = out[0], out[1]
    assert m0 == m1 == 15.0  # both ranks report the slowest rank
    assert n0 == n1  # same shape on every rank
    assert g0[0] != g0[1]  # but different requests (own seed per rank)
    import bench

    v = bench.aggregate_gbs(b0, 10, world, 15.0)
    assert v == pytest.approx(b0 * 10 * 2 / 15e-3 / 1e9)
