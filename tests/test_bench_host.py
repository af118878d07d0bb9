"""Host logic of bench.py: algorithmic work counts and the multi-rank timing
reduction (world size 2 over gloo on the CPU)."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

import bench
import workloads


def test_decode_bytes_counts_visible_kv_once():
    b = workloads.paged_batch(3, [1, 1], [10, 33], 8, 2, 128, 16, "bf16")
    kv = (10 + 33) * 2 * 128 * 2 * 2
    qo = 2 * 2 * 8 * 128 * 2
    lse = 2 * 8 * 4
    meta = 4 * (len(b.kv_indices) + 2 * 3 + 2)
    assert bench.decode_bytes(b) == kv + qo + lse + meta


def test_prefill_flops_causal_pairs():
    b = workloads.paged_batch(4, [3, 2], [3, 5], 4, 2, 128, 16, "bf16", causal=True)
    # request 0: 1 + 2 + 3 visible pairs; request 1 (kv 5, qo 2): 4 + 5
    assert bench.prefill_flops(b) == 4.0 * 128 * 4 * (6 + 9)


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=world)
    bench.barrier(world)
    mx = bench.max_over_ranks(1.0 + rank, world)
    sm = bench.sum_over_ranks(10.0 * (rank + 1), world)
    out[rank] = (mx, sm)
    dist.destroy_process_group()


def test_two_rank_timing_reduction():
    world = 2
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    assert res[0] == res[1] == (2.0, 30.0)
