"""Host-side logic of bench.py for N > 1 replicas, on CPU with two gloo ranks.

Each rank times its own replica; the reported time is the max over ranks and the throughput
counts the work of every rank.  No data-path collective exists (the units are independent).
"""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        bench.barrier(world)
        t = bench.max_over_ranks(1.0 + rank * 2.5, world)
        q.put((rank, t))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    assert all(p.exitcode == 0 for p in procs)
    got = dict(q.get(timeout=10) for _ in range(2))
    assert got == {0: 3.5, 1: 3.5}


def test_single_rank_is_identity():
    import bench
    assert bench.max_over_ranks(2.0, 1) == 2.0
    bench.barrier(1)


def test_algorithmic_counts():
    import bench
    # 1,152 bytes per token-head for bf16 q, k, v, out at dk = 96, dv = 192
    assert bench.prefill_bytes(1, 1, 1, 96, 192, False, False) == 1152
    assert bench.prefill_bytes(8, 2048, 16, 96, 192, False, True) == 8 * 2048 * 16 * 1152 + 8 * 16 * 96 * 192 * 4
    # 147,456 issued FLOPs per token-head at chunk 128
    assert bench.prefill_flops(1, 1, 1, 96, 192, 128) == 147456
    state, io = bench.decode_bytes(1280, 16, 96, 192)
    assert state == 1280 * 16 * 96 * 192 * 8 and io == 1280 * 16 * 576 * 2


def test_backward_counts():
    import bench
    # the method's bytes: q, k, v, dout read and dq, dk, dv written once in bf16, 1,920 B per token-head at
    # dk = 96, dv = 192; dh0 (f32) per chain
    assert bench.backward_bytes(1, 1, 1, 96, 192, with_dh0=False) == 2 * (2 * 96 + 2 * 192) + 2 * (2 * 96 + 192) == 1920
    assert bench.backward_bytes(8, 2048, 16, 96, 192) == 8 * 2048 * 16 * 1920 + 8 * 16 * 96 * 192 * 4
    # what this implementation moves on top: the state passes' second read of q, k, v, dout and the bf16
    # state images (two 96 x 192 tiles per 128-token chunk, written and read once)
    assert bench.backward_impl_bytes(1, 1, 1, 96, 192) == 2 * 576 + 8 * 96 * 192 // 128 == 2304
    # FLOPs of the chunked backward: six score / gradient contractions over the chunk plus the three
    # inter-chunk terms and the gradient-state recurrence
    assert bench.backward_flops(1, 1, 1, 96, 192, 128) == 6 * 128 * 288 + 8 * 96 * 192
