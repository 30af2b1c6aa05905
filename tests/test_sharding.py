"""Multi-rank host logic on CPU: sequence partitioning and the max-over-ranks
timing reduction, run as two gloo processes (world_size 2)."""
import os
import socket

import numpy as np
import pytest
import torch.multiprocessing as mp

from gated_deltanet_linear_mixer_gb300 import sharding


def test_partition_covers_every_sequence_once_and_balances():
    rng = np.random.default_rng(3)
    lens = rng.integers(128, 8193, 16).tolist()
    for world in (1, 2, 3, 4, 8):
        parts = sharding.partition_sequences(lens, world)
        flat = sorted(i for p in parts for i in p)
        assert flat == list(range(16))
        loads = [sum(lens[i] for i in p) for p in parts]
        # greedy longest-first: imbalance at most one (largest) sequence
        assert max(loads) - min(loads) <= max(lens)
    assert sharding.partition_sequences([5, 5, 5, 5], 2) == [[0, 2], [1, 3]]


def test_local_rows_reassemble_the_batch():
    cu = np.array([0, 3, 3, 10, 12], dtype=np.int32)
    rows, cu_l = sharding.local_rows(cu, [0, 2, 3])
    assert rows.tolist() == [0, 1, 2, 3, 4, 5, 6, 7, 8, 9, 10, 11]
    assert cu_l.tolist() == [0, 3, 10, 12]
    rows, cu_l = sharding.local_rows(cu, [3])
    assert rows.tolist() == [10, 11] and cu_l.tolist() == [0, 2]
    rows, cu_l = sharding.local_rows(cu, [])
    assert rows.size == 0 and cu_l.tolist() == [0]


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        lens = [700, 100, 300, 300, 50]
        parts = sharding.partition_sequences(lens, world)
        mine = parts[rank]
        t = sharding.max_over_ranks(1.5 + rank)       # per-rank "time"
        tok = sum(lens[i] for i in mine)
        q.put((rank, mine, t, tok))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_partition_and_reduce():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(2))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    (r0, m0, t0, k0), (r1, m1, t1, k1) = res
    assert sorted(m0 + m1) == [0, 1, 2, 3, 4]
    assert t0 == t1 == 2.5                            # max over ranks
    assert k0 + k1 == 1450
