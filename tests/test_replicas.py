"""Replica coordination for bench.py --gpus N, on CPU with gloo (world size 2)."""
import os
import socket

import pytest
import torch.multiprocessing as mp

from lfm2_gated_short_gb300 import replicas


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    r, w, lr = replicas.env_rank()
    g = replicas.Group(w, backend="gloo")
    g.barrier()
    m = g.max(10.0 * (rank + 1))           # rank 1 is the slowest replica
    v = replicas.aggregate_gbs(1_000_000_000, 4, w, m)
    g.barrier()
    g.close()
    out.put((r, w, lr, m, v))


def test_two_replicas_take_the_slowest_rank_and_sum_bytes():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for r, (rank, world, local, m, v) in enumerate(res):
        assert (rank, world, local) == (r, 2, r)
        assert m == 20.0
        # 2 ranks x 4 steps x 1 GB in 20 ms
        assert v == pytest.approx(2 * 4 * 1.0 / 0.020)


def test_single_process_needs_no_process_group():
    g = replicas.Group(1)
    g.barrier()
    assert g.max(3.5) == 3.5
    assert replicas.aggregate_gbs(2_000_000_000, 1, 1, 1000.0) == pytest.approx(2.0)
    with pytest.raises(ValueError):
        replicas.aggregate_gbs(1, 1, 1, 0.0)
