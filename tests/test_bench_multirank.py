"""The benchmark's multi-rank aggregation (replicas, weak scaling) on two gloo
ranks on the CPU: the job time is the slowest rank's, the value sums ranks."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    ms = [2.5, 3.75][rank]
    m = bench.max_over_ranks(ms, dist, "cpu")
    q.put((rank, m, bench.job_tokens_per_s(8, world, m)))
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks():
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
    assert [r[1] for r in res] == [3.75, 3.75]
    assert res[0][2] == pytest.approx(8 * 2 / 3.75e-3)


def test_single_rank_identity():
    assert bench.max_over_ranks(1.5, None, "cpu") == 1.5
