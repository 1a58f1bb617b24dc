"""The host side of expert parallelism across ranks, on CPU with gloo
(world size 2 and 3): every rank owns a contiguous shard of the experts
(``ep.shard_range``), computes its partial output (here the oracle's shard,
rounded to bf16 as the GPU's partial is) and ``ep.combine_partials`` sums
the partials over the ranks; the sum must equal the whole layer."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import synthetic_inputs as si
        from nvfp4_mixture_experts_moe_gb300 import ep
        from oracle import moe as omoe
        cfg = si.LayerConfig("ep_gloo", T=12, H=128, I=64, I_s=64, E=7, k=3)
        lo, hi = ep.shard_range(cfg.E, world, rank)
        W = si.make_layer_weights(cfg, threads=1)
        trips = {e: tuple(omoe.QuantWeight.from_dense(m.float().numpy()) for m in W[e]) for e in W}
        x = si.make_x(cfg).float().numpy().astype(np.float64)
        logits = si.make_logits(cfg).numpy()
        experts = [trips[e] for e in range(cfg.E)]
        part = omoe.layer(x, logits, experts, trips[cfg.E] if rank == 0 else None, cfg.k, experts_range=(lo, hi))
        out = ep.combine_partials(torch.from_numpy(part).to(torch.bfloat16))
        if rank == 0:
            full = omoe.layer(x, logits, experts, trips[cfg.E], cfg.k)
            err = float(np.abs(out.float().numpy() - full).max())
            bound = float((world + 1) * 2.0 ** -8 * np.abs(full).max() + 1e-6)
            q.put((lo, hi, err, bound))
        else:
            q.put((lo, hi, None, None))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 3])
def test_expert_parallel_exchange_gloo(world):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    results = [q.get(timeout=240) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    shards = sorted((lo, hi) for lo, hi, _, _ in results)
    assert shards[0][0] == 0 and shards[-1][1] == 7
    assert all(a[1] == b[0] for a, b in zip(shards, shards[1:]))     # contiguous, no gaps
    (err, bound), = [(e, b) for _, _, e, b in results if e is not None]
    assert err <= bound, (err, bound)


def test_shard_ranges():
    from nvfp4_mixture_experts_moe_gb300 import ep
    assert [ep.shard_range(320, 2, r) for r in range(2)] == [(0, 160), (160, 320)]  # the pages' split
    assert [ep.shard_range(10, 3, r) for r in range(3)] == [(0, 4), (4, 7), (7, 10)]
    with pytest.raises(ValueError):
        ep.shard_range(8, 2, 2)
