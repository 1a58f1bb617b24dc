"""Builders shared by the GPU parity tests: one seeded layer, prepared once on
the device through the C ABI, and the oracle's view of the same weights."""
import functools

import numpy as np
import torch

import synthetic_inputs as si
from oracle import moe as omoe
from oracle import nvfp4 as onv


@functools.lru_cache(maxsize=3)
def device_layer(name, T=None):
    """(cfg, Nvfp4MoeLayer) with every expert of workload ``name`` (a CONFIGS
    key or a LayerConfig) prepared on the device."""
    import __graft_entry__
    __graft_entry__.build()
    from nvfp4_mixture_experts_moe_gb300 import Nvfp4MoeLayer, MOE_MXFP4, MOE_W4A16, MOE_W4A4
    cfg = si.CONFIGS[name] if isinstance(name, str) else name
    if T is not None:
        cfg = cfg.with_tokens(T)
    mode = {"w4a4": MOE_W4A4, "mxfp4": MOE_MXFP4}.get(cfg.mode, MOE_W4A16)
    layer = Nvfp4MoeLayer(cfg.T, cfg.H, cfg.I, cfg.E, cfg.k, mode=mode, I_shared=cfg.I_s, device="cuda")
    chunk = 32
    for e0 in range(0, cfg.E + 1, chunk):
        W = si.make_layer_weights(cfg, experts=list(range(e0, min(cfg.E + 1, e0 + chunk))), threads=16)
        for e, (g, u, d) in W.items():
            layer.set_expert(e, g, u, d)
    torch.cuda.synchronize()
    return cfg, layer


class OracleWeights:
    """Lazily quantised (by the oracle) experts of a workload, cached: NVFP4,
    or MXFP4 for an "mxfp4" workload."""

    def __init__(self, cfg):
        self.cfg = cfg
        self.cache = {}
        self.kind = omoe.QuantWeightMX if cfg.mode == "mxfp4" else omoe.QuantWeight

    def __call__(self, e):
        if e not in self.cache:
            mats = [si.make_expert_weight(self.cfg, e, m) for m in ("gate", "up", "down")]
            self.cache[e] = tuple(self.kind.from_dense(m.float().numpy()) for m in mats)
        return self.cache[e]

    def all(self):
        return [self(e) for e in range(self.cfg.E)], self(self.cfg.E)

    def prefetch(self, experts, threads=16):
        from concurrent.futures import ThreadPoolExecutor
        todo = [e for e in set(experts) if e not in self.cache]

        def one(e):
            mats = [si.make_expert_weight(self.cfg, e, m) for m in ("gate", "up", "down")]
            return e, tuple(self.kind.from_dense(m.float().numpy()) for m in mats)

        with ThreadPoolExecutor(threads) as ex:
            for e, w in ex.map(one, todo):
                self.cache[e] = w
