"""Expert parallelism on one GPU ("Serving Solar Open 2 on DGX Spark",
"Adding Expert Parallelism to b12x"): the experts split into contiguous
shards, each forward computing only the pairs routed to its own experts
(global ids remapped to local ones, other pairs filtered out), the shared
expert on one shard. Each shard's partial output against the oracle's shard,
and the shards' sum against the oracle's whole layer."""
import numpy as np
import pytest
import torch

import synthetic_inputs as si
from oracle import moe as omoe
from tests.gpu_layers import OracleWeights
from tests.tolerance import check_outputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__
    __graft_entry__.build()


def _shard_layers(cfg, bounds):
    from nvfp4_mixture_experts_moe_gb300 import MOE_MXFP4, MOE_W4A16, MOE_W4A4, Nvfp4MoeLayer
    mode = {"w4a4": MOE_W4A4, "mxfp4": MOE_MXFP4}.get(cfg.mode, MOE_W4A16)
    W = si.make_layer_weights(cfg)
    layers = []
    for i in range(len(bounds) - 1):
        lo, hi = bounds[i], bounds[i + 1]
        layer = Nvfp4MoeLayer(cfg.T, cfg.H, cfg.I, cfg.E, cfg.k, mode=mode, I_shared=cfg.I_s, shared=i == 0,
                              device="cuda", expert_offset=lo, local_experts=hi - lo)
        for e in range(lo, hi):
            layer.set_expert(e, *W[e])
        if i == 0:
            layer.set_expert(cfg.E, *W[cfg.E])
        layers.append(layer)
    torch.cuda.synchronize()
    return layers


@pytest.mark.parametrize("cfg,bounds", [
    (si.LayerConfig("ep_dec", T=8, H=512, I=256, I_s=256, E=16, k=4), [0, 8, 16]),
    (si.LayerConfig("ep_pre", T=300, H=512, I=256, I_s=256, E=8, k=2), [0, 3, 8]),
    (si.LayerConfig("ep_big", T=1200, H=256, I=128, I_s=128, E=16, k=8), [0, 5, 11, 16]),
    (si.LayerConfig("ep_mx", T=64, H=512, I=256, I_s=256, E=8, k=2, mode="mxfp4"), [0, 4, 8]),
    (si.LayerConfig("ep_w4a4", T=64, H=512, I=256, I_s=256, E=8, k=2, mode="w4a4"), [0, 2, 8]),
], ids=["decode", "tensor_core", "multi_cta_permute", "mxfp4", "w4a4"])
def test_expert_shards(cfg, bounds):
    from nvfp4_mixture_experts_moe_gb300 import binding
    layers = _shard_layers(cfg, bounds)
    x = si.make_x(cfg)
    logits = si.make_logits(cfg)
    rids, _ = omoe.route(logits.numpy(), cfg.k)
    experts, shared = OracleWeights(cfg).all()
    xs = x.float().numpy()
    partials = []
    for i, layer in enumerate(layers):
        ids = torch.empty(cfg.T, cfg.k, dtype=torch.int32, device="cuda")
        ws = layer.workspace()
        out = layer.forward(x.cuda(), logits.cuda(), topk_ids=ids, ws=ws)
        torch.cuda.synchronize()
        assert binding.moe_get_device_status(ws) == 0   # filtered pairs are not errors
        assert (ids.cpu().numpy() == rids).all()         # global ids
        got = out.float().cpu().numpy()
        ref = omoe.layer(xs, logits.numpy(), experts, shared if i == 0 else None, cfg.k, mode=cfg.mode,
                         experts_range=(bounds[i], bounds[i + 1]))
        check_outputs(got, ref, what=f"{cfg.name} shard {bounds[i]}..{bounds[i + 1]}")
        partials.append(got)
    if cfg.mode != "w4a4":  # dynamic W4A4 scales differ per shard: only the shards are compared there
        full = omoe.layer(xs, logits.numpy(), experts, shared, cfg.k, mode=cfg.mode)
        # every partial carries its own bf16 output rounding (2^-8 |partial|)
        extra = sum(2.0 ** -8 * np.abs(p) for p in partials)
        check_outputs(sum(partials), full, extra=extra, what=f"{cfg.name} shards summed")
