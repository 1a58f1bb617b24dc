"""The seeded input generators are deterministic and have the stated shapes."""
import torch

import synthetic_inputs as si


def test_shapes_dtypes_and_determinism():
    cfg = si.CONFIGS["tiny"]
    x1, x2 = si.make_x(cfg), si.make_x(cfg)
    assert x1.dtype == torch.bfloat16 and x1.shape == (cfg.T, cfg.H) and torch.equal(x1, x2)
    lg = si.make_logits(cfg)
    assert lg.dtype == torch.float32 and lg.shape == (cfg.T, cfg.E)
    g = si.make_expert_weight(cfg, 3, "gate")
    d = si.make_expert_weight(cfg, cfg.E, "down")
    assert g.shape == (cfg.I, cfg.H) and d.shape == (cfg.H, cfg.I_s)
    assert torch.equal(g, si.make_expert_weight(cfg, 3, "gate"))
    assert not torch.equal(g, si.make_expert_weight(cfg, 4, "gate"))
    assert torch.equal(si.make_x(cfg, rows=slice(2, 5)), x1[2:5])


def test_zipf_bias_skews_routing():
    cfg = si.LayerConfig("z", T=256, H=16, I=16, I_s=16, E=320, k=8, logits="zipf")
    top = torch.topk(si.make_logits(cfg), 8, dim=1).indices
    counts = torch.bincount(top.reshape(-1), minlength=320)
    assert counts[:20].sum() > 0.8 * counts.sum()
    assert (counts == 0).sum() > 100
