"""Router GEMM, static W4A4 activation scales and checkpoint import on the GPU,
through the C ABI, against the CPU oracle."""
import numpy as np
import pytest
import torch

import synthetic_inputs as si
from oracle import moe as omoe
from oracle import nvfp4 as onv
from tests.gpu_layers import OracleWeights, device_layer
from tests.tolerance import check_outputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__
    __graft_entry__.build()


def _B():
    from nvfp4_mixture_experts_moe_gb300 import binding
    return binding


def _router_inputs(T, H, E, seed):
    cfg = si.LayerConfig("router", T=T, H=H, I=64, I_s=64, E=E, k=1, seed=seed)
    return si.make_x(cfg), si.make_router_weight(cfg)


def _gpu_logits(x, w):
    T, H = x.shape
    E = w.shape[0]
    out = torch.full((T, E), float("nan"), dtype=torch.float32, device="cuda")
    _B().moe_router_gemm(x.cuda(), w.cuda(), T, H, E, out)
    torch.cuda.synchronize()
    return out


# (T, H, E): few-token path (T <= 16) and tiled path; ragged T, E and a K tail
# (H % 64 != 0); the decode and prefill router shapes and the W4A4 layer's H, E
ROUTER_CASES = [(1, 256, 8), (8, 4096, 320), (16, 264, 33), (17, 264, 33), (130, 520, 65), (300, 512, 320),
                (4096, 4096, 320), (300, 7168, 256)]


@pytest.mark.parametrize("T,H,E", ROUTER_CASES)
def test_router_gemm_matches_oracle(T, H, E):
    x, w = _router_inputs(T, H, E, seed=T + H + E)
    got = _gpu_logits(x, w).cpu().numpy().astype(np.float64)
    xf, wf = x.float().numpy(), w.float().numpy()
    ref = omoe.router_logits(xf, wf)
    # bf16 products are exact in fp32; an fp32 sum of H terms in any order is
    # within H * 2^-24 * sum |x_i w_i| of the exact sum
    bound = H * 2.0 ** -24 * omoe.router_logits(np.abs(xf), np.abs(wf)) + 1e-30
    err = np.abs(got - ref)
    assert np.isfinite(got).all()
    assert (err <= bound).all(), float((err / bound).max())
    # typical size: rounding errors of H fp32 additions add like a random
    # walk, about sqrt(H) * 2^-24 relative; allow 4x that
    assert np.linalg.norm(got - ref) <= 4 * np.sqrt(H) * 2.0 ** -24 * np.linalg.norm(ref)


def test_router_gemm_deterministic():
    x, w = _router_inputs(300, 512, 320, seed=1)
    a = _gpu_logits(x, w)
    b = _gpu_logits(x, w)
    assert torch.equal(a, b)


@pytest.mark.parametrize("name,T", [("tiny", None), ("tiny", 100), ("decode", None)])
def test_forward_with_router_equals_forward_on_router_logits(name, T):
    cfg, layer = device_layer(name, T)
    x = si.make_x(cfg).cuda()
    w_router = si.make_router_weight(cfg)
    logits = _gpu_logits(x, w_router)
    ids_a = torch.empty(cfg.T, cfg.k, dtype=torch.int32, device="cuda")
    ids_b = torch.empty_like(ids_a)
    out_a = layer.forward(x, logits, topk_ids=ids_a)
    layer.set_router(w_router)
    try:
        ws = layer.workspace()
        out_b = layer.forward(x, None, topk_ids=ids_b, ws=ws)
        torch.cuda.synchronize()
        assert _B().moe_get_device_status(ws) == 0
    finally:
        layer.set_router(None)
    assert torch.equal(ids_a, ids_b) and torch.equal(out_a, out_b)
    # the routing decision, taken on the GPU's fp32 logits, is the oracle's
    # decision on those same logits
    ids_ref, _ = omoe.route(logits.cpu().numpy(), cfg.k)
    assert (ids_b.cpu().numpy() == ids_ref).all()


def test_forward_with_router_tiny_full_oracle_check():
    cfg, layer = device_layer("tiny")
    x = si.make_x(cfg)
    w_router = si.make_router_weight(cfg)
    logits = _gpu_logits(x, w_router)
    layer.set_router(w_router)
    try:
        out = layer.forward(x.cuda(), None)
        torch.cuda.synchronize()
    finally:
        layer.set_router(None)
    experts, shared = OracleWeights(cfg).all()
    ref = omoe.layer(x.float().numpy(), logits.cpu().numpy(), experts, shared, cfg.k)
    check_outputs(out.float().cpu().numpy(), ref, what="tiny with router")
    # and the logits themselves are the oracle's router product
    ref_logits = omoe.router_logits(x.float().numpy(), w_router.float().numpy())
    assert np.abs(logits.cpu().numpy() - ref_logits).max() < 1e-4


# --- static W4A4 activation scales ------------------------------------------

@pytest.mark.parametrize("factor", [1.0, 0.25, 4.0, 64.0])
def test_quantize_static_bit_exact(factor):
    g = torch.Generator().manual_seed(11)
    rows, K = 37, 272
    x = (torch.randn(rows, K, generator=g) * torch.exp(torch.randn(rows, 1, generator=g))).to(torch.bfloat16)
    xf = x.float().numpy()
    _, _, gs_dyn = onv.quantize(xf)
    gs = np.float32(gs_dyn * np.float32(factor))
    q = torch.empty(rows, K // 2, dtype=torch.uint8, device="cuda")
    sf = torch.empty(rows, K // 16, dtype=torch.uint8, device="cuda")
    _B().moe_nvfp4_quantize_static(x.cuda(), rows, K, float(gs), q, sf)
    torch.cuda.synchronize()
    codes, sf_ref, g2 = onv.quantize(xf, gs=gs)
    assert g2 == gs
    assert (sf.cpu().numpy() == sf_ref).all()
    assert (q.cpu().numpy() == onv.pack(codes)).all()
    if factor > 1:
        assert (sf_ref == 0x7E).any()  # saturated blocks are part of the check


W4A4_SMALL = si.LayerConfig("w4a4_static", T=64, H=512, I=256, I_s=256, E=8, k=2, mode="w4a4", outliers=True)


def test_w4a4_forward_static_scales_matches_oracle():
    cfg, layer = device_layer(W4A4_SMALL)
    x = si.make_x(cfg)
    logits = si.make_logits(cfg)
    experts, shared = OracleWeights(cfg).all()
    # calibration: the dynamic scales of another seeded batch of the same workload
    cal = si.LayerConfig(cfg.name, cfg.T, cfg.H, cfg.I, cfg.I_s, cfg.E, cfg.k, cfg.mode, cfg.logits,
                         cfg.outliers, seed=cfg.seed + 1)
    _, cal_parts = omoe.layer(si.make_x(cal).float().numpy(), si.make_logits(cal).numpy(), experts, shared,
                              cfg.k, mode="w4a4", return_parts=True)
    x_gs, h_gs = cal_parts["xgs"], cal_parts["hgs"]
    layer.set_static_scales(float(x_gs), float(h_gs))
    try:
        ws = layer.workspace()
        ids = torch.empty(cfg.T, cfg.k, dtype=torch.int32, device="cuda")
        out = layer.forward(x.cuda(), logits.cuda(), topk_ids=ids, ws=ws)
        out2 = layer.forward(x.cuda(), logits.cuda(), ws=ws)
        torch.cuda.synchronize()
        assert _B().moe_get_device_status(ws) == 0
    finally:
        layer.set_static_scales(0.0, 0.0)
    assert torch.equal(out, out2)
    ref, parts = omoe.layer(x.float().numpy(), logits.numpy(), experts, shared, cfg.k, mode="w4a4",
                            return_parts=True, x_gs=x_gs, h_gs=h_gs)
    assert parts["xgs"] == x_gs and parts["hgs"] == h_gs
    assert (ids.cpu().numpy() == parts["ids"]).all()
    check_outputs(out.float().cpu().numpy(), ref, what="w4a4 static scales")


# --- checkpoint import -------------------------------------------------------

FINITE = np.arange(0x7F, dtype=np.uint8)


@pytest.mark.parametrize("ratio", [0.3, 0.77, 1.0 / 3.0, 1.0, 1.9, 3.1, 1000.0, 2.0 ** -3])
def test_fold_scales_bit_exact(ratio):
    codes = np.tile(FINITE, 5)
    sf_in = torch.from_numpy(codes).cuda()
    sf_out = torch.empty_like(sf_in)
    _B().moe_nvfp4_fold_scales(sf_in, codes.size, float(np.float32(ratio)), sf_out)
    assert (sf_out.cpu().numpy() == onv.fold_block_scales(codes, np.float32(ratio))).all()
    # in place
    _B().moe_nvfp4_fold_scales(sf_in, codes.size, float(np.float32(ratio)), sf_in)
    assert torch.equal(sf_in, sf_out)


def test_fold_scales_refuses_bad_codes():
    codes = np.array([0x10, 0x7F, 0x38, 0x90, 0x7E], dtype=np.uint8)
    sf_in = torch.from_numpy(codes).cuda()
    sf_out = torch.zeros_like(sf_in)
    B = _B()
    with pytest.raises(B.MoeError) as e:
        B.moe_nvfp4_fold_scales(sf_in, codes.size, 2.0, sf_out)
    assert e.value.status == B.MOE_ERR_INVALID_ARG
    got = sf_out.cpu().numpy()
    good = np.array([0, 2, 4])
    assert (got[good] == onv.fold_block_scales(codes[good], 2.0)).all()
    assert got[1] == 0x7F and got[3] == 0x90


IMPORT_CFG = si.LayerConfig("import", T=48, H=256, I=128, I_s=128, E=4, k=2)


@pytest.mark.parametrize("fmt_name", ["dequant", "quant"])
def test_import_expert_checkpoint_matches_oracle(fmt_name):
    """Checkpoint matrices quantised by the oracle, their global scales stored
    in ModelOpt (dequant) or compressed-tensors (quant) form, imported through
    moe_import_global_scale and prepared; the up matrix is moved onto the gate's
    global scale with moe_nvfp4_fold_scales (one scale for the pair)."""
    from nvfp4_mixture_experts_moe_gb300 import Nvfp4MoeLayer, MOE_W4A16
    B = _B()
    cfg = IMPORT_CFG
    fmt = B.MOE_SCALE_DEQUANT if fmt_name == "dequant" else B.MOE_SCALE_QUANT
    layer = Nvfp4MoeLayer(cfg.T, cfg.H, cfg.I, cfg.E, cfg.k, mode=MOE_W4A16, I_shared=cfg.I_s, device="cuda")
    oracle_experts = []
    for e in range(cfg.E + 1):
        mats = [onv.quantize(si.make_expert_weight(cfg, e, m).float().numpy()) for m in ("gate", "up", "down")]
        (cg, sg, gg), (cu, su, gu), (cd, sd, gd) = mats
        # fold up onto the gate's scale, on the device
        ratio = np.float32(gg / gu)
        su_dev = torch.from_numpy(su.copy()).cuda()
        B.moe_nvfp4_fold_scales(su_dev, su.size, float(ratio), su_dev)
        su_f = su_dev.cpu().numpy()
        assert (su_f == onv.fold_block_scales(su, ratio)).all()

        def stored(gs):
            return float(np.float32(1.0) / gs) if fmt_name == "dequant" else float(gs)

        got = layer.import_expert(
            e,
            (torch.from_numpy(onv.pack(cg)), torch.from_numpy(sg), stored(gg)),
            (torch.from_numpy(onv.pack(cu)), torch.from_numpy(su_f), stored(gg)),
            (torch.from_numpy(onv.pack(cd)), torch.from_numpy(sd), stored(gd)),
            fmt)
        imp = [onv.import_global_scale(stored(g), fmt_name) for g in (gg, gg, gd)]
        assert [np.float32(v) for v in got] == imp
        oracle_experts.append((omoe.QuantWeight(cg, sg, imp[0]), omoe.QuantWeight(cu, su_f, imp[1]),
                               omoe.QuantWeight(cd, sd, imp[2])))
    x = si.make_x(cfg)
    logits = si.make_logits(cfg)
    out = layer.forward(x.cuda(), logits.cuda())
    torch.cuda.synchronize()
    ref = omoe.layer(x.float().numpy(), logits.numpy(), oracle_experts[:cfg.E], oracle_experts[cfg.E], cfg.k)
    check_outputs(out.float().cpu().numpy(), ref, what=f"imported ({fmt_name})")
