"""Pins of the oracle's router GEMM, static W4A4 scales and checkpoint scale
import to facts outside itself: the pages' worked value (golden file), exact
rational arithmetic, closed forms of the E4M3 format, torch's float8_e4m3fn
rounding, and reductions to the already pinned dynamic quantiser.
"""
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import synthetic_inputs as si
from oracle import moe, nvfp4

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
F32 = np.float32


def _golden_pairs(name):
    out = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                key, val = line.split()
                out[key] = float(val)
    return out


# --- router GEMM ------------------------------------------------------------

def test_router_logits_exact_rational_tiny():
    g = torch.Generator().manual_seed(5)
    x = torch.randn(3, 16, generator=g).to(torch.bfloat16).float().numpy()
    w = torch.randn(4, 16, generator=g).to(torch.bfloat16).float().numpy()
    got = moe.router_logits(x, w)
    for t in range(3):
        for e in range(4):
            exact = sum(Fraction(float(a)) * Fraction(float(b)) for a, b in zip(x[t], w[e]))
            assert abs(got[t, e] - float(exact)) <= 1e-14 * max(1.0, abs(float(exact)))


def test_router_logits_one_hot_rows_pick_columns():
    T, H, E = 5, 32, 6
    x = torch.randn(T, H, generator=torch.Generator().manual_seed(1)).to(torch.bfloat16).float().numpy()
    cols = [3, 0, 31, 7, 7, 12]
    scale = [1.0, -2.0, 0.5, 0.25, 3.0, -1.5]
    w = np.zeros((E, H), dtype=np.float32)
    for e in range(E):
        w[e, cols[e]] = scale[e]
    got = moe.router_logits(x, w)
    for e in range(E):
        assert (got[:, e] == scale[e] * x[:, cols[e]].astype(np.float64)).all()


def test_router_weight_recipe_gives_unit_logits():
    cfg = si.LayerConfig("r", T=256, H=1024, I=64, I_s=64, E=64, k=2)
    x = si.make_x(cfg).float().numpy()
    w = si.make_router_weight(cfg).float().numpy()
    logits = moe.router_logits(x, w)
    assert abs(logits.std() - 1.0) < 0.05 and abs(logits.mean()) < 0.05


# --- static W4A4 scales -----------------------------------------------------

def _x(rows, K, seed=0, scale=1.0):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(rows, K, generator=g) * scale).to(torch.bfloat16).float().numpy()


def test_static_scale_equal_to_dynamic_reproduces_dynamic():
    x = _x(7, 64, seed=2)
    q0, sf0, gs0 = nvfp4.quantize(x)
    q1, sf1, gs1 = nvfp4.quantize(x, gs=gs0)
    assert gs1 == gs0 and (q1 == q0).all() and (sf1 == sf0).all()


def test_static_power_of_two_scale_shifts_block_exponents():
    # scaling gs by 2^j multiplies every block scale s by 2^j exactly; while s
    # stays in E4M3's normal range, its code moves by 8*j (the exponent field)
    # and r = gs / sf is unchanged, so the e2m1 codes are unchanged
    x = _x(4, 128, seed=3)
    _, _, gs_dyn = nvfp4.quantize(x)
    gs0 = gs_dyn * F32(2.0 ** -4)          # block scales well inside the normal range
    q0, sf0, _ = nvfp4.quantize(x, gs=gs0)
    for j in (-3, -1, 1, 2):
        q1, sf1, _ = nvfp4.quantize(x, gs=gs0 * F32(2.0 ** j))
        vals = nvfp4.e4m3_decode(sf0)
        normal = (vals >= 2.0 ** -6) & (vals * 2.0 ** j >= 2.0 ** -6) & (vals * 2.0 ** j <= 448)
        assert normal.sum() > 0.9 * normal.size
        assert (sf1[normal].astype(int) == sf0[normal].astype(int) + 8 * j).all()
        rows_ok = normal.all(axis=1)
        assert (q1[rows_ok] == q0[rows_ok]).all()


def test_static_scale_saturates_out_of_range_blocks():
    # a calibrated scale too large for a block: s = (amax_b / 6) * gs > 448,
    # so the block scale clamps to 448 (code 0x7E) and r = gs / 448; elements
    # with |x| * r >= 6 clamp to the e2m1 maximum (codes 7 / 15)
    x = np.zeros((1, 32), dtype=np.float32)
    x[0, :16] = np.linspace(-4.0, 4.0, 16).astype(np.float32)
    x[0, 16:] = 0.01
    gs = F32(2000.0)                     # (4/6)*2000 = 1333 > 448
    q, sf, g = nvfp4.quantize(x, gs=gs)
    assert g == gs and sf[0, 0] == 0x7E
    r = np.float64(gs) / 448.0
    mags = np.abs(x[0, :16]).astype(np.float64) * r
    codes = q[0, :16]
    assert ((codes[mags >= 6.0] & 7) == 7).all()
    assert ((codes[x[0, :16] < 0] & 8) == 8).all()
    # the second block is in range: the static scale acts like a dynamic one
    s2 = np.float64(F32(F32(F32(0.01) / F32(6)) * gs))
    assert nvfp4.e4m3_decode(sf[0, 1]) == nvfp4.e4m3_decode(nvfp4.e4m3_encode(F32(s2)))


def test_static_scale_rejects_bad_values():
    x = _x(1, 16)
    for bad in (0.0, -1.0, float("inf"), float("nan")):
        with pytest.raises(ValueError):
            nvfp4.quantize(x, gs=bad)


def test_layer_static_scales_equal_dynamic_reproduce_dynamic():
    cfg = si.LayerConfig("s", T=6, H=64, I=32, I_s=32, E=4, k=2, mode="w4a4", outliers=True)
    x = si.make_x(cfg).float().numpy()
    logits = si.make_logits(cfg).numpy()
    wts = si.make_layer_weights(cfg, threads=1)
    experts = [tuple(moe.QuantWeight.from_dense(m.float().numpy()) for m in wts[e]) for e in range(cfg.E)]
    shared = tuple(moe.QuantWeight.from_dense(m.float().numpy()) for m in wts[cfg.E])
    out0, p0 = moe.layer(x, logits, experts, shared, cfg.k, mode="w4a4", return_parts=True)
    out1, p1 = moe.layer(x, logits, experts, shared, cfg.k, mode="w4a4", return_parts=True,
                         x_gs=p0["xgs"], h_gs=p0["hgs"])
    assert (out1 == out0).all()
    assert (p1["hq"] == p0["hq"]).all() and (p1["xsf"] == p0["xsf"]).all()
    # a different static scale changes the result, but only by quantisation noise
    out2 = moe.layer(x, logits, experts, shared, cfg.k, mode="w4a4",
                     x_gs=p0["xgs"] * F32(0.75), h_gs=p0["hgs"] * F32(0.75))
    assert not (out2 == out0).all()
    rel = np.linalg.norm(out2 - out0) / np.linalg.norm(out0)
    assert rel < 0.2


# --- checkpoint global-scale import -----------------------------------------

def test_import_worked_reciprocal_pair():
    gold = _golden_pairs("global_scale_worked_example.txt")
    gs = nvfp4.import_global_scale(gold["dequant_scale"], "dequant")
    assert gs == F32(gold["quant_scale"])
    assert nvfp4.import_global_scale(gold["quant_scale"], "quant") == F32(gold["quant_scale"])
    # the dequant value printed is the fp32 reciprocal of the quant value
    assert F32(1.0) / F32(gold["quant_scale"]) == F32(gold["dequant_scale"])
    # the wrong inversion is off by a factor of about 2e9
    wrong = F32(gold["dequant_scale"])
    assert gs / wrong > 1e8


def test_import_powers_of_two_and_round_trip():
    for j in range(-20, 21):
        assert nvfp4.import_global_scale(2.0 ** j, "dequant") == F32(2.0 ** -j)
    vals = np.random.default_rng(0).uniform(1e-6, 1e4, 2000).astype(np.float32)
    for v in vals:
        back = F32(1.0) / nvfp4.import_global_scale(v, "dequant")
        assert abs(int(back.view(np.int32)) - int(v.view(np.int32))) <= 1


def test_import_refuses_zero_and_non_finite():
    for fmt in ("quant", "dequant"):
        for bad in (0.0, -2.0, float("inf"), float("nan")):
            with pytest.raises(ValueError):
                nvfp4.import_global_scale(bad, fmt)
    with pytest.raises(ValueError):
        nvfp4.import_global_scale(1.0, "modelopt")


# --- folding a global-scale ratio into the block scales ---------------------

FINITE = np.arange(0x7F, dtype=np.uint8)   # 0x00..0x7E: zero, subnormals, normals


def test_fold_ratio_one_is_identity():
    assert (nvfp4.fold_block_scales(FINITE, 1.0) == FINITE).all()


def test_fold_power_of_two_moves_exponent_field():
    vals = nvfp4.e4m3_decode(FINITE)
    for j in (-2, -1, 1, 3):
        got = nvfp4.fold_block_scales(FINITE, 2.0 ** j).astype(int)
        ok = (vals >= 2.0 ** -6) & (vals * 2.0 ** j >= 2.0 ** -6) & (vals * 2.0 ** j <= 448)
        assert (got[ok] == FINITE[ok].astype(int) + 8 * j).all()
        sat = vals * 2.0 ** j > 448
        assert (got[sat] == 0x7E).all()


@pytest.mark.parametrize("ratio", [0.3, 0.77, 1.0 / 3.0, 1.9, 3.1, 1000.0])
def test_fold_matches_torch_e4m3_rounding(ratio):
    r = F32(ratio)
    prod = (nvfp4.e4m3_decode(FINITE).astype(np.float32) * r).astype(np.float32)
    got = nvfp4.fold_block_scales(FINITE, r)
    inr = prod < 448
    ref = torch.from_numpy(prod[inr]).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert (got[inr] == ref).all()
    assert (got[~inr] == 0x7E).all()


def test_fold_refuses_sign_and_nan_codes():
    for bad in (0x7F, 0xFF, 0x80, 0x90):
        with pytest.raises(ValueError):
            nvfp4.fold_block_scales(np.array([bad], dtype=np.uint8), 1.0)
    with pytest.raises(ValueError):
        nvfp4.fold_block_scales(FINITE, 0.0)


def test_fold_keeps_dequantised_values_within_half_an_e4m3_step():
    # moving a quantised matrix to a shared global scale: values change by at
    # most the E4M3 re-rounding of the block scale (relative 2^-4 for normals)
    w = _x(8, 64, seed=9, scale=0.02)
    q, sf, gs = nvfp4.quantize(w)
    gs_new = F32(gs * F32(0.8))
    sf2 = nvfp4.fold_block_scales(sf, gs_new / gs)
    a = nvfp4.dequantize(q, sf, gs)
    b = nvfp4.dequantize(q, sf2, gs_new)
    s_old = nvfp4.e4m3_decode(sf)
    normal = np.repeat(nvfp4.e4m3_decode(sf2) >= 2.0 ** -6, 16, axis=1)
    assert np.all(np.abs(b - a)[normal] <= np.abs(a)[normal] * 2.0 ** -4 + 1e-30)
    assert np.isfinite(s_old).all()
