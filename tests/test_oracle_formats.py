"""Pins of the oracle's NVFP4 formats and quantiser to facts outside itself.

Each test names what fixes the expected value: the pages (golden files), a
library routine (torch's float8_e4m3fn and bf16 conversions), numpy's
half-to-even rounding, or a closed-form error bound.
"""
import os

import numpy as np
import pytest
import torch

from oracle import nvfp4, moe

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _read_golden(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append(line.split())
    return rows


def test_e2m1_table_matches_page_magnitudes():
    mags = [float(v) for v in _read_golden("e2m1_magnitudes.txt")[0]]
    table = nvfp4.e2m1_decode(np.arange(16))
    assert sorted(set(np.abs(table).tolist())) == sorted(mags)
    assert np.max(np.abs(table)) == 6.0
    # codes 0..7 are the magnitudes in increasing order; bit 3 is the sign
    assert table[:8].tolist() == mags
    assert (table[8:] == -table[:8]).all() and np.signbit(table[8])


def test_e4m3_decode_matches_torch_all_codes():
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).float().numpy().astype(np.float64)
    got = nvfp4.e4m3_decode(codes)
    nan = np.isnan(ref)
    assert (np.isnan(got) == nan).all()
    assert nan.sum() == 2 and nan[0x7F] and nan[0xFF]
    assert (got[~nan] == ref[~nan]).all()
    assert np.nanmax(got) == 448.0


def test_e4m3_encode_matches_torch_rounding_dense_grid():
    # every fp32 between consecutive E4M3 values is hit at quarter steps plus
    # the exact midpoints; torch rounds to nearest even below the 464 midpoint
    vals = nvfp4.e4m3_decode(np.arange(0x7F))
    mids = (vals[:-1] + vals[1:]) / 2
    grid = np.concatenate([vals, mids, np.linspace(0, 463.99, 200001)]).astype(np.float32)
    grid = grid[grid < 464]
    ref = torch.from_numpy(grid).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = nvfp4.e4m3_encode(grid)
    assert (got == ref).all()
    # saturation: everything above 448 clamps to 448 (code 0x7E)
    big = np.array([448.0, 464.0, 500.0, 1e30, np.finfo(np.float32).max], dtype=np.float32)
    assert (nvfp4.e4m3_encode(big) == 0x7E).all()


def _e2m1_reference(y):
    """Binade-wise numpy round-half-even: step 0.5 below 2, 1 in [2,4), 2 above."""
    a = np.abs(y.astype(np.float64))
    step = np.where(a < 2, 0.5, np.where(a < 4, 1.0, 2.0))
    r = np.round(a / step) * step
    r = np.minimum(r, 6.0)
    return r


def test_e2m1_encode_matches_binadewise_rounding():
    y = np.linspace(-8, 8, 160001).astype(np.float32)
    y = np.concatenate([y, np.arange(-32, 33, dtype=np.float32) / 4])  # all quarter points
    codes = nvfp4.e2m1_encode(y)
    got = np.abs(nvfp4.e2m1_decode(codes))
    assert (got == _e2m1_reference(y)).all()
    # sign kept, including for values that round to zero
    assert ((codes & 8) != 0).tolist() == np.signbit(y).tolist()


def test_e2m1_tie_table():
    for a, b in _read_golden("e2m1_ties.txt"):
        for s in (1.0, -1.0):
            c = nvfp4.e2m1_encode(np.array([s * float(a)], dtype=np.float32))
            assert nvfp4.e2m1_decode(c)[0] == s * float(b), (a, b, s)


def test_global_scale_worked_example():
    g = dict((k, float(v)) for k, v in _read_golden("global_scale_worked_example.txt"))
    gs = nvfp4.global_scale(np.float32(g["amax"]))
    assert gs == np.float32(g["quant_scale"])
    # the dequant convention: amax/(448*6) equals 1/gs here, and is the value
    # the page prints (an fp32 number)
    dq = np.float32(np.float32(g["amax"]) / nvfp4.QUANT_RANGE)
    assert float(dq) == g["dequant_scale"]
    assert float(np.float32(1) / gs) == g["dequant_scale"]
    # a block whose amax is the tensor amax decodes back to amax exactly
    x = np.zeros((1, 16), dtype=np.float32)
    x[0, 3] = g["amax"]
    q, sf, gsq = nvfp4.quantize(x)
    assert gsq == np.float32(g["quant_scale"])
    assert nvfp4.dequantize(q, sf, gsq)[0, 3] == g["amax"]


def _bound(x):
    """Closed-form error bound of one NVFP4 round trip, per element.

    sf is within a relative 2**-4 of amax_b*gs/6 (E4M3 has 3 mantissa bits),
    so |x*gs/sf| <= 6*(1+2**-4); the e2m1 step is at most 2 (between 4 and 6)
    and saturation costs at most 0.375, so |x - deq| <= (sf/gs) <=
    (amax_b/6) * (1 + 2**-4), plus the E4M3 subnormal spacing 2**-9/gs when
    the block scale is tiny.
    """
    rows, K = x.shape
    amax_b = np.max(np.abs(x.reshape(rows, K // 16, 16)), axis=2)
    return np.repeat(amax_b / 6 * (1 + 2 ** -4), 16, axis=1)


def test_quantize_roundtrip_error_bound_and_quality():
    rng = np.random.default_rng(0)
    w = (rng.standard_normal((64, 512)) * 0.02).astype(np.float32)
    q, sf, gs = nvfp4.quantize(w)
    d = nvfp4.dequantize(q, sf, gs)
    tiny = 2.0 ** -9 / float(gs)
    assert (np.abs(d - w) <= _bound(w) + tiny).all()
    cos = float((d * w).sum() / np.linalg.norm(d) / np.linalg.norm(w))
    rel = float(np.linalg.norm(d - w) / np.linalg.norm(w))
    # soft, order-of-magnitude check: the GLM-5.3 conversion reports a mean
    # round-trip cosine of 0.998 on real weights; FP4 tensors show ~9% error
    assert cos > 0.99
    assert 0.02 < rel < 0.2


def test_quantize_wrong_inversion_fails_loudly():
    # Multiplying by the quant-convention scale instead of dividing by it is the
    # silent failure the GLM-5.3 thread warns about; the error bar must catch it.
    rng = np.random.default_rng(1)
    w = (rng.standard_normal((8, 256)) * 0.02).astype(np.float32)
    q, sf, gs = nvfp4.quantize(w)
    good = nvfp4.dequantize(q, sf, gs)
    wrong = nvfp4.e2m1_decode(q) * np.repeat(nvfp4.e4m3_decode(sf), 16, axis=1) * float(gs)
    err_good = np.abs(good - w).max()
    err_wrong = np.abs(wrong - w).max()
    assert err_good <= _bound(w).max()
    assert err_wrong > 1e6 * err_good


def test_g16_blocks_are_independent():
    rng = np.random.default_rng(2)
    x = rng.standard_normal((2, 64)).astype(np.float32)
    x[1, 63] = 50.0                      # pins the tensor amax, so gs is fixed
    q0, sf0, gs0 = nvfp4.quantize(x)
    y = x.copy()
    y[0, 16:32] *= 3.0                   # change block 1 of row 0 only
    q1, sf1, gs1 = nvfp4.quantize(y)
    assert gs0 == gs1
    keep = np.ones(4, dtype=bool)
    keep[1] = False
    assert (sf0[0, keep] == sf1[0, keep]).all() and (sf0[1] == sf1[1]).all()
    qb0 = q0.reshape(2, 4, 16)
    qb1 = q1.reshape(2, 4, 16)
    assert (qb0[0, keep] == qb1[0, keep]).all() and (qb0[1] == qb1[1]).all()
    assert (sf0[0, 1] != sf1[0, 1]) or (qb0[0, 1] != qb1[0, 1]).any()
    # one element at 6*s with tiny neighbours decodes with block scale s
    z = np.full((1, 16), 1e-3, dtype=np.float32)
    z[0, 0] = 6.0
    qz, sfz, gsz = nvfp4.quantize(z)
    assert nvfp4.e2m1_decode(qz[0, 0]) == 6.0
    assert nvfp4.dequantize(qz, sfz, gsz)[0, 0] == 6.0


def test_zero_tensor_and_zero_blocks():
    q, sf, gs = nvfp4.quantize(np.zeros((2, 32), dtype=np.float32))
    assert gs == 1.0 and (q == 0).all() and (sf == 0).all()
    x = np.zeros((1, 32), dtype=np.float32)
    x[0, 20] = -1.0
    q, sf, gs = nvfp4.quantize(x)
    assert sf[0, 0] == 0 and (q[0, :16] == 0).all()
    assert nvfp4.dequantize(q, sf, gs)[0, 20] == -1.0


def test_pack_nibble_order():
    codes = np.array([[1, 2, 3, 4]], dtype=np.uint8)
    packed = nvfp4.pack(codes)
    assert packed.tolist() == [[0x21, 0x43]]
    assert (nvfp4.unpack(packed) == codes).all()


def test_bf16_round_matches_torch():
    rng = np.random.default_rng(3)
    x = np.concatenate([rng.standard_normal(100000) * 10.0 ** rng.integers(-30, 30, 100000),
                        np.array([1 + 2 ** -8, 1 + 3 * 2 ** -8, -(1 + 2 ** -8), 0.0, -0.0])])
    x32 = x.astype(np.float32)
    ref = torch.from_numpy(x32).to(torch.bfloat16).float().numpy()
    got = moe.bf16_round(x32)
    assert (got.view(np.uint32) == ref.view(np.uint32)).all()
