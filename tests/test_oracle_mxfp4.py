"""Pins of the oracle's MXFP4 format (e2m1 elements, E8M0 scales per 32) to
torch's float8_e8m0fnu decoding and to closed forms of the format."""
import numpy as np
import pytest
import torch

from oracle import mxfp4, nvfp4


def test_e8m0_decode_matches_torch_all_codes():
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e8m0fnu).to(torch.float64).numpy()
    got = mxfp4.e8m0_decode(codes)
    assert np.isnan(got[255]) and np.isnan(ref[255])
    assert (got[:255] == ref[:255]).all()
    assert got[0] == 2.0 ** -127 and got[127] == 1.0 and got[254] == 2.0 ** 127


def _x(rows, K, seed, scale=1.0):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(rows, K, generator=g) * scale).to(torch.bfloat16).float().numpy()


def test_block_scale_puts_block_max_in_4_to_8():
    x = _x(16, 256, 1) * np.exp2(np.random.default_rng(0).integers(-20, 20, (16, 1))).astype(np.float32)
    codes, sc = mxfp4.quantize(x)
    amax = np.abs(x.reshape(16, 8, 32)).max(axis=2)
    ratio = amax / mxfp4.e8m0_decode(sc)
    assert ((ratio >= 4) & (ratio < 8)).all()


def test_power_of_two_factor_moves_scale_codes_only():
    x = _x(8, 128, 2)
    c0, s0 = mxfp4.quantize(x)
    for j in (-9, -1, 3, 17):
        c1, s1 = mxfp4.quantize((x * np.float32(2.0 ** j)).astype(np.float32))
        assert (c1 == c0).all() and (s1.astype(int) == s0.astype(int) + j).all()


def test_blocks_of_e2m1_values_round_trip_exactly():
    rng = np.random.default_rng(3)
    codes = rng.integers(0, 16, (4, 64)).astype(np.uint8)
    codes[:, 0] = 6   # magnitude 4.0 in every block: block max in [4, 8)
    codes[:, 32] = 7  # 6.0
    vals = nvfp4.e2m1_decode(codes) * np.exp2(rng.integers(-10, 10, (4, 1)))
    q, s = mxfp4.quantize(vals.astype(np.float32))
    assert (mxfp4.dequantize(q, s) == vals).all()


def test_values_above_six_units_saturate():
    x = np.zeros((1, 32), dtype=np.float32)
    x[0, 0] = 7.5      # scale 2^(2-2) = 1: 7.5 > 6 saturates to the code of 6
    x[0, 1] = -6.9
    x[0, 2] = 5.0      # tie between 4 and 6 -> even code (4)
    x[0, 3] = 0.25     # tie between 0 and 0.5 -> 0
    q, s = mxfp4.quantize(x)
    assert s[0, 0] == 127
    assert q[0, 0] == 7 and q[0, 1] == 15 and q[0, 2] == 6 and q[0, 3] == 0


def test_zero_block_and_block_independence():
    x = _x(2, 96, 4)
    x[1, 32:64] = 0
    q, s = mxfp4.quantize(x)
    assert s[1, 1] == 0 and (q[1, 32:64] == 0).all()
    y = x.copy()
    y[0, 40] *= 64  # only block 1 of row 0 changes
    q2, s2 = mxfp4.quantize(y)
    assert (q2[0, :32] == q[0, :32]).all() and (q2[0, 64:] == q[0, 64:]).all()
    assert s2[0, 0] == s[0, 0] and s2[0, 2] == s[0, 2] and s2[0, 1] != s[0, 1]


def test_round_trip_error_bound():
    x = _x(32, 512, 5)
    q, s = mxfp4.quantize(x)
    d = mxfp4.dequantize(q, s)
    scale = np.repeat(mxfp4.e8m0_decode(s), 32, axis=1)
    err = np.abs(d - x)
    # below 6 units the e2m1 spacing is at most 2, so the error is at most 1
    # unit; values in (6, 8) units saturate to 6 (error below 2 units)
    inside = np.abs(x) / scale <= 6
    assert (err[inside] <= scale[inside]).all()
    assert (err[~inside] < 2 * scale[~inside]).all()


def test_rejects_ragged_k():
    with pytest.raises(ValueError):
        mxfp4.quantize(np.zeros((1, 48), dtype=np.float32))
