"""NVFP4 number formats and the block quantiser, written out plainly.

Test infrastructure only (see the package docstring for who may import it).

Format, from "vLLM on the NVIDIA DGX Spark: A Complete Technical Guide",
section 6.1 "NVFP4 format" and section 6.4 "NVFP4 vs MXFP4":

* element: e2m1, a 4-bit float (sign, 2 exponent bits, 1 mantissa bit,
  largest magnitude 6.0), two elements per byte;
* block scale: FP8 E4M3, one per 16 consecutive elements along K;
* global scale: one fp32 per tensor.

Readings adopted where the pages are silent:

* element ``2j`` of a row sits in the low nibble of byte ``j``;
* the global scale handed around is the *quant* convention
  ``gs = (448 * 6) / amax`` ("GLM-5.3-Flash-NVFP4 #4" discussion, follow-up on
  the MoE fault), so the dequantised value is ``e2m1 * e4m3 / gs``;
* the quantiser's operations and their order are those of ``quantize`` below,
  each one a correctly rounded fp32 operation; E4M3 and E2M1 both round to
  nearest with ties to the even code and saturate at their largest finite
  value (448 is the clamp named in "Serving Solar Open 2 on DGX Spark",
  "Supporting real NVFP4 checkpoints"; 6.0 is e2m1's maximum).
"""
from __future__ import annotations

import numpy as np

F32 = np.float32

#: e2m1 code -> value, codes 0..15 (bit 3 is the sign). The magnitudes are the
#: eight values an e2m1 number can take, largest 6.0.
E2M1_VALUES = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0,
                        -0.0, -0.5, -1.0, -1.5, -2.0, -3.0, -4.0, -6.0], dtype=np.float64)

E2M1_MAX = 6.0
E4M3_MAX = 448.0
#: The product of the two maxima, 2688: gs = 2688 / amax maps a tensor's amax
#: onto the largest representable block-scaled element.
QUANT_RANGE = F32(E4M3_MAX * E2M1_MAX)


def e4m3_decode(code):
    """FP8 E4M3 ("fn" variant) code -> float64, by the format's definition.

    Bias 7, 3 mantissa bits, subnormals when the exponent field is 0, no
    infinities, 0x7F and 0xFF are NaN, largest finite magnitude 448.
    Pinned by: torch.float8_e4m3fn over all 256 codes (tests).
    """
    code = np.asarray(code, dtype=np.int64)
    sign = np.where(code & 0x80, -1.0, 1.0)
    exp = (code >> 3) & 0xF
    man = code & 0x7
    sub = man / 8.0 * 2.0 ** -6
    nrm = (1.0 + man / 8.0) * np.exp2(exp.astype(np.float64) - 7.0)
    val = sign * np.where(exp == 0, sub, nrm)
    return np.where((code & 0x7F) == 0x7F, np.nan, val)


def e2m1_decode(code):
    """e2m1 code (0..15) -> float64 via the explicit 16-entry table.

    Pinned by: the magnitude set {0, 0.5, 1, 1.5, 2, 3, 4, 6} (golden file).
    """
    return E2M1_VALUES[np.asarray(code, dtype=np.int64) & 0xF]


# The non-negative finite E4M3 values in code order 0x00..0x7E (increasing).
_E4M3_POS = e4m3_decode(np.arange(0x7F))
_E2M1_POS = E2M1_VALUES[:8]


def _round_to_grid(mag, grid, maximum):
    """Nearest grid point to each non-negative ``mag``; ties to the even code.

    ``grid`` lists the representable non-negative values in code order (so the
    code of ``grid[i]`` is ``i`` and "even code" means even ``i``); values
    above ``maximum`` saturate to the last code. Returns the codes.
    """
    mag = np.asarray(mag, dtype=np.float64)
    hi = np.searchsorted(grid, mag, side="left")          # grid[hi-1] < mag <= grid[hi]
    hi = np.clip(hi, 1, len(grid) - 1)
    lo = hi - 1
    d_lo = mag - grid[lo]
    d_hi = grid[hi] - mag
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (hi % 2 == 0))
    code = np.where(pick_hi, hi, lo)
    code = np.where(mag >= maximum, len(grid) - 1, code)
    code = np.where(mag <= 0.0, 0, code)
    return code.astype(np.int64)


def e4m3_encode(s):
    """Non-negative fp32 -> E4M3 code, round-to-nearest-even, saturating at 448.

    Pinned by: torch.float8_e4m3fn conversion (round to nearest even) on every
    fp32 value of a dense grid below 448; saturation by the 448 clamp.
    """
    s = np.asarray(s, dtype=F32)
    if np.any(s < 0) or np.any(np.isnan(s)):
        raise ValueError("block scales are non-negative and finite")
    return _round_to_grid(s.astype(np.float64), _E4M3_POS, E4M3_MAX)


def e2m1_encode(y):
    """fp32 -> e2m1 code (sign in bit 3), nearest-even, saturating at 6.0.

    The sign of the input is kept even when the magnitude rounds to zero.
    Pinned by: binade-wise numpy half-to-even rounding on a dense grid, and the
    tie table 0.25->0, 0.75->1, 1.25->1, 1.75->2, 2.5->2, 3.5->4, 5->4.
    """
    y = np.asarray(y, dtype=F32)
    mag_code = _round_to_grid(np.abs(y).astype(np.float64), _E2M1_POS, E2M1_MAX)
    return (mag_code | np.where(np.signbit(y), 8, 0)).astype(np.uint8)


def global_scale(amax):
    """Quant-convention global scale ``gs = 2688 / amax`` (fp32); 1 when amax is 0.

    Pinned by: the worked value amax 0.125 -> 21504.0 (golden file).
    """
    amax = F32(amax)
    if amax == 0:
        return F32(1.0)
    return F32(QUANT_RANGE / amax)


def quantize(x, gs=None):
    """Quantise a 2-D tensor to NVFP4 with one per-tensor global scale.

    ``x`` is ``[rows, K]`` with ``K % 16 == 0``, given in any dtype whose values
    are exact in fp32 (bf16 activations and weights). Steps, each a correctly
    rounded fp32 operation:

    1. ``amax = max |x|`` over the whole tensor, ``gs = 2688 / amax``; a
       static (calibrated) ``gs`` given by the caller replaces this step
       ("Serving Solar Open 2 on DGX Spark", "The fix": static and dynamic
       W4A4 paths; "GLM-5.3-Flash-NVFP4 #4", calibrated per-projection input
       scales). With a static scale a block can exceed the range: its scale
       saturates at 448 and its codes at 6;
    2. per block of 16 along K: ``amax_b = max |x_i|``,
       ``s = (amax_b / 6) * gs``, ``sf = E4M3(s)`` (nearest even, clamp 448);
    3. if ``sf`` decodes to 0 the 16 codes are 0; otherwise
       ``r = gs / sf`` and each code is ``e2m1(x_i * r)``.

    Returns ``(codes [rows, K] uint8 unpacked, sf [rows, K/16] uint8, gs fp32)``.
    Pinned by: the golden worked scale; round-trip error bounds; g16 block
    independence; the tie tables of the two encoders; static scale: the
    dynamic result when the static scale equals the dynamic one, the exponent
    shift of the block scales under a power-of-two scale, the saturation of
    out-of-range blocks (tests).
    """
    x = np.asarray(x, dtype=F32)
    rows, K = x.shape
    if K % 16:
        raise ValueError("K must be a multiple of 16")
    if gs is None:
        amax = F32(np.max(np.abs(x))) if x.size else F32(0)
        gs = global_scale(amax)
    else:
        gs = F32(gs)
        if not (np.isfinite(gs) and gs > 0):
            raise ValueError("a static global scale is positive and finite")
    blocks = x.reshape(rows, K // 16, 16)
    amax_b = np.max(np.abs(blocks), axis=2).astype(F32)
    with np.errstate(over="ignore"):
        s = ((amax_b / F32(E2M1_MAX)).astype(F32) * gs).astype(F32)
    sf = e4m3_encode(s).astype(np.uint8)
    sf_val = e4m3_decode(sf).astype(F32)
    with np.errstate(divide="ignore", invalid="ignore"):
        r = np.where(sf_val > 0, gs / np.where(sf_val > 0, sf_val, F32(1)), F32(0)).astype(F32)
    with np.errstate(over="ignore"):
        y = (blocks * r[:, :, None]).astype(F32)
    codes = e2m1_encode(y)
    codes = np.where((sf_val > 0)[:, :, None], codes, np.uint8(0)).astype(np.uint8)
    return codes.reshape(rows, K), sf, gs


def dequantize(codes, sf, gs):
    """NVFP4 -> float64: ``e2m1[code] * e4m3[sf] / gs`` element by element.

    ``codes`` is unpacked ``[rows, K]``, ``sf`` is ``[rows, K/16]``.
    Pinned by: the worked reciprocal value and the wrong-inversion test.
    """
    codes = np.asarray(codes)
    rows, K = codes.shape
    scale = np.repeat(e4m3_decode(sf), 16, axis=1)
    return e2m1_decode(codes) * scale / np.float64(F32(gs))


def pack(codes):
    """Unpacked codes ``[rows, K]`` -> bytes ``[rows, K/2]``, element 2j low nibble."""
    codes = np.asarray(codes, dtype=np.uint8)
    return (codes[:, 0::2] & 0xF) | ((codes[:, 1::2] & 0xF) << 4)


def unpack(packed):
    """Bytes ``[rows, K/2]`` -> codes ``[rows, K]`` (inverse of ``pack``)."""
    packed = np.asarray(packed, dtype=np.uint8)
    out = np.empty((packed.shape[0], packed.shape[1] * 2), dtype=np.uint8)
    out[:, 0::2] = packed & 0xF
    out[:, 1::2] = packed >> 4
    return out


# ---------------------------------------------------------------------------
# Checkpoint import ("Serving Solar Open 2 on DGX Spark", "Supporting real
# NVFP4 checkpoints"; "GLM-5.3-Flash-NVFP4 #4" discussion, follow-up on the
# MoE fault).

#: How a checkpoint stores a tensor's global scale. ModelOpt keeps the dequant
#: scale amax/(448*6) (``weight_scale_2``, ``input_scale``); compressed-tensors
#: keeps the quant scale (448*6)/amax (``global_scale``).
SCALE_FORMATS = ("quant", "dequant")


def import_global_scale(value, fmt):
    """A checkpoint's stored global scale -> the quant-convention ``gs`` (fp32).

    ``fmt`` is "quant" (the value already is ``gs``) or "dequant" (the value is
    ``amax / 2688`` and ``gs`` is its fp32 reciprocal, correctly rounded). A
    value that is not positive and finite is refused: a zero scale multiplies
    every expert by zero without any error, the fault the GLM thread traces.
    Pinned by: the worked pair 4.650297705666162e-05 <-> 21504.0 (golden
    file); exact powers of two; the round trip within one ulp (tests).
    """
    if fmt not in SCALE_FORMATS:
        raise ValueError(fmt)
    v = F32(value)
    if not (np.isfinite(v) and v > 0):
        raise ValueError("a global scale is positive and finite")
    return v if fmt == "quant" else F32(F32(1.0) / v)


def fold_block_scales(sf, ratio):
    """Re-round E4M3 block scales by a factor: ``E4M3(e4m3[sf] * ratio)``.

    Moving a matrix from global scale ``gs_old`` to ``gs_new`` keeps its
    dequantised values ``e2m1 * sf / gs`` when every block scale is multiplied
    by ``ratio = gs_new / gs_old``; the product (one correctly rounded fp32
    multiply) is rounded back to E4M3, nearest even, clamped at 448. A scale
    that underflows to code 0 zeroes its block. Sign-bit and NaN codes are
    refused.
    Pinned by: ratio 1 is the identity on every finite code; a power-of-two
    ratio adds its exponent to the code's exponent field; every code times a
    few ratios against torch's float8_e4m3fn rounding, saturating at 448
    (tests).
    """
    sf = np.asarray(sf, dtype=np.uint8)
    if np.any(sf & 0x80) or np.any((sf & 0x7F) == 0x7F):
        raise ValueError("block scales are non-negative and finite")
    ratio = F32(ratio)
    if not (np.isfinite(ratio) and ratio > 0):
        raise ValueError("the fold ratio is positive and finite")
    with np.errstate(over="ignore"):
        prod = (e4m3_decode(sf).astype(F32) * ratio).astype(F32)
    return e4m3_encode(prod).astype(np.uint8)
