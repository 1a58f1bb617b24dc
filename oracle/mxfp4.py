"""MXFP4 (e2m1 elements, one power-of-two E8M0 scale per 32) written out plainly.

Test infrastructure only (see the package docstring for who may import it).

Format, from "vLLM on the NVIDIA DGX Spark: A Complete Technical Guide",
section 6.4 "NVFP4 vs MXFP4": the same 4-bit e2m1 elements as NVFP4, but
blocks of 32 along K and an exponent-only E8M0 block scale (no FP8 mantissa,
no per-tensor global scale).

Reading adopted where the page is silent (the plain definition of a
microscaling format): the block scale is 2^(floor(log2 amax_b) - 2), 2 being
the exponent of e2m1's largest value 6 = 1.5 * 2^2, so amax_b / scale lies in
[4, 8); each element is x / scale rounded to e2m1 (nearest, ties to the even
code, saturating at 6, sign kept); an all-zero block takes the smallest scale
2^-127 (code 0) and zero codes. E8M0 code c means 2^(c - 127); 0xFF is NaN.
"""
from __future__ import annotations

import numpy as np

from . import nvfp4

F32 = np.float32
BLOCK = 32
E2M1_EMAX = 2       # 6 = 1.5 * 2^2
E8M0_BIAS = 127


def e8m0_decode(code):
    """E8M0 code -> float64: 2^(code - 127); 0xFF is NaN.

    Pinned by: torch.float8_e8m0fnu over all 256 codes (tests).
    """
    code = np.asarray(code, dtype=np.int64)
    val = np.exp2(code.astype(np.float64) - E8M0_BIAS)
    return np.where(code == 0xFF, np.nan, val)


def _floor_log2(a):
    """floor(log2 a) of positive finite fp32 values, exactly (from the bits)."""
    a = np.asarray(a, dtype=F32)
    bits = a.view(np.uint32).astype(np.int64)
    exp = (bits >> 23) & 0xFF
    man = bits & 0x7FFFFF
    # subnormals: the position of the leading mantissa bit
    sub = np.where(man > 0, np.floor(np.log2(np.maximum(man, 1))).astype(np.int64), 0) - 149
    return np.where(exp > 0, exp - 127, sub)


def quantize(x):
    """Quantise ``[rows, K]`` (``K % 32 == 0``, values exact in fp32) to MXFP4.

    Per block of 32 along K: ``e = floor(log2 amax_b) - 2`` (clamped to
    [-127, 127]), scale code ``e + 127``, codes ``e2m1(x_i / 2^e)``.
    Returns ``(codes [rows, K] uint8 unpacked, scale codes [rows, K/32] uint8)``.
    Pinned by: amax_b / scale in [4, 8) (closed form); a power-of-two factor
    on x moves every scale code by its exponent and leaves the codes alone;
    blocks built from e2m1 values round-trip exactly; the saturation of
    amax_b / scale in (6, 8) to 6; block independence; the round-trip bound
    (tests).
    """
    x = np.asarray(x, dtype=F32)
    rows, K = x.shape
    if K % BLOCK:
        raise ValueError("K must be a multiple of 32")
    blocks = x.reshape(rows, K // BLOCK, BLOCK)
    amax = np.max(np.abs(blocks), axis=2)
    zero = amax == 0
    e = np.where(zero, -E8M0_BIAS, _floor_log2(np.where(zero, F32(1), amax)) - E2M1_EMAX)
    e = np.clip(e, -E8M0_BIAS, E8M0_BIAS)
    scale = np.exp2(e.astype(np.float64))
    y = (blocks.astype(np.float64) / scale[:, :, None]).astype(F32)   # exact: a power of two
    codes = nvfp4.e2m1_encode(y)
    codes = np.where(zero[:, :, None], np.uint8(0), codes).astype(np.uint8)
    return codes.reshape(rows, K), (e + E8M0_BIAS).astype(np.uint8)


def dequantize(codes, scale_codes):
    """MXFP4 -> float64: ``e2m1[code] * 2^(scale - 127)`` element by element."""
    codes = np.asarray(codes)
    scale = np.repeat(e8m0_decode(scale_codes), BLOCK, axis=1)
    return nvfp4.e2m1_decode(codes) * scale
