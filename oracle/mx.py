"""MX block-scaled formats, MXFP8 (E4M3 elements) and MXFP4 (E2M1 elements)
(oracle side).  TEST INFRASTRUCTURE ONLY - see the package docstring.

"LLM and AIGC quantization: from number formats to W4A4", block-scaled
formats: every block of elements shares one E8M0 scale, a power of two,

    scale = 2 ^ (floor(log2(absmax)) - e_max)

where e_max is the exponent of the element format's largest value (8 for
E4M3, 448 = 1.75 . 2^8; 2 for E2M1, 6 = 1.5 . 2^2).  The elements are the
block divided by its scale, encoded in the element format.  The same page
puts the block at 16 or 32 elements for the block-scaled formats; MX takes 32.
The tensor core reads the elements and the block scales and applies each
block's scales during accumulation.

Readings where the pages are silent (each is listed in the design notes):
* Block = 32 consecutive elements of a row along K.
* The E8M0 scale code is the biased exponent e + 127.  e is clamped to
  [-127, 127], the codes 0 .. 254 (255 is NaN).  An all-zero block has
  floor(log2 0) = -inf and takes the smallest scale, code 0.
* Division by the power-of-two scale is one float32 multiply by 2^-e (exact
  unless the product is below the float32 normal range, where every element
  format rounds it to zero anyway).
* Quotients above the element format's largest value saturate to it (the
  block maximum divided by its scale lies in [2^e_max, 2^(e_max+1)), above
  448 and 6 for the top of that range), with round-half-to-even codes and
  the sign kept, as in the E2M1 / E4M3 encoders.
Pins: tests/test_oracle_pins.py (the pages' MXFP4 block with its printed
scale 0.5 and 4.8 -> 4, the MXFP8 MSE of the pages' eight-weight example,
the range of the scaled maximum, power-of-two invariance, GEMM brute force).
"""
import numpy as np

from .formats import e2m1_decode, e2m1_encode, e4m3_decode, e4m3_encode

MX_BLOCK = 32
MX_EMAX = {"e4m3": 8, "e2m1": 2}
E8M0_BIAS = 127


def _check_fmt(fmt):
    if fmt not in MX_EMAX:
        raise ValueError("fmt must be 'e4m3' (MXFP8) or 'e2m1' (MXFP4)")


def mx_block_exponent(amax, fmt):
    """e = floor(log2(amax)) - e_max per block, clamped to [-127, 127]; -127
    for amax = 0.  amax: non-negative float32 array."""
    _check_fmt(fmt)
    amax = np.asarray(amax, dtype=np.float32)
    # frexp: amax = m . 2^p with m in [0.5, 1), so floor(log2(amax)) = p - 1
    # (exact, subnormal inputs included)
    _, p = np.frexp(amax.astype(np.float64))
    e = np.where(amax > 0, p.astype(np.int64) - 1 - MX_EMAX[fmt], -E8M0_BIAS)
    return np.clip(e, -E8M0_BIAS, E8M0_BIAS).astype(np.int64)


def mx_quantize(x, fmt):
    """x float32 [rows][K], K a multiple of 32 -> (codes uint8, sf uint8 [rows][K/32]).

    codes are E4M3-FN bytes [rows][K] for 'e4m3', or E2M1 codes 0..15 (one per
    element, unpacked) [rows][K] for 'e2m1'; sf holds the E8M0 codes e + 127.
    """
    _check_fmt(fmt)
    x = np.asarray(x, dtype=np.float32)
    rows, k = x.shape
    if k % MX_BLOCK:
        raise ValueError("K must be a multiple of 32")
    blocks = x.reshape(rows, k // MX_BLOCK, MX_BLOCK)
    amax = np.abs(blocks).max(axis=2) if k else np.zeros((rows, 0), np.float32)
    e = mx_block_exponent(amax, fmt)
    inv_scale = np.ldexp(np.float32(1.0), -e).astype(np.float32)       # 2^-e, a normal float32
    y = (blocks * inv_scale[:, :, None]).astype(np.float32)            # one float32 multiply
    enc = e4m3_encode if fmt == "e4m3" else e2m1_encode
    return enc(y).reshape(rows, k), (e + E8M0_BIAS).astype(np.uint8)


def e8m0_decode(sf):
    """E8M0 codes 0..254 -> float64 powers of two 2^(code - 127)."""
    sf = np.asarray(sf, dtype=np.int64)
    if np.any(sf > 254):
        raise ValueError("E8M0 NaN code")
    return np.ldexp(1.0, sf - E8M0_BIAS)


def mx_dequantize(codes, sf, fmt):
    """Element values times their block scales, float64 [rows][K]."""
    _check_fmt(fmt)
    dec = e4m3_decode(codes) if fmt == "e4m3" else e2m1_decode(codes)
    return dec * np.repeat(e8m0_decode(sf), MX_BLOCK, axis=1)


def mx_gemm_reference(qa, sfa, qb, sfb, fmt):
    """out[t, n] = sum_k deq(a)[t, k] . deq(b)[n, k] in float64 (every product of
    two MX values and every partial sum here is exact or rounded only in
    float64); qa [T][K], qb [N][K] unpacked codes."""
    return mx_dequantize(qa, sfa, fmt) @ mx_dequantize(qb, sfb, fmt).T
