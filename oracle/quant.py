"""Quantizers of the quantized linear layer (oracle side).

TEST INFRASTRUCTURE ONLY - see the package docstring.

All arithmetic is float32, one IEEE operation at a time, in the order the
pages write it; integer rounding is round-half-to-even ("LLM and AIGC
quantization", notation paragraph: hand examples use round-half-to-even).

Functions and the passages they follow:

* quantize_affine / dequantize_affine - q = round(x/s) + z, x^ = s (q - z)
  ("Chapter 9 - Quantization kernels", section 9.2; zero-point added on
  quantize and subtracted on dequantize).
* quant_sym_rows / quant_int8_sym - per-token symmetric int8: s = max|x| / 127, codes in
  [-127, 127] ("LLM and AIGC quantization", "Symmetric and asymmetric":
  s = max|x| / q_max, q_max = 2^(b-1) - 1; "Granularity": per-token
  dynamic scales for W8A8).  Also used per output channel for W8A8 weights.
* quant_int8_asym - per-token asymmetric int8 mapping [min, max] onto
  [-128, 127] with an integer zero-point so that 0 is exact (same section;
  the zero-point form of the W8A8 epilogue page, section 2).
* quant_w4_g128 - asymmetric unsigned 4-bit weights, one fp16 scale and one
  4-bit zero-point per 128 consecutive K elements of a row (AWQ offline flow,
  ``pseudo_quant``: s = clamp(max - min, 1e-5) / 15, z = round(-min / s),
  q = clamp(round(w / s) + z, 0, 15)).
* nvfp4_global_scale / nvfp4_quantize / nvfp4_dequantize - 16-element blocks
  of E2M1 with an E4M3 block scale absmax / 6, elements divided by the
  decoded scale and rounded to the nearest E2M1 value ("LLM and AIGC
  quantization", "Block-scaled formats", the 16-element NVFP4 example), with
  a per-tensor fp32 second-level scale.
* quant_fp8_rows / quant_fp8_tensor - FP8 W8A8: x / s converted to E4M3
  instead of rounded to an integer, s = max|x| / 448 per token (activations)
  or per output channel (weights), or one scale per tensor ("LLM and AIGC
  quantization", "W4A4, FP8 and block-scaled formats": the FP8 W8A8 item;
  "FP8: robustness from dynamic range": the per-tensor worked example
  [0.6, -45.0, 1.1, -0.8] -> 6, -448, 11, -8).
* rmsnorm_rows / rmsnorm_quant_int8 / rmsnorm_quant_fp8 - RMSNorm with the
  per-token quantization fused into it ("Chapter 9 - Quantization kernels",
  practical notes: the per-row max and the quantization fused into the
  upstream operator, vLLM's rms_norm_dynamic_per_token_quant; "LLM and AIGC
  quantization", "Static and dynamic quantization": the per-token reduction
  is usually fused into the preceding RMSNorm; "SmoothQuant" inference
  configuration: the RMSNorm kernel emits per-token quantized output).  The
  normalized row is y = (x . (1 / sqrt(mean(x^2) + eps))) . gamma, quantized
  per token by quant_int8_sym or quant_fp8_rows without being rounded first.
* arc_perm / arc_quantize_activation / arc_quantize_weight - ARCQuant
  residual-channel augmentation ("NVFP4 quantization and ARCQuant",
  sections 2.1 and 2.2): reorder channels by magnitude, quantize, re-quantize
  the residual of the first S channels and append it along K; weights get
  the same order and a copy of their first S columns.

Readings where the pages are silent (each is also listed in the design
notes):

* quant_int8_sym: an all-zero row uses s = 1 (all codes 0).
* quant_int8_asym: the range always includes 0 (min <= 0 <= max) because the
  zero-point must make 0 exactly representable; the range is floored at
  1e-5 as in the AWQ code; z = -128 - round(min / s) and the code is
  round(x / s) + z (round first, then add the integer zero-point).
* quant_w4_g128: the scale is rounded to fp16 first and the rounded value is
  the one used to quantize (it is what dequantization uses); z is clamped to
  [0, 15].
* NVFP4: the per-tensor scale is g = amax(|X|) / (6 * 448) so block scales
  land in E4M3 range (the pages' example sets it to 1); a block whose decoded
  scale d = dec(s) * g is 0 gets all-zero codes; the residual of the ARCQuant
  channels uses the same g as the main part.
* quant_fp8_*: the scale maps the largest magnitude onto the largest finite
  E4M3 value, s = max|x| / 448 (the pages print the codes of their example,
  which this scale reproduces, not the formula); an all-zero row or tensor
  uses s = 1; x / s is a float32 division, then the E4M3 encode (nearest,
  ties to even, saturating).
* rmsnorm_*: RMSNorm is y = (x . inv) . gamma with inv = 1 / sqrt(mean(x^2)
  + eps); the pages fix neither the formula nor eps (it is an argument).
  The mean of squares is the exact sum of the row's squares (exact
  rational arithmetic; every float32 square is exact in it) rounded once
  to float32, round to nearest, ties to even, then one float32 division by
  K: the pages fix no order of summation, and this is the one result that
  no order of float32 additions can change.  The remaining steps are
  separate float32 operations (add eps, square root, divide 1 by it once
  per row, then two multiplies per element).  A row whose mean(x^2) + eps
  is 0 (eps = 0 and every square 0 or rounding to 0) normalizes to 0.  The
  normalized values are quantized as they are, never rounded to the input
  dtype first.
* arc_perm: calibration statistic = max over rows of |X| per channel, taken
  on X itself; channels sorted by descending statistic, ties by ascending
  channel index.

Parity pins: tests/test_oracle_pins.py.
"""

import numpy as np

from .formats import e2m1_decode, e2m1_encode, e4m3_decode, e4m3_encode

F32 = np.float32


def quantize_affine(x, s, z, qmin, qmax):
    """q = clamp(round(x / s) + z, qmin, qmax), float32 division, RNE."""
    x = np.asarray(x, dtype=np.float32)
    s = np.asarray(s, dtype=np.float32)
    r = np.rint(x / s).astype(np.float64)
    return np.clip(r + np.asarray(z, dtype=np.float64), qmin, qmax).astype(np.int64)


def dequantize_affine(q, s, z):
    """x^ = s * (q - z), in float64."""
    return np.asarray(s, dtype=np.float64) * (np.asarray(q, dtype=np.float64) - np.asarray(z, dtype=np.float64))


def quant_sym_rows(x, qmax):
    """Per-row symmetric quantization with codes in [-qmax, qmax].

    s = max|x| / qmax (float32), q = clamp(round(x / s), -qmax, qmax); an
    all-zero row uses s = 1.  Returns (q int64, s float32 [rows]).
    """
    x = np.asarray(x, dtype=np.float32)
    a = np.abs(x).max(axis=1)
    s = a / F32(qmax)
    s = np.where(a == 0, F32(1.0), s).astype(np.float32)
    q = np.clip(np.rint(x / s[:, None]), -qmax, qmax).astype(np.int64)
    return q, s


def quant_int8_sym(x):
    """Per-row symmetric int8.  x: float32 [rows][K] -> (q int8, s float32 [rows])."""
    q, s = quant_sym_rows(x, 127)
    return q.astype(np.int8), s


def quant_int8_asym(x):
    """Per-row asymmetric int8.  x: float32 [rows][K] -> (q int8, s float32, z int32)."""
    x = np.asarray(x, dtype=np.float32)
    mn = np.minimum(x.min(axis=1), F32(0.0))
    mx = np.maximum(x.max(axis=1), F32(0.0))
    s = (np.maximum(mx - mn, F32(1e-5)) / F32(255.0)).astype(np.float32)
    z = (-128 - np.rint(mn / s).astype(np.int64)).astype(np.int32)
    r = np.rint(x / s[:, None]).astype(np.int64)
    q = np.clip(r + z[:, None].astype(np.int64), -128, 127).astype(np.int8)
    return q, s, z


def quant_w4_g128(w, group=128):
    """Asymmetric 4-bit group quantization of weights W [N][K] (float32).

    Returns (codes uint8 [N][K] in 0..15, scales float16 [N][K/group],
    zeros uint8 [N][K/group] in 0..15).
    """
    w = np.asarray(w, dtype=np.float32)
    n, k = w.shape
    if k % group:
        raise ValueError("K must be a multiple of the group size")
    g = w.reshape(n, k // group, group)
    mx = g.max(axis=2)
    mn = g.min(axis=2)
    s16 = (np.maximum(mx - mn, F32(1e-5)) / F32(15.0)).astype(np.float16)
    s = s16.astype(np.float32)
    z = np.clip(np.rint(-mn / s), 0, 15)
    q = np.clip(np.rint(g / s[:, :, None]) + z[:, :, None], 0, 15)
    return q.reshape(n, k).astype(np.uint8), s16, z.astype(np.uint8)


def nvfp4_global_scale(x):
    """Per-tensor second-level scale g = amax(|x|) / (6 * 448), float32."""
    x = np.asarray(x, dtype=np.float32)
    return F32(np.abs(x).max()) / F32(2688.0)


def _block_divisor(sf, g):
    """Decoded block scale times the per-tensor scale, d = dec(sf) * g (float32)."""
    return (e4m3_decode(sf).astype(np.float32) * F32(g)).astype(np.float32)


def nvfp4_quantize(x, g):
    """NVFP4 block quantization of x [rows][K] (float32, K % 16 == 0).

    Per 16-element block b of a row:
      s_b  = E4M3((max|x_b| / 6) / g)
      d_b  = dec(s_b) * g
      q    = E2M1(x / d_b)           (all zero when d_b == 0)
    Returns (codes uint8 [rows][K], sf uint8 [rows][K/16]).
    """
    x = np.asarray(x, dtype=np.float32)
    rows, k = x.shape
    if k % 16:
        raise ValueError("K must be a multiple of 16")
    g = F32(g)
    blocks = x.reshape(rows, k // 16, 16)
    amax = np.abs(blocks).max(axis=2)
    v = (amax / F32(6.0)) / g
    sf = e4m3_encode(v)
    d = _block_divisor(sf, g)
    with np.errstate(divide="ignore", invalid="ignore"):
        y = blocks / d[:, :, None]
    q = e2m1_encode(y)
    q[d == 0] = 0
    return q.reshape(rows, k), sf


def nvfp4_dequantize(codes, sf, g):
    """Exact float64 value of each NVFP4 element: e2m1(q) * dec(s) * g."""
    codes = np.asarray(codes, dtype=np.uint8)
    rows, k = codes.shape
    e = e2m1_decode(codes).reshape(rows, k // 16, 16)
    sc = e4m3_decode(sf)[:, :, None] * np.float64(F32(g))
    return (e * sc).reshape(rows, k)


def arc_perm(x):
    """Channel order by descending max over rows of |x|, ties by ascending index."""
    x = np.asarray(x, dtype=np.float32)
    stat = np.abs(x).max(axis=0)
    return np.argsort(-stat.astype(np.float64), kind="stable").astype(np.int32)


def arc_quantize_activation(x, perm, s_res, g):
    """ARCQuant activation quantization.

    1. reorder channels: xs = x[:, perm]
    2. main part: NVFP4(xs) with per-tensor scale g
    3. residual of the first S reordered channels:
       r = xs[:, :S] - e2m1(q) * d      (float32, the divisor d of step 2)
    4. NVFP4(r) with the same g, appended along K
    Returns (codes [rows][K+S], sf [rows][(K+S)/16]).
    """
    x = np.asarray(x, dtype=np.float32)
    rows, k = x.shape
    if s_res % 16 or s_res < 0 or s_res > k:
        raise ValueError("S must be a multiple of 16 in [0, K]")
    xs = x[:, np.asarray(perm)] if perm is not None else x
    q, sf = nvfp4_quantize(xs, g)
    if s_res == 0:
        return q, sf
    d = _block_divisor(sf[:, : s_res // 16], g)                      # [rows][S/16]
    e = e2m1_decode(q[:, :s_res]).astype(np.float32).reshape(rows, s_res // 16, 16)
    deq = (e * d[:, :, None]).astype(np.float32)                      # one float32 multiply
    r = (xs[:, :s_res].reshape(rows, s_res // 16, 16) - deq).astype(np.float32)
    qr, sfr = nvfp4_quantize(r.reshape(rows, s_res), g)
    return np.concatenate([q, qr], axis=1), np.concatenate([sf, sfr], axis=1)


def arc_quantize_weight(w, perm, s_res, g):
    """ARCQuant weight side: NVFP4(W[:, perm]) with the codes and scales of the
    first S columns copied (not recomputed) and appended along K."""
    w = np.asarray(w, dtype=np.float32)
    if s_res % 16 or s_res < 0 or s_res > w.shape[1]:
        raise ValueError("S must be a multiple of 16 in [0, K]")
    ws = w[:, np.asarray(perm)] if perm is not None else w
    q, sf = nvfp4_quantize(ws, g)
    if s_res == 0:
        return q, sf
    return (np.concatenate([q, q[:, :s_res]], axis=1),
            np.concatenate([sf, sf[:, : s_res // 16]], axis=1))


def quant_fp8_rows(x):
    """Per-row FP8 E4M3.  x: float32 [rows][K] -> (codes uint8 [rows][K], s float32 [rows]).

    s = max|x| / 448 in float32 (1 for an all-zero row); codes = E4M3(x / s)
    with x / s a float32 division.
    """
    x = np.asarray(x, dtype=np.float32)
    a = np.abs(x).max(axis=1)
    s = (a / F32(448.0)).astype(np.float32)
    s = np.where(a == 0, F32(1.0), s).astype(np.float32)
    return e4m3_encode(x / s[:, None]), s


def quant_fp8_tensor(x):
    """Per-tensor FP8 E4M3: one scale max|x| / 448 for the whole array."""
    x = np.asarray(x, dtype=np.float32)
    a = np.abs(x).max() if x.size else F32(0.0)
    s = F32(1.0) if a == 0 else F32(a / F32(448.0))
    return e4m3_encode(x / s), s


def _f32_fields(x):
    """(m, p) per float32 element, with x = m . 2^(p/2 - 149) exactly: m the
    integer significand (implicit bit included), p = 2 max(E, 1) - 2 for the
    exponent field E, so that x^2 = m^2 . 2^(p - 298)."""
    bits = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.int64)
    e = (bits >> 23) & 0xFF
    man = bits & 0x7FFFFF
    m = np.where(e > 0, man | 0x800000, man)
    return m, 2 * np.maximum(e, 1) - 2


def _round_to_f32(n):
    """The float32 nearest to n . 2^-298 (n a non-negative Python integer),
    ties to even, +inf past the largest finite float32."""
    if n == 0:
        return np.float32(0.0)
    lead = n.bit_length() - 1               # position of the leading bit
    ulp = max(lead - 23, 149)               # 24 significant bits, nothing below 2^-149
    q, r = divmod(n, 1 << ulp)
    half = 1 << (ulp - 1)
    if r > half or (r == half and q & 1):
        q += 1
    if ulp - 298 + q.bit_length() - 1 > 127:
        return np.float32(np.inf)
    return np.float32(float(q) * 2.0 ** (ulp - 298))   # q <= 2^24: exact in float64 and float32


def sum_squares_f32(x):
    """Per row: the exact sum of the squares of the float32 values, rounded
    once to float32 (nearest, ties to even).  A NaN element gives NaN, an
    infinite one +inf.  x: float32 [rows][K] -> float32 [rows]."""
    x = np.asarray(x, dtype=np.float32)
    out = np.empty(x.shape[0], dtype=np.float32)
    for i, row in enumerate(x):
        if np.isnan(row).any():
            out[i] = np.float32(np.nan)
            continue
        if np.isinf(row).any():
            out[i] = np.float32(np.inf)
            continue
        m, p = _f32_fields(row)
        n = 0
        for pos in np.unique(p):                        # squares sharing an exponent: one integer sum
            sq = [int(v) * int(v) for v in m[p == pos]]
            n += sum(sq) << int(pos)
        out[i] = _round_to_f32(n)
    return out


def rmsnorm_rows(x, gamma, eps):
    """y = (x . (1 / sqrt(mean(x^2) + eps))) . gamma per row in float32, the mean
    of squares being sum_squares_f32(x) / K.  x: float32 [rows][K], gamma:
    float32 [K] -> y float32 [rows][K]."""
    x = np.asarray(x, dtype=np.float32)
    g = np.asarray(gamma, dtype=np.float32)
    k = x.shape[1]
    with np.errstate(over="ignore", invalid="ignore"):
        ms = (sum_squares_f32(x) / np.float32(k)).astype(np.float32)
        r = np.sqrt((ms + np.float32(eps)).astype(np.float32)).astype(np.float32)
    with np.errstate(divide="ignore"):
        inv = np.where(r == 0, np.float32(0.0), np.float32(1.0) / r).astype(np.float32)
    with np.errstate(invalid="ignore"):
        return ((x * inv[:, None]).astype(np.float32) * g[None, :]).astype(np.float32)


def rmsnorm_quant_int8(x, gamma, eps):
    """RMSNorm fused with per-token symmetric int8: (q int8, s float32 [rows])."""
    return quant_int8_sym(rmsnorm_rows(x, gamma, eps))


def rmsnorm_quant_fp8(x, gamma, eps):
    """RMSNorm fused with per-token FP8 E4M3: (codes uint8, s float32 [rows])."""
    return quant_fp8_rows(rmsnorm_rows(x, gamma, eps))


def rmsnorm_arc_quantize_activation(x, gamma, eps, perm, s_res, g):
    """RMSNorm fused with the ARCQuant NVFP4 activation quantizer: the float32
    RMSNorm output y of rmsnorm_rows (gamma applied at each channel's own
    position), then arc_quantize_activation(y, perm, S, g).  g and perm belong
    to y, the activations the GEMM consumes."""
    return arc_quantize_activation(rmsnorm_rows(x, gamma, eps), perm, s_res, g)
