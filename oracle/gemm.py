"""Matrix products of the quantized linear layer (oracle side).

TEST INFRASTRUCTURE ONLY - see the package docstring.

Each product is its plain definition: dequantize both operands exactly
(every dequantized value is a short product, exact in float64), then one
matrix product.  Integer GEMMs are exact.

* w4a16_reference - Y = X . (s (q - z))^T with one scale and zero-point per
  group of consecutive K elements ("Chapter 9 - Quantization kernels",
  section 9.5 dequant-fused GEMM; "LLM and AIGC quantization", section W4A16).
* fp8_gemm_reference - FP8 W8A8: E4M3 operands decoded exactly, one
  product, then s_a[t] . s_b[n] (+ bias) ("LLM and AIGC quantization",
  "W4A4, FP8 and block-scaled formats", the FP8 W8A8 item).
* int8_gemm_exact - D^ = A^ . B^^T with int32 accumulation ("LLM and AIGC
  quantization", W8A8 section: a single product is at most 127^2 = 16129 and
  a K = 4096 sum reaches 6.6e7, so the accumulator must be int32).
* azp_adj_from_weight - 1 . B^, the per-output-channel sum of the int8 weight
  codes ("vLLM W8A8 ... CUTLASS epilogue design", sections 2 and 5).
* w8a8_epilogue - out = s_a s_b (D^ - azp * azp_adj) + bias, the four
  epilogues of the same page (sections 2.1-2.4); bias absent means 0, scalar
  scales broadcast.
* nvfp4_gemm_reference - Y = g_a g_b sum_b s^a_b s^b_b sum_{k in b} a_k b_k over
  the augmented K ("LLM and AIGC quantization", "Block-scaled formats";
  "NVFP4 quantization and ARCQuant", section 2.2).

Parity pins: tests/test_oracle_pins.py (the pages' 2x3 W8A8 example, brute
force on tiny inputs, the azp identity against dequantize-then-multiply,
permutation invariance and S = 0 of the augmented GEMM).
"""

import numpy as np

from .formats import e4m3_decode, unpack_u4
from .quant import nvfp4_dequantize


def w4a16_reference(x, codes, scales, zeros, group=128):
    """float64 Y [T][N] for fp16 X [T][K], codes uint8 [N][K] (0..15),
    scales fp16 [N][K/group], zeros uint8 [N][K/group] or None (meaning 8)."""
    x = np.asarray(x)
    codes = np.asarray(codes, dtype=np.uint8)
    n, k = codes.shape
    g = k // group
    s = np.asarray(scales).astype(np.float64).reshape(n, g, 1)
    z = np.full((n, g, 1), 8.0) if zeros is None else np.asarray(zeros).astype(np.float64).reshape(n, g, 1)
    w = (codes.reshape(n, g, group).astype(np.float64) - z) * s
    return x.astype(np.float64) @ w.reshape(n, k).T


def w4a16_reference_packed(x, wq, scales, zeros_packed, group=128):
    """Same as w4a16_reference, from the packed byte layout."""
    n = wq.shape[0]
    k = wq.shape[1] * 2
    codes = unpack_u4(wq, k)
    zeros = None if zeros_packed is None else unpack_u4(zeros_packed, k // group)
    return w4a16_reference(x, codes, scales, zeros, group)


def w4a16_act_order_reference(x, codes, scales, zeros, g_idx, group=128):
    """W4A16 with act-order ("LLM and AIGC quantization", GPTQ engineering
    details: desc_act quantizes the columns in descending diag(H) order, so
    g_idx records each input channel's group and the scale reads are no longer
    contiguous): column k is dequantized with the scale and zero-point of
    group g_idx[k].  float64 Y [T][N]; codes uint8 [N][K], scales fp16 [N][G],
    zeros uint8 [N][G] or None (8), g_idx int [K] in [0, G)."""
    codes = np.asarray(codes, dtype=np.uint8)
    g_idx = np.asarray(g_idx, dtype=np.int64)
    n, k = codes.shape
    s = np.asarray(scales).astype(np.float64)[:, g_idx]                    # [N][K]
    z = np.full((n, k), 8.0) if zeros is None else np.asarray(zeros).astype(np.float64)[:, g_idx]
    w = (codes.astype(np.float64) - z) * s
    return np.asarray(x).astype(np.float64) @ w.T


def act_order_perm(g_idx, group=128):
    """The column order that makes every group contiguous: a stable sort of the
    columns by g_idx (column perm[j] goes to position j).  Each group must hold
    exactly `group` columns, as GPTQ's act-order assigns them."""
    g_idx = np.asarray(g_idx, dtype=np.int64)
    counts = np.bincount(g_idx, minlength=len(g_idx) // group)
    if len(g_idx) % group or np.any(counts != group):
        raise ValueError("every group must hold exactly `group` columns")
    return np.argsort(g_idx, kind="stable").astype(np.int32)


def int8_gemm_exact(a, b):
    """Exact D^ = A^ B^^T for int8 A^ [T][K], B^ [N][K] -> int64 [T][N].

    Every product and partial sum is an integer below 2^53, so a float64
    matrix product is exact whatever its summation order.  The result is
    checked to fit the int32 accumulator.
    """
    a = np.asarray(a, dtype=np.int8)
    b = np.asarray(b, dtype=np.int8)
    k = a.shape[1]
    assert k * 128 * 128 < 2 ** 53
    d = (a.astype(np.float64) @ b.astype(np.float64).T).astype(np.int64)
    assert d.min(initial=0) >= -(2 ** 31) and d.max(initial=0) < 2 ** 31
    return d


def azp_adj_from_weight(b):
    """1 . B^ : sum over K of the int8 weight codes per output channel (int32 [N])."""
    return np.asarray(b, dtype=np.int8).astype(np.int64).sum(axis=1).astype(np.int32)


def w8a8_epilogue(dhat, scale_a, scale_b, azp=None, azp_adj=None, bias=None):
    """out = s_a * s_b * (D^ - azp * azp_adj) + bias, float64 [T][N].

    azp is None and azp_adj given: per-tensor asymmetric case, azp_adj already
    holds z * (1 . B^).  Both None: symmetric.  Scalar (size-1) scales
    broadcast.  bias None means 0.
    """
    d = np.asarray(dhat, dtype=np.int64)
    t, n = d.shape
    if azp_adj is not None:
        adj = np.asarray(azp_adj, dtype=np.int64).reshape(1, n)
        if azp is not None:
            corr = np.asarray(azp, dtype=np.int64).reshape(t, 1) * adj
        else:
            corr = np.broadcast_to(adj, (t, n))
        d = d - corr
    sa = np.asarray(scale_a, dtype=np.float64).reshape(-1, 1)
    sb = np.asarray(scale_b, dtype=np.float64).reshape(1, -1)
    out = sa * (sb * d.astype(np.float64))
    if bias is not None:
        out = out + np.asarray(bias).astype(np.float64).reshape(1, n)
    return out


def nvfp4_gemm_reference(qa, sfa, ga, qb, sfb, gb):
    """float64 Y [T][N] from NVFP4 operands (codes [rows][K_aug], scales
    [rows][K_aug/16], per-tensor scales ga, gb)."""
    a = nvfp4_dequantize(qa, sfa, ga)
    b = nvfp4_dequantize(qb, sfb, gb)
    return a @ b.T


def fp8_gemm_reference(qa, sa, qb, sb, bias=None):
    """float64 Y [T][N] = sa[t] . sb[n] . sum_k dec(qa[t,k]) . dec(qb[n,k]) (+ bias[n])
    for E4M3 codes qa [T][K], qb [N][K] and float32 scales sa [T], sb [N]
    ("LLM and AIGC quantization", "W4A4, FP8 and block-scaled formats": FP8
    products accumulated in high precision, both scales applied after the
    sum).  The decoded products have at most 8 significant bits and the sums
    stay within 53, so the float64 contraction is exact."""
    a = e4m3_decode(qa)
    b = e4m3_decode(qb)
    y = (a @ b.T) * np.asarray(sa, dtype=np.float64)[:, None] * np.asarray(sb, dtype=np.float64)[None, :]
    if bias is not None:
        y = y + np.asarray(bias, dtype=np.float64)[None, :]
    return y
