"""Pins of the CPU oracle to facts fixed outside the oracle itself.

Each check ties an oracle function to a value printed on one of the pages
(fixtures under tests/golden/, each naming its source), to a closed form, to
an independent library routine (torch's float8_e4m3fn), to exact brute force
on tiny inputs, or to an invariant of the mathematics.  The mutation tests at
the end plant plausible mistakes in the oracle and check that a pin fails.
"""

import fractions
import itertools

import numpy as np
import pytest

import oracle
from oracle import formats as ofmt
from oracle import gemm as ogemm
from oracle import quant as oquant
from oracle import mx as oquant_mx
from oracle import hadamard as oquant_had
from conftest import load_golden

F32 = np.float32


# --------------------------------------------------------------------------
# Affine quantization (Chapter 9, section 9.2; LLM quantization, linear
# quantization / symmetric and asymmetric / granularity)
# --------------------------------------------------------------------------

def pin_int8_range_example():
    g = load_golden("int8_range_example.json")
    s_exact = g["scale_exact_num"] / g["scale_exact_den"]
    for s in (s_exact, g["scale_printed"]):
        for x, q in g["quantize"]:
            assert int(oracle.quantize_affine(x, s, 0, -128, 127)) == q
    d = g["dequantize_printed"]
    x = float(oracle.dequantize_affine(d["q"], g["scale_printed"], 0))
    assert abs(x - d["x"]) < 5e-4
    assert abs(abs(x - 1.5) - d["abs_err_printed"]) < 5e-4


def test_int8_range_example():
    pin_int8_range_example()


def pin_linear_ruler():
    """The 4-bit ruler over [-1.5, 3.0]: spacing 0.3, zero-point 5, via the
    group weight quantizer on a group spanning that range."""
    g = load_golden("linear_ruler.json")
    w = np.linspace(g["x_min"], g["x_max"], 128, dtype=np.float32)[None, :]
    codes, s16, z = oracle.quant_w4_g128(w, group=128)
    assert abs(float(s16[0, 0]) - g["scale"]) < 1e-3     # fp16 rounding of 0.3
    assert int(z[0, 0]) == g["zero_point"]
    for code, value in g["code_to_value"]:
        i = int(np.argmin(np.abs(w[0] - value)))
        assert int(codes[0, i]) == code
    # every element is reproduced to within half a step
    deq = (codes.astype(np.float64) - z.astype(np.float64)) * float(s16[0, 0])
    assert np.max(np.abs(deq - w)) <= float(s16[0, 0]) / 2 + 1e-6


def test_linear_ruler():
    pin_linear_ruler()


def pin_sym_asym_vector():
    g = load_golden("sym_asym_vector.json")
    x = np.array(g["x"], dtype=np.float32)[None, :]
    # symmetric INT4: s = max|x| / 7, codes -7..7
    q, s = oracle.quant_sym_rows(x, g["sym_int4"]["qmax"])
    assert q.min() >= -7 and q.max() <= 7
    mse_sym = np.mean((oracle.dequantize_affine(q, s[:, None], 0) - x) ** 2)
    assert abs(mse_sym - g["sym_int4"]["mse_printed"]) < 5e-5
    # asymmetric unsigned INT4 (the group quantizer with a group of 8)
    codes, s16, z = oracle.quant_w4_g128(x, group=8)
    a = g["asym_uint4"]
    assert int(z[0, 0]) == a["zero_point"]
    deq = oracle.dequantize_affine(codes, float(s16[0, 0]), float(z[0, 0]))
    assert abs(np.mean((deq - x) ** 2) - a["mse_printed"]) < 5e-5
    assert abs(deq[0, 5] - a["x_minus_2_80_dequant_printed"]) < 5e-3
    assert abs((float(z[0, 0]) - 2.80 / float(s16[0, 0])) - a["grid_shift_in_steps_printed"]) < 5e-3
    assert abs((mse_sym - np.mean((deq - x) ** 2)) / mse_sym - g["asym_vs_sym_improvement_printed"]) < 0.01
    # INT8 symmetric: scale about 1/18 of INT4's, MSE about 460x smaller
    q8, s8 = oracle.quant_int8_sym(x)
    r = g["int8_vs_int4"]
    assert abs(float(s[0]) / float(s8[0]) - r["scale_ratio_printed"]) < 0.5
    mse8 = np.mean((oracle.dequantize_affine(q8, s8[:, None], 0) - x) ** 2)
    assert abs(mse_sym / mse8 / r["mse_ratio_printed"] - 1) < 0.02
    # the GELU vector
    ge = g["gelu"]
    xg = np.array(ge["x"], dtype=np.float32)[None, :]
    qg, sg = oracle.quant_sym_rows(xg, 7)
    assert abs(np.mean((oracle.dequantize_affine(qg, sg[:, None], 0) - xg) ** 2) - ge["sym_int4_mse_printed"]) < 5e-6
    cg, s16g, zg = oracle.quant_w4_g128(xg, group=8)
    assert int(zg[0, 0]) == ge["asym_zero_point"]
    assert abs(float(s16g[0, 0]) - ge["asym_scale_num"] / ge["asym_scale_den"]) < 2e-4
    deqg = oracle.dequantize_affine(cg, float(s16g[0, 0]), float(zg[0, 0]))
    assert abs(np.mean((deqg - xg) ** 2) - ge["asym_uint4_mse_printed"]) < 5e-6


def test_sym_asym_vector():
    pin_sym_asym_vector()


def pin_granularity():
    g = load_golden("granularity_example.json")
    w = np.array(g["W"], dtype=np.float32)
    s_t = np.abs(w).max() / F32(7)
    assert abs(float(s_t) - g["per_tensor"]["scale_printed"]) < 5e-5
    q_t = oracle.quantize_affine(w, s_t, 0, -7, 7)
    assert q_t[0].tolist() == g["per_tensor"]["row1_codes"]
    mse_row1 = np.mean((oracle.dequantize_affine(q_t[0], s_t, 0) - w[0]) ** 2)
    assert abs(mse_row1 - g["per_tensor"]["row1_mse_printed"]) < 5e-5
    pc = g["per_channel_row1"]
    q, s = oracle.quant_sym_rows(w, 7)
    assert q[0].tolist() == pc["codes"]                     # 3.5 -> 4 (RNE tie)
    assert abs(float(s[0]) - pc["scale_num"] / pc["scale_den"]) < 1e-7
    deq = oracle.dequantize_affine(q[0], s[0], 0)
    assert np.max(np.abs(deq - np.array(pc["dequant_printed"]))) < 5e-4
    assert abs(np.mean((deq - w[0]) ** 2) - pc["mse_printed"]) < 5e-5


def test_granularity():
    pin_granularity()


def test_round_half_to_even():
    # ties at the integer level go to the even integer
    xs = np.array([0.5, 1.5, 2.5, -0.5, -1.5, -2.5], dtype=np.float32)
    assert oracle.quantize_affine(xs, 1.0, 0, -128, 127).tolist() == [0, 2, 2, 0, -2, -2]


def test_int8_sym_properties():
    rng = np.random.default_rng(11)
    x = rng.standard_normal((64, 96)).astype(np.float16).astype(np.float32)
    x[3] = 0.0
    q, s = oracle.quant_int8_sym(x)
    assert q.dtype == np.int8 and q.min() >= -127
    assert s[3] == 1.0 and not q[3].any()
    nz = np.arange(64) != 3
    # the largest magnitude in each row maps to +-127
    assert np.all(np.abs(q[nz]).max(axis=1) == 127)
    # every element is reproduced to within half a step
    err = np.abs(q.astype(np.float64) * s[:, None] - x)
    assert np.all(err <= s[:, None].astype(np.float64) * (0.5 + 2e-5))


def test_int8_asym_properties():
    rng = np.random.default_rng(12)
    x = rng.uniform(-1, 3, size=(64, 96)).astype(np.float16).astype(np.float32)
    x[5] = np.abs(x[5])          # a row that does not straddle 0
    q, s, z = oracle.quant_int8_asym(x)
    assert q.dtype == np.int8 and z.dtype == np.int32
    assert np.all((z >= -128) & (z <= 127))
    # 0 is exactly representable: dequant(z) == 0
    assert np.all(oracle.dequantize_affine(z, s, z) == 0)
    # the row minimum (or 0) maps to -128; everything within half a step
    mn = np.minimum(x.min(axis=1), 0)
    i = np.argmin(x, axis=1)
    assert np.all(q[np.arange(64), i][mn < 0] == -128)
    deq = oracle.dequantize_affine(q, s[:, None], z[:, None])
    assert np.all(np.abs(deq - x) <= s[:, None].astype(np.float64) * (0.5 + 2e-5))


def pin_zero_point_added_after_rounding():
    """Chapter 9, section 9.2 writes x_int = round(x / s) + z: the integer
    zero-point is added after rounding (AWQ's pseudo_quant on the LLM
    quantization page does the same: (w / s).round().add(z)).  The order
    matters on a tie with an odd zero-point.

    int8, per token: the row range [-17/16, 14.875] gives s = (255/16) / 255
    = 1/16 exactly and z = -128 - round(-17) = -111; x = 5/32 is x / s = 2.5,
    so round(2.5) + z = 2 - 111 = -109 (rounding 2.5 - 111 instead gives
    -108).  The range ends map to -128 and 127, and 0 to z.

    4-bit weights, per group of 128: the range [-5/16, 10/16] gives s = 1/16
    (exact in fp16) and z = round(5) = 5; w = 5/32 is w / s = 2.5, so the code
    is 2 + 5 = 7 (not round(7.5) = 8)."""
    x = np.array([[-17 / 16, 14.875, 5 / 32, 0.0]], dtype=np.float32)
    q, sc, z = oracle.quant_int8_asym(x)
    assert sc[0] == np.float32(1 / 16) and z[0] == -111
    assert q.tolist() == [[-128, 127, -109, -111]]
    w = np.zeros((1, 128), dtype=np.float32)
    w[0, :3] = [-5 / 16, 10 / 16, 5 / 32]
    codes, s16, zw = oracle.quant_w4_g128(w)
    assert s16[0, 0] == np.float16(1 / 16) and zw[0, 0] == 5
    assert codes[0, :4].tolist() == [0, 15, 7, 5]


def test_zero_point_added_after_rounding():
    pin_zero_point_added_after_rounding()


def test_w4_g128_properties():
    rng = np.random.default_rng(13)
    w = (rng.standard_normal((8, 512)) * 0.02).astype(np.float32)
    codes, s16, z = oracle.quant_w4_g128(w)
    assert codes.shape == (8, 512) and s16.shape == (8, 4) and s16.dtype == np.float16
    assert codes.max() <= 15 and z.max() <= 15
    deq = (codes.reshape(8, 4, 128).astype(np.float64) - z[..., None]) * s16[..., None].astype(np.float64)
    assert np.all(np.abs(deq.reshape(8, 512) - w) <= s16.astype(np.float64).repeat(128, axis=1) * (0.5 + 2e-5))


# --------------------------------------------------------------------------
# Integer formats and packing (LLM quantization, "Integers", "W4A16")
# --------------------------------------------------------------------------

def test_int4_twos_complement():
    g = load_golden("int_formats.json")
    for bits, v in g["int4_twos_complement"]:
        assert oracle.int4_decode(int(bits, 2), signed=True) == v
    for bits, v in g["int4_unsigned"]:
        assert oracle.int4_decode(int(bits, 2), signed=False) == v
    # signed codes q - 8 with zero-point z - 8 dequantize identically
    q = np.arange(16)
    for z in range(16):
        assert np.array_equal(oracle.dequantize_affine(q, 0.02, z), oracle.dequantize_affine(q - 8, 0.02, z - 8))


def test_packing_example():
    g = load_golden("int_formats.json")["packing"]
    packed = oracle.pack_u4(np.array(g["codes"], dtype=np.uint8))
    assert packed.view("<u4")[0] == int(g["word_hex"], 16)
    assert oracle.unpack_u4(packed, 8).tolist() == g["codes"]
    # q_i << 4i, read back by shifting right 4i and masking
    word = int(g["word_hex"], 16)
    assert [(word >> (4 * i)) & 0xF for i in range(8)] == g["codes"]


def test_int4_unpack_magic_constants():
    """The constants of the register-level INT4 -> FP16/BF16 unpack."""
    torch = pytest.importorskip("torch")
    g = load_golden("int4_unpack_magic.json")

    def h(bits):
        return float(np.array([int(bits, 16)], dtype=np.uint16).view(np.float16)[0])

    def b(bits):
        return float(torch.from_numpy(np.array([int(bits, 16)], dtype=np.uint16).view(np.int16)).view(torch.bfloat16).float()[0])

    f = g["fp16"]
    assert h(f["EX"]) == f["EX_value"] and h(f["SUB"]) == f["SUB_value"]
    assert h(f["MUL"]) == f["MUL_value"] and h(f["ADD"]) == f["ADD_value"]
    e = g["example"]
    assert h(e["or_bits"]) == e["or_value"] and e["or_value"] - e["minus"] == e["int_value"]
    assert abs(e["int_value"] * e["s"] - e["dequant"]) < 1e-12
    # every nibble n: (0x6400 | n) - 0x6408 == n - 8 and (1024 + 16n)/16 - 72 == n - 8
    for n in range(16):
        assert h(hex(0x6400 | n)) - h(f["SUB"]) == n - 8
        assert h(hex(0x6400 | (n << 4))) * h(f["MUL"]) + h(f["ADD"]) == n - 8
    bf = g["bf16"]
    assert b(bf["EX"]) == bf["EX_value"] and b(bf["MUL"]) == bf["MUL_value"] and b(bf["ADD"]) == bf["ADD_value"]
    for n in range(16):
        assert b(hex(0x4300 | n)) * b(bf["MUL"]) + b(bf["ADD"]) == n - 8


# --------------------------------------------------------------------------
# FP4 E2M1 / FP8 E4M3-FN (LLM quantization, "Floating point", "FP8")
# --------------------------------------------------------------------------

def pin_fp_formats():
    g = load_golden("fp_formats.json")
    assert oracle.e2m1_decode(np.arange(8)).tolist() == g["e2m1_magnitudes"]
    assert oracle.e2m1_decode(np.arange(8, 16)).tolist() == [-v for v in g["e2m1_magnitudes"]]
    mags = oracle.e4m3_finite_magnitudes()
    assert mags.max() == g["e4m3fn_max"] == 1.75 * 2 ** 8
    x, bits, val = g["e4m3_encode"][0]
    c = int(oracle.e4m3_encode(np.float32(x)))
    assert c == int(bits.replace(" ", ""), 2) and oracle.e4m3_decode(c) == val
    x, _, val = g["e4m3_encode"][1]
    assert oracle.e4m3_decode(oracle.e4m3_encode(np.float32(x))) == val
    for lo, hi, step in g["e4m3_spacing"]:
        inside = mags[(mags >= lo) & (mags <= hi)]
        assert np.all(np.diff(inside) == step)
    for x, v in g["e4m3_rounding_printed"]:
        assert oracle.e4m3_decode(oracle.e4m3_encode(np.float32(x))) == v


def test_fp_formats():
    pin_fp_formats()


def pin_e2m1_ties_even():
    mags = np.array(oracle.E2M1_MAGNITUDES)
    for c in range(7):
        mid = (mags[c] + mags[c + 1]) / 2
        even = c if c % 2 == 0 else c + 1
        for sign in (1, -1):
            code = int(oracle.e2m1_encode(np.float32(sign * mid)))
            assert code & 7 == even
            above = np.nextafter(np.float32(mid), np.float32(10))
            below = np.nextafter(np.float32(mid), np.float32(-10))
            assert int(oracle.e2m1_encode(sign * above)) & 7 == c + 1
            assert int(oracle.e2m1_encode(sign * below)) & 7 == c
    # saturation and signed zero
    assert int(oracle.e2m1_encode(np.float32(7.0))) == 7
    assert int(oracle.e2m1_encode(np.float32(1e30))) == 7
    assert int(oracle.e2m1_encode(np.float32(-1e30))) == 15
    assert int(oracle.e2m1_encode(np.float32(-0.1))) == 8
    assert int(oracle.e2m1_encode(np.float32(0.0))) == 0
    for c in range(16):
        assert int(oracle.e2m1_encode(np.float32(oracle.e2m1_decode(c) if c != 8 else -0.0))) == c


def test_e2m1_ties_even():
    pin_e2m1_ties_even()


def test_e4m3_against_torch():
    """Exhaustive decode and a dense encode sweep against torch's float8_e4m3fn."""
    torch = pytest.importorskip("torch")
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).float().numpy().astype(np.float64)
    assert np.array_equal(oracle.e4m3_decode(codes), ref)
    mags = oracle.e4m3_finite_magnitudes()
    mids = (mags[:-1] + mags[1:]) / 2
    pts = np.concatenate([mags, mids]).astype(np.float32)
    pts = np.concatenate([pts, np.nextafter(pts, np.float32(0)), np.nextafter(pts, np.float32(1e9))])
    rng = np.random.default_rng(5)
    pts = np.concatenate([pts, (rng.random(20000) * 460).astype(np.float32),
                          np.exp2(rng.uniform(-14, 9, 20000)).astype(np.float32)])
    pts = pts[(pts >= 0) & (pts < 448)]
    pts = np.concatenate([pts, -pts])
    tq = torch.from_numpy(pts).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(oracle.e4m3_encode(pts), tq)
    # saturation beyond 448 (the pages' 500 -> 448)
    assert np.all(oracle.e4m3_encode(np.array([449, 470, 480, 500, 1e6], dtype=np.float32)) == 0x7E)


# --------------------------------------------------------------------------
# NVFP4 (LLM quantization, "Block-scaled formats")
# --------------------------------------------------------------------------

def pin_nvfp4_block():
    g = load_golden("nvfp4_block.json")
    x = np.array(g["block"], dtype=np.float32)[None, :]
    q, sf = oracle.nvfp4_quantize(x, np.float32(1.0))
    assert int(sf[0, 0]) == int(g["block_scale_bits"].replace(" ", ""), 2)
    assert oracle.e4m3_decode(sf[0, 0]) == g["block_scale_e4m3"]
    assert oracle.e2m1_decode(q[0]).tolist() == g["codes_values"]
    deq = oracle.nvfp4_dequantize(q, sf, np.float32(1.0))
    assert abs(np.mean((deq - x) ** 2) - g["mse_printed"]) < 5e-5
    w = g["worst"]
    i = g["block"].index(w["x"])
    assert abs(x[0, i] / g["block_scale_e4m3"] - w["scaled_printed"]) < 5e-3
    assert oracle.e2m1_decode(q[0, i]) == w["value"]
    assert abs(deq[0, i] - w["dequant_printed"]) < 5e-3
    qs, ss = oracle.quant_sym_rows(x, 7)
    assert abs(np.mean((oracle.dequantize_affine(qs, ss[:, None], 0) - x) ** 2) - g["sym_int4_mse_printed"]) < 5e-5


def test_nvfp4_block():
    pin_nvfp4_block()


def test_nvfp4_global_scale_properties():
    rng = np.random.default_rng(21)
    x = rng.standard_normal((32, 256)).astype(np.float16).astype(np.float32)
    x[7, 100] = 37.0
    gsc = oracle.nvfp4_global_scale(x)
    assert gsc.dtype == np.float32
    q, sf = oracle.nvfp4_quantize(x, gsc)
    # the block holding the tensor's largest magnitude gets the top scale 448
    assert sf[7, 100 // 16] == 0x7E
    assert oracle.e2m1_decode(q[7, 100]) == 6.0
    # every block: |x| / d <= 6 up to rounding of the scale, elements within a half step of the grid
    deq = oracle.nvfp4_dequantize(q, sf, gsc)
    d = oracle.e4m3_decode(sf).repeat(16, axis=1) * float(gsc)
    assert np.all(np.abs(deq - x) <= d * 1.0 + 1e-12)
    # an all-zero block has scale code 0 and zero codes
    x2 = x.copy()
    x2[0, :16] = 0
    q2, sf2 = oracle.nvfp4_quantize(x2, gsc)
    assert sf2[0, 0] == 0 and not q2[0, :16].any()


def test_arc_perm_order_and_ties():
    x = np.array([[1, -5, 2, 5, 0], [-3, 1, 2, -1, 0]], dtype=np.float32)
    # column maxima of |x|: [3, 5, 2, 5, 0] -> 1, 3 (tie, lower index first), 0, 2, 4
    assert oracle.arc_perm(x).tolist() == [1, 3, 0, 2, 4]


def _arc_case(seed=3, t=24, k=128, n=20, s_res=32):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((t, k)).astype(np.float32)
    out = rng.choice(k, 6, replace=False)
    x[:, out] *= 50
    x = x.astype(np.float16).astype(np.float32)
    w = (rng.standard_normal((n, k)) * 0.02).astype(np.float32)
    return x, w, s_res


def test_arc_s0_is_plain_nvfp4():
    x, w, _ = _arc_case()
    perm = oracle.arc_perm(x)
    g = oracle.nvfp4_global_scale(x)
    qa, sfa = oracle.arc_quantize_activation(x, perm, 0, g)
    qb, sfb = oracle.nvfp4_quantize(x[:, perm], g)
    assert np.array_equal(qa, qb) and np.array_equal(sfa, sfb)


def test_arc_weight_columns_copied():
    x, w, s = _arc_case()
    perm = oracle.arc_perm(x)
    gw = oracle.nvfp4_global_scale(w)
    q, sf = oracle.arc_quantize_weight(w, perm, s, gw)
    k = w.shape[1]
    assert q.shape == (w.shape[0], k + s) and sf.shape == (w.shape[0], (k + s) // 16)
    assert np.array_equal(q[:, k:], q[:, :s]) and np.array_equal(sf[:, k // 16:], sf[:, : s // 16])


def pin_arc_residual_reduces_error():
    """Adding the re-quantized residual of the outlier channels must bring
    the augmented product closer to the exact X W^T than plain NVFP4 RTN."""
    x, w, s = _arc_case()
    perm = oracle.arc_perm(x)
    gx, gw = oracle.nvfp4_global_scale(x), oracle.nvfp4_global_scale(w)
    exact = x.astype(np.float64) @ w.astype(np.float64).T
    qa, sfa = oracle.arc_quantize_activation(x, perm, s, gx)
    qb, sfb = oracle.arc_quantize_weight(w, perm, s, gw)
    y_arc = oracle.nvfp4_gemm_reference(qa, sfa, gx, qb, sfb, gw)
    qa0, sfa0 = oracle.arc_quantize_activation(x, perm, 0, gx)
    qb0, sfb0 = oracle.arc_quantize_weight(w, perm, 0, gw)
    y_rtn = oracle.nvfp4_gemm_reference(qa0, sfa0, gx, qb0, sfb0, gw)
    e_arc = np.linalg.norm(y_arc - exact)
    e_rtn = np.linalg.norm(y_rtn - exact)
    assert e_arc < 0.9 * e_rtn
    # the main part plus the residual reproduces the outlier channels better
    main = oracle.nvfp4_dequantize(qa[:, : x.shape[1]], sfa[:, : x.shape[1] // 16], gx)[:, :s]
    res = oracle.nvfp4_dequantize(qa[:, x.shape[1]:], sfa[:, x.shape[1] // 16:], gx)
    xs = x[:, perm][:, :s]
    assert np.linalg.norm(main + res - xs) < 0.5 * np.linalg.norm(main - xs)


def test_arc_residual_reduces_error():
    pin_arc_residual_reduces_error()


def test_nvfp4_gemm_block_permutation_invariance():
    x, w, s = _arc_case()
    gx, gw = oracle.nvfp4_global_scale(x), oracle.nvfp4_global_scale(w)
    qa, sfa = oracle.nvfp4_quantize(x, gx)
    qb, sfb = oracle.nvfp4_quantize(w, gw)
    y = oracle.nvfp4_gemm_reference(qa, sfa, gx, qb, sfb, gw)
    nb = x.shape[1] // 16
    bp = np.random.default_rng(0).permutation(nb)
    cols = (bp[:, None] * 16 + np.arange(16)).reshape(-1)
    y2 = oracle.nvfp4_gemm_reference(qa[:, cols], sfa[:, bp], gx, qb[:, cols], sfb[:, bp], gw)
    assert np.allclose(y, y2, rtol=1e-12, atol=1e-12)


# --------------------------------------------------------------------------
# GEMMs: brute force on tiny inputs, the pages' W8A8 example, azp identity
# --------------------------------------------------------------------------

def pin_w8a8_example():
    g = load_golden("w8a8_example.json")
    xq = np.array(g["Xq"], dtype=np.int8)
    wq = np.array(g["Wq"], dtype=np.int8)
    d = oracle.int8_gemm_exact(xq, wq)
    assert d[0, 0] == g["D11_printed"]
    sx = np.array(g["scale_x_absmax"], dtype=np.float32) / F32(g["qmax"])
    sw = np.array(g["scale_w_absmax"], dtype=np.float32) / F32(g["qmax"])
    assert np.allclose(sx, g["scale_x_printed"], atol=5e-7) and np.allclose(sw, g["scale_w_printed"], atol=5e-7)
    y = oracle.w8a8_epilogue(d, sx, sw)
    assert np.max(np.abs(y - np.array(g["Y_printed"]))) < 1.5e-4
    assert 127 ** 2 == g["max_single_product_printed"]
    assert abs(4096 * 127 ** 2 - g["k4096_sum_bound_printed"]) / g["k4096_sum_bound_printed"] < 0.01
    # worst case of the int32 accumulator at K = 4096 (activation code -128)
    assert 4096 * 128 * 127 < 2 ** 31


def test_w8a8_example():
    pin_w8a8_example()


def _fr(v):
    return fractions.Fraction(float(v))


def pin_azp_identity():
    """s_a s_b (A^ B^^T - z (1 . B^)) + bias equals dequantize-then-multiply,
    exactly (rational arithmetic), for per-token and per-tensor zero-points."""
    rng = np.random.default_rng(7)
    for trial in range(4):
        t, k, n = 3, 5, 4
        a = rng.integers(-128, 128, size=(t, k)).astype(np.int8)
        b = rng.integers(-127, 128, size=(n, k)).astype(np.int8)
        sa = rng.uniform(0.01, 0.1, size=t).astype(np.float32)
        sb = rng.uniform(0.01, 0.1, size=n).astype(np.float32)
        bias = rng.standard_normal(n).astype(np.float16)
        per_token = trial % 2 == 0
        z = rng.integers(-128, 128, size=t).astype(np.int32) if per_token else np.full(t, int(rng.integers(-128, 128)), np.int32)
        adj = oracle.azp_adj_from_weight(b)
        d = oracle.int8_gemm_exact(a, b)
        if per_token:
            out = oracle.w8a8_epilogue(d, sa, sb, azp=z, azp_adj=adj, bias=bias)
        else:
            out = oracle.w8a8_epilogue(d, sa, sb, azp=None, azp_adj=int(z[0]) * adj, bias=bias)
        for i, j in itertools.product(range(t), range(n)):
            exact = sum(_fr(sa[i]) * (int(a[i, kk]) - int(z[i])) * _fr(sb[j]) * int(b[j, kk]) for kk in range(k)) + _fr(bias[j])
            assert abs(_fr(out[i, j]) - exact) <= abs(exact) * fractions.Fraction(1, 10 ** 12) + fractions.Fraction(1, 10 ** 15)


def test_azp_identity():
    pin_azp_identity()


def pin_w4a16_brute_force():
    rng = np.random.default_rng(9)
    t, n, k, group = 2, 3, 64, 32
    x = rng.standard_normal((t, k)).astype(np.float16)
    codes = rng.integers(0, 16, size=(n, k)).astype(np.uint8)
    scales = rng.uniform(0.005, 0.02, size=(n, k // group)).astype(np.float16)
    zeros = rng.integers(0, 16, size=(n, k // group)).astype(np.uint8)
    for zz in (zeros, None):
        y = oracle.w4a16_reference(x, codes, scales, zz, group)
        y2 = oracle.w4a16_reference_packed(x, oracle.pack_u4(codes), scales, None if zz is None else oracle.pack_u4(zz), group)
        assert np.array_equal(y, y2)
        for i in range(t):
            for j in range(n):
                acc = 0.0
                for kk in range(k):
                    zp = 8 if zz is None else int(zz[j, kk // group])
                    acc += float(x[i, kk]) * float(scales[j, kk // group]) * (int(codes[j, kk]) - zp)
                assert abs(y[i, j] - acc) <= 1e-12 * (1 + abs(acc))


def test_w4a16_brute_force():
    pin_w4a16_brute_force()


def pin_nvfp4_gemm_brute_force():
    rng = np.random.default_rng(10)
    t, n, k = 2, 3, 48
    qa = rng.integers(0, 16, size=(t, k)).astype(np.uint8)
    qb = rng.integers(0, 16, size=(n, k)).astype(np.uint8)
    sfa = rng.integers(0, 0x7E, size=(t, k // 16)).astype(np.uint8)
    sfb = rng.integers(0, 0x7E, size=(n, k // 16)).astype(np.uint8)
    ga, gb = np.float32(0.37), np.float32(1.7)
    y = oracle.nvfp4_gemm_reference(qa, sfa, ga, qb, sfb, gb)
    e2 = [0, 0.5, 1, 1.5, 2, 3, 4, 6]

    def val(c):
        return (-1 if c & 8 else 1) * e2[c & 7]

    def sc(c):
        e, m = (c >> 3) & 15, c & 7
        return (m / 8) * 2.0 ** -6 if e == 0 else (1 + m / 8) * 2.0 ** (e - 7)

    for i in range(t):
        for j in range(n):
            acc = 0.0
            for bb in range(k // 16):
                part = sum(val(int(qa[i, bb * 16 + u])) * val(int(qb[j, bb * 16 + u])) for u in range(16))
                acc += sc(int(sfa[i, bb])) * sc(int(sfb[j, bb])) * part
            acc *= float(ga) * float(gb)
            assert abs(y[i, j] - acc) <= 1e-12 * (1 + abs(acc))


def test_nvfp4_gemm_brute_force():
    pin_nvfp4_gemm_brute_force()


# --------------------------------------------------------------------------
# Planted mistakes: each must make at least one pin fail
# --------------------------------------------------------------------------


# ---- FP8 W8A8 (E4M3 per tensor / per token / per channel) ----

def _e4m3_value(code):
    """E4M3-FN value from the bit fields (S.EEEE.MMM, bias 7), written out here
    independently of the oracle's table."""
    code = int(code)
    sign = -1.0 if code & 0x80 else 1.0
    e, m = (code >> 3) & 0xF, code & 7
    return sign * ((m / 8.0) * 2.0 ** -6 if e == 0 else (1.0 + m / 8.0) * 2.0 ** (e - 7))


def pin_fp8_per_tensor_example():
    g = load_golden("fp8_w8a8_example.json")
    x = np.array(g["x"], dtype=np.float32)
    q, s = oracle.quant_fp8_tensor(x)
    dec = oracle.e4m3_decode(q)
    quot = x.astype(np.float64) / np.float64(s)
    # the printed quotients (two decimals) and their printed E4M3 roundings
    for printed, code in g["printed_roundings"]:
        i = int(np.argmin(np.abs(quot - printed)))
        assert abs(quot[i] - printed) <= 0.005, (quot[i], printed)
        assert dec[i] == code
    # every element within half of the printed spacing of its interval; the
    # largest magnitude lands on the E4M3 maximum
    for lo, hi, step in g["printed_spacing"]:
        inside = (np.abs(quot) >= lo) & (np.abs(quot) <= hi)
        assert np.all(np.abs(dec[inside] - quot[inside]) <= step / 2 + 1e-9)
    assert np.max(np.abs(dec)) == g["e4m3_max"]
    assert np.all(np.sign(dec) == np.sign(x))


def test_fp8_per_tensor_example():
    pin_fp8_per_tensor_example()


def pin_fp8_rows_properties():
    rng = np.random.default_rng(11)
    x = (rng.standard_normal((64, 256)) * np.exp(rng.uniform(-6, 6, size=(64, 1)))).astype(np.float32)
    x[3] = 0.0
    x[5, 7] = 300.0
    q, s = oracle.quant_fp8_rows(x)
    dec = oracle.e4m3_decode(q)
    assert s[3] == 1.0 and np.all(dec[3] == 0)
    nz = np.abs(x).max(axis=1) > 0
    assert np.all(np.abs(dec[nz]).max(axis=1) == 448.0)
    # three mantissa bits: at most 1/16 relative error in the normal range
    quot = np.abs(x.astype(np.float64) / s[:, None])
    normal = quot >= 2.0 ** -6
    err = np.abs(dec * s[:, None].astype(np.float64) - x)
    assert np.all(err[normal] <= np.abs(x[normal]) / 16 * (1 + 1e-6))
    for r in (0, 5, 40):
        q1, s1 = oracle.quant_fp8_tensor(x[r])
        assert s1 == s[r] and np.array_equal(q1, q[r])


def test_fp8_rows_properties():
    pin_fp8_rows_properties()


def pin_fp8_gemm_brute_force():
    rng = np.random.default_rng(12)
    T, N, K = 3, 4, 37
    qa = rng.integers(0, 256, size=(T, K)).astype(np.uint8)
    qb = rng.integers(0, 256, size=(N, K)).astype(np.uint8)
    qa[(qa & 0x7F) == 0x7F] = 0x10
    qb[(qb & 0x7F) == 0x7F] = 0x91
    sa = rng.uniform(0.01, 1.0, size=T).astype(np.float32)
    sb = rng.uniform(0.01, 1.0, size=N).astype(np.float32)
    bias = rng.standard_normal(N).astype(np.float32)
    y = oracle.fp8_gemm_reference(qa, sa, qb, sb, bias)
    for t in range(T):
        for n in range(N):
            acc = sum(_e4m3_value(qa[t, k]) * _e4m3_value(qb[n, k]) for k in range(K))
            want = acc * float(sa[t]) * float(sb[n]) + float(bias[n])
            assert abs(y[t, n] - want) <= 1e-12 * (1 + abs(want)), (t, n, y[t, n], want)


def test_fp8_gemm_brute_force():
    pin_fp8_gemm_brute_force()


# ---- RMSNorm fused with the per-token quantizers ----

def pin_rmsnorm_formula():
    rng = np.random.default_rng(13)
    for k, eps in ((4096, 1e-6), (4160, 1e-5), (16, 0.0), (8, 1e-3)):
        x = (rng.standard_normal((5, k)) * np.exp(rng.uniform(-4, 4, size=(5, 1)))).astype(np.float32)
        g = rng.uniform(0.25, 2.0, size=k).astype(np.float32)
        y = oracle.rmsnorm_rows(x, g, eps)
        x64 = x.astype(np.float64)
        ref = x64 / np.sqrt((x64 ** 2).mean(axis=1, keepdims=True) + eps) * g.astype(np.float64)
        # a handful of float32 roundings (the sum of squares is rounded once)
        tol = 8 * 2.0 ** -24
        assert np.all(np.abs(y - ref) <= tol * np.abs(ref) + 1e-30), k


def test_rmsnorm_formula():
    pin_rmsnorm_formula()


def test_rmsnorm_power_of_two_invariance():
    """With eps = 0, x and 2^j x normalize to the same bits (every step scales
    exactly), so the fused quantizers give the same codes."""
    rng = np.random.default_rng(14)
    x = rng.standard_normal((4, 1024)).astype(np.float32)
    g = rng.uniform(0.5, 1.5, size=1024).astype(np.float32)
    y = oracle.rmsnorm_rows(x, g, 0.0)
    for j in (-20, -3, 5, 30):
        assert np.array_equal(oracle.rmsnorm_rows(x * np.float32(2.0 ** j), g, 0.0), y)
    q1, s1 = oracle.rmsnorm_quant_int8(x, g, 0.0)
    q2, s2 = oracle.rmsnorm_quant_int8(x * np.float32(8.0), g, 0.0)
    assert np.array_equal(q1, q2) and np.array_equal(s1, s2)


def test_rmsnorm_constant_row():
    """A constant row 0.5 with gamma = 1 and eps = 0 normalizes to exactly 1
    (mean of squares 0.25, root 0.5, inverse 2): int8 codes 127 with s = 1/127,
    FP8 codes 448; a zero row with eps = 0 normalizes to 0 (codes 0, s = 1)."""
    x = np.full((2, 4096), 0.5, dtype=np.float32)
    x[1] = 0.0
    g = np.ones(4096, dtype=np.float32)
    y = oracle.rmsnorm_rows(x, g, 0.0)
    assert np.all(y[0] == 1.0) and np.all(y[1] == 0.0)
    q, s = oracle.rmsnorm_quant_int8(x, g, 0.0)
    assert np.all(q[0] == 127) and s[0] == np.float32(1.0) / np.float32(127.0) and np.all(q[1] == 0) and s[1] == 1.0
    c, sf = oracle.rmsnorm_quant_fp8(x, g, 0.0)
    assert np.all(oracle.e4m3_decode(c[0]) == 448.0) and np.all(oracle.e4m3_decode(c[1]) == 0.0)


def pin_sum_squares_exact():
    """The mean of squares starts from the exact sum of squares rounded once to
    float32 (nearest, ties to even).  Values worked out by hand:
    [1, 2^-12] sums to 1 + 2^-24, halfway between 1 and 1 + 2^-23, and rounds
    to the even 1; adding 2^-40 puts it above halfway, so it rounds up to
    1 + 2^-23 (a float32 sum from the left gives 1 in both cases); 3^2 + 4^2
    = 25; (2^-75)^2 = 2^-150 is half the smallest subnormal and rounds to 0,
    (1.5 . 2^-75)^2 = 1.125 . 2^-149 rounds to 2^-149; 2^64 squared is 2^128,
    past the float32 range: +inf; 2^63 twice gives 2^127."""
    rows = [([1.0, 2.0 ** -12], 1.0),
            ([1.0, 2.0 ** -12, 2.0 ** -40], 1.0 + 2.0 ** -23),
            ([3.0, 4.0], 25.0),
            ([2.0 ** -75], 0.0),
            ([1.5 * 2.0 ** -75], 2.0 ** -149),
            ([2.0 ** 64], np.inf),
            ([2.0 ** 63, 2.0 ** 63], 2.0 ** 127),
            ([0.0, -0.0], 0.0)]
    for vals, want in rows:
        x = np.zeros((1, 8), dtype=np.float32)
        x[0, :len(vals)] = vals
        got = oracle.sum_squares_f32(x)[0]
        assert got == np.float32(want), (vals, got, want)
        # the order of the elements does not matter
        assert oracle.sum_squares_f32(x[:, ::-1])[0] == got
    assert np.isnan(oracle.sum_squares_f32(np.array([[1.0, np.nan]], dtype=np.float32))[0])
    assert oracle.sum_squares_f32(np.array([[1.0, -np.inf]], dtype=np.float32))[0] == np.inf


def test_sum_squares_exact():
    pin_sum_squares_exact()


def test_sum_squares_against_fsum():
    """math.fsum returns the exact sum correctly rounded to float64 (Shewchuk's
    method); rounding that to float32 gives the same float32 unless the exact
    sum sits within 2^-53 of a float32 midpoint, which these rows do not.
    Any order of the rows' elements gives the same bits."""
    import math
    rng = np.random.default_rng(15)
    x = (rng.standard_normal((24, 4160)) * np.exp(rng.uniform(-8, 8, size=(24, 1)))).astype(np.float16)
    x = x.astype(np.float32)
    x[3, :7] = 3000.0
    got = oracle.sum_squares_f32(x)
    for i in range(x.shape[0]):
        assert got[i] == np.float32(math.fsum(float(v) * float(v) for v in x[i])), i
    perm = rng.permutation(x.shape[1])
    assert np.array_equal(oracle.sum_squares_f32(x[:, perm]), got)


def pin_rmsnorm_arc_unit_rms():
    """Rows of +-1 with eps = 0 have mean of squares exactly 1, so the RMSNorm
    output is x . gamma exactly; the fused NVFP4 quantizer must then equal the
    plain quantizer of the reordered values x[i, perm[j]] . gamma[perm[j]],
    built here element by element (gamma travels with its channel)."""
    rng = np.random.default_rng(16)
    rows, k, s_res = 6, 256, 32
    x = np.where(rng.random((rows, k)) < 0.5, -1.0, 1.0).astype(np.float32)
    gamma = rng.uniform(0.1, 4.0, size=k).astype(np.float32)
    perm = rng.permutation(k).astype(np.int32)
    ys = np.empty((rows, k), dtype=np.float32)
    for i in range(rows):
        for j in range(k):
            ys[i, j] = x[i, perm[j]] * gamma[perm[j]]
    g = np.float32(oracle.nvfp4_global_scale(ys))
    q, sf = oracle.rmsnorm_arc_quantize_activation(x, gamma, 0.0, perm, s_res, g)
    rq, rsf = oracle.arc_quantize_activation(ys, None, s_res, g)
    assert np.array_equal(q, rq) and np.array_equal(sf, rsf)


def test_rmsnorm_arc_unit_rms():
    pin_rmsnorm_arc_unit_rms()


# ---- W4A16 act-order (g_idx) ----

def _act_order_case(seed, n=6, k=512, t=3):
    rng = np.random.default_rng(seed)
    g = k // 128
    g_idx = rng.permutation(np.repeat(np.arange(g), 128))          # every group 128 columns, scattered
    codes = rng.integers(0, 16, size=(n, k)).astype(np.uint8)
    scales = rng.uniform(0.001, 0.02, size=(n, g)).astype(np.float16)
    zeros = rng.integers(0, 16, size=(n, g)).astype(np.uint8)
    x = rng.standard_normal((t, k)).astype(np.float16)
    return x, codes, scales, zeros, g_idx


def pin_act_order():
    x, codes, scales, zeros, g_idx = _act_order_case(31)
    y = oracle.w4a16_act_order_reference(x, codes, scales, zeros, g_idx)
    # contiguous groups: the plain g128 definition (pinned by brute force above)
    plain = np.arange(512) // 128
    assert np.allclose(oracle.w4a16_act_order_reference(x, codes, scales, zeros, plain),
                       oracle.w4a16_reference(x, codes, scales, zeros), rtol=0, atol=1e-12)
    # brute force, one column at a time
    t, n = 1, 4
    want = sum(float(x[t, k]) * (int(codes[n, k]) - int(zeros[n, g_idx[k]])) * float(scales[n, g_idx[k]])
               for k in range(512))
    assert abs(y[t, n] - want) <= 1e-12 * (1 + abs(want))
    # sorting the columns by group (the same permutation on x, the codes and
    # g_idx) leaves Y unchanged and makes the groups contiguous
    perm = oracle.act_order_perm(g_idx)
    assert np.array_equal(g_idx[perm], plain)
    assert np.all(np.diff(perm[g_idx[perm] == 2]) > 0)                 # stable inside a group
    y2 = oracle.w4a16_reference(x[:, perm], codes[:, perm], scales, zeros)
    assert np.allclose(y, y2, rtol=1e-12, atol=1e-12)


def test_act_order():
    pin_act_order()


def test_act_order_perm_rejects_uneven_groups():
    g_idx = np.repeat(np.arange(4), 128)
    g_idx[0] = 1
    with pytest.raises(ValueError):
        oracle.act_order_perm(g_idx)


# ---- online Hadamard rotation ----

def _sylvester_by_formula(n):
    """H_n written out from its element formula: (-1)^popcount(i & j)."""
    i = np.arange(n)
    return np.array([[(-1.0) ** bin(a & b).count("1") for b in i] for a in i])


def _regular_by_formula(n):
    """The Kronecker power of H4 element by element: the product over the
    base-4 digits (i_d, j_d) of the indices of H4[i_d][j_d]."""
    h4 = [[1, 1, 1, -1], [1, 1, -1, 1], [1, -1, 1, 1], [-1, 1, 1, 1]]
    out = np.ones((n, n))
    for a in range(n):
        for b in range(n):
            v, i, j = 1, a, b
            while i or j:            # leading digit pairs (0, 0) contribute H4[0][0] = 1
                v *= h4[i % 4][j % 4]
                i //= 4
                j //= 4
            out[a, b] = v
    return out


def pin_hadamard_page_examples():
    g = load_golden("hadamard_examples.json")
    ex = g["sylvester_h8"]
    xh = oracle.hadamard_rotate(np.array([ex["x"]]), 8, "sylvester")[0]
    wh = oracle.hadamard_rotate(np.array([ex["w"]]), 8, "sylvester")[0]
    assert np.all(np.abs(xh - ex["xH_printed"]) <= 1e-3)
    assert np.all(np.abs(wh - ex["wH_printed"]) <= 1e-3)
    # orthogonal: the dot product is unchanged
    assert abs(float(xh @ wh) - ex["dot_printed"]) <= 5e-4
    assert abs(float(np.dot(ex["x"], ex["w"])) - ex["dot_printed"]) <= 5e-4
    r = g["regular_h4"]
    y = oracle.hadamard_rotate(np.array([r["x"]]), 4, "regular")[0]
    assert abs(y[0] - r["y0_printed"]) <= 1e-12
    assert abs(y[0] - float(np.dot(r["x"], r["first_column"])) / 2.0) <= 1e-12


def test_hadamard_page_examples():
    pin_hadamard_page_examples()


def pin_hadamard_dense():
    """Every group times the matrix built from its element formula, over sqrt(n),
    to float64 rounding; the signs multiply the rotated columns."""
    rng = np.random.default_rng(41)
    for kind, sizes in (("sylvester", (2, 8, 64, 256)), ("regular", (4, 16, 64))):
        for n in sizes:
            x = rng.standard_normal((3, 2 * n))
            h = _sylvester_by_formula(n) if kind == "sylvester" else _regular_by_formula(n)
            ref = (x.reshape(-1, n) @ h / np.sqrt(n)).reshape(x.shape)
            y = oracle.hadamard_rotate(x, n, kind)
            assert np.max(np.abs(y - ref)) <= 1e-12 * np.sqrt(n) * np.abs(x).max(), (kind, n)
            signs = np.where(rng.random(2 * n) < 0.5, -1.0, 1.0)
            assert np.array_equal(oracle.hadamard_rotate(x, n, kind, signs), y * signs)


def test_hadamard_dense():
    pin_hadamard_dense()


def test_hadamard_matrices():
    """The doubling equals the element formula; both matrices are symmetric and
    orthogonal; the regular one has every column sum +-sqrt(n), so a row of
    ones rotates to +-1 ("every channel is +-c")."""
    assert np.array_equal(oracle.sylvester_matrix(32), _sylvester_by_formula(32))
    assert np.array_equal(oracle.regular_matrix(64), _regular_by_formula(64))
    for n in (4, 16, 64, 256):
        h = oracle.regular_matrix(n)
        assert np.array_equal(h @ h.T, n * np.eye(n)) and np.array_equal(h, h.T)
        assert np.array_equal(np.abs(h.sum(axis=0)), np.full(n, np.sqrt(n)))
        y = oracle.hadamard_rotate(np.ones((1, n)), n, "regular")
        assert np.allclose(np.abs(y), 1.0, rtol=0, atol=1e-12)
    h = oracle.sylvester_matrix(256)
    assert np.array_equal(h @ h.T, 256 * np.eye(256))
    # Sylvester: the first column sums to n, the others to 0 (a constant row
    # lands entirely in the first channel)
    y = oracle.hadamard_rotate(np.full((1, 16), 3.0), 16, "sylvester")[0]
    assert abs(y[0] - 12.0) <= 1e-12 and np.all(np.abs(y[1:]) <= 1e-12)


def test_hadamard_involution_and_doubling():
    rng = np.random.default_rng(42)
    x = rng.standard_normal((4, 8192))
    for kind, n in (("sylvester", 8192), ("sylvester", 128), ("regular", 256)):
        y = oracle.hadamard_rotate(oracle.hadamard_rotate(x, n, kind), n, kind)
        assert np.max(np.abs(y - x)) <= 1e-11 * np.abs(x).max()


def test_hadamard_doubling_step_equals_dense(monkeypatch):
    """The one doubling step used above 4096 x 4096, checked at a small order
    by lowering the dense limit: the result equals the dense product."""
    rng = np.random.default_rng(43)
    x = rng.standard_normal((3, 128))
    dense = oracle.hadamard_rotate(x, 64, "sylvester")
    monkeypatch.setattr(oquant_had, "_DENSE_MAX", 8)
    assert np.allclose(oracle.hadamard_rotate(x, 64, "sylvester"), dense, rtol=0, atol=1e-12)


# ---- MX block-scaled formats (MXFP8, MXFP4) ----

def _pad32(v):
    x = np.zeros((1, 32), dtype=np.float32)
    x[0, :len(v)] = np.asarray(v, dtype=np.float32)
    return x


def pin_mx_page_examples():
    g = load_golden("mx_examples.json")
    assert oracle.MX_EMAX["e4m3"] == g["emax"]["e4m3"] and oracle.MX_EMAX["e2m1"] == g["emax"]["e2m1"]
    # MXFP4: scale 2^(floor(log2 2.4) - 2) = 0.5; 2.4 / 0.5 = 4.8 -> 4 -> 2.0, error 0.4
    x = _pad32(g["mxfp4_block"])
    q, sf = oracle.mx_quantize(x, "e2m1")
    assert oracle.e8m0_decode(sf)[0, 0] == g["mxfp4_scale_printed"]
    deq = oracle.mx_dequantize(q, sf, "e2m1")[0]
    i = int(np.argmax(np.abs(x[0])))
    m = g["mxfp4_max"]
    assert x[0, i] == np.float32(m["x"]) and oracle.e2m1_decode(q[0, i]) == m["value"]
    assert deq[i] == m["dequant_printed"] and abs(abs(deq[i] - x[0, i]) - m["error_printed"]) < 1e-6
    # MXFP8 of the eight weights: the printed MSE (three significant digits)
    w = _pad32(g["mxfp8_weights"])
    q8, sf8 = oracle.mx_quantize(w, "e4m3")
    err = oracle.mx_dequantize(q8, sf8, "e4m3")[0, :8] - w[0, :8].astype(np.float64)
    assert abs(np.mean(err ** 2) - g["mxfp8_mse_printed"]) <= 0.005e-3


def test_mx_page_examples():
    pin_mx_page_examples()


def test_mx_scaled_max_range():
    """The block maximum over its scale lies in [2^e_max, 2^(e_max+1)) wherever
    the exponent is not clamped; the scale is a power of two; every element's
    code is the nearest value of the element format to x / scale."""
    rng = np.random.default_rng(21)
    x = (rng.standard_normal((6, 256)) * np.exp(rng.uniform(-20, 20, size=(6, 1)))).astype(np.float32)
    for fmt, top in (("e4m3", 448.0), ("e2m1", 6.0)):
        q, sf = oracle.mx_quantize(x, fmt)
        scale = oracle.e8m0_decode(sf)
        amax = np.abs(x.reshape(6, 8, 32)).max(axis=2).astype(np.float64)
        r = amax / scale
        emax = oracle.MX_EMAX[fmt]
        assert np.all((r >= 2.0 ** emax) & (r < 2.0 ** (emax + 1)))
        dec = oracle.e4m3_decode(q) if fmt == "e4m3" else oracle.e2m1_decode(q)
        y = x.astype(np.float64) / np.repeat(scale, 32, axis=1)
        table = oracle.e4m3_finite_magnitudes() if fmt == "e4m3" else np.array([0, .5, 1, 1.5, 2, 3, 4, 6.])
        best = np.abs(np.abs(np.minimum(np.abs(y), top))[..., None] - table).min(axis=-1)
        assert np.all(np.abs(np.abs(dec) - np.minimum(np.abs(y), top)) == best)


def test_mx_power_of_two_invariance_and_edges():
    rng = np.random.default_rng(22)
    x = rng.standard_normal((3, 64)).astype(np.float32)
    for fmt in ("e4m3", "e2m1"):
        q, sf = oracle.mx_quantize(x, fmt)
        for j in (-30, -1, 7, 40):
            q2, sf2 = oracle.mx_quantize(x * np.float32(2.0 ** j), fmt)
            assert np.array_equal(q2, q) and np.array_equal(sf2.astype(int), sf.astype(int) + j)
        z = np.zeros((1, 32), dtype=np.float32)
        qz, sfz = oracle.mx_quantize(z, fmt)
        assert sfz[0, 0] == 0 and not np.any(qz)
        big = np.full((1, 32), 3.0e38, dtype=np.float32)             # floor(log2) = 127: unclamped
        _, sfb = oracle.mx_quantize(big, fmt)
        assert int(sfb[0, 0]) == 127 + 127 - oracle.MX_EMAX[fmt]
        tiny = np.full((1, 32), 1e-45, dtype=np.float32)             # subnormal: exponent clamped to -127
        _, sft = oracle.mx_quantize(tiny, fmt)
        assert sft[0, 0] == 0


def pin_mx_gemm_brute_force():
    rng = np.random.default_rng(23)
    T, N, K = 2, 3, 64
    e2m1 = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    for fmt in ("e4m3", "e2m1"):
        hi = 256 if fmt == "e4m3" else 16
        qa = rng.integers(0, hi, size=(T, K)).astype(np.uint8)
        qb = rng.integers(0, hi, size=(N, K)).astype(np.uint8)
        if fmt == "e4m3":
            qa[(qa & 0x7F) == 0x7F] = 0x21
            qb[(qb & 0x7F) == 0x7F] = 0xA2
        sfa = rng.integers(100, 150, size=(T, K // 32)).astype(np.uint8)
        sfb = rng.integers(100, 150, size=(N, K // 32)).astype(np.uint8)
        y = oracle.mx_gemm_reference(qa, sfa, qb, sfb, fmt)

        def val(code):
            if fmt == "e4m3":
                return _e4m3_value(code)
            return (-1.0 if code & 8 else 1.0) * e2m1[code & 7]

        for t in range(T):
            for n in range(N):
                want = sum(val(qa[t, k]) * 2.0 ** (int(sfa[t, k // 32]) - 127) *
                           val(qb[n, k]) * 2.0 ** (int(sfb[n, k // 32]) - 127) for k in range(K))
                assert abs(y[t, n] - want) <= 1e-12 * (1 + abs(want)), (fmt, t, n)


def test_mx_gemm_brute_force():
    pin_mx_gemm_brute_force()


def _mut_e2m1_ties_odd(monkeypatch):
    orig = ofmt._nearest_code

    def bad(mag, table):
        idx = orig(mag, table)
        mids = (table[:-1] + table[1:]) / 2
        on = np.isin(np.asarray(mag, dtype=np.float64), mids)
        return np.where(on & (idx % 2 == 0), np.maximum(idx - 1, 0), idx)

    monkeypatch.setattr(ofmt, "_nearest_code", bad)
    return pin_e2m1_ties_even


def _mut_azp_sign(monkeypatch):
    orig = ogemm.w8a8_epilogue

    def bad(dhat, sa, sb, azp=None, azp_adj=None, bias=None):
        return orig(dhat, sa, sb, None if azp is None else -np.asarray(azp), None if azp_adj is None else (-np.asarray(azp_adj) if azp is None else azp_adj), bias)

    monkeypatch.setattr(oracle, "w8a8_epilogue", bad)
    return pin_azp_identity


def _mut_azp_adj_axis(monkeypatch):
    def bad(b):
        b = np.asarray(b, dtype=np.int64)
        return np.resize(b.sum(axis=0), b.shape[0]).astype(np.int32)

    monkeypatch.setattr(oracle, "azp_adj_from_weight", bad)
    return pin_azp_identity


def _mut_residual_sign(monkeypatch):
    orig = oquant.nvfp4_quantize
    calls = {"n": 0}

    def bad(x, g):
        calls["n"] += 1
        q, sf = orig(x, g)
        return (q ^ 8, sf) if calls["n"] % 2 == 0 else (q, sf)

    monkeypatch.setattr(oquant, "nvfp4_quantize", bad)
    return pin_arc_residual_reduces_error


def _mut_w8a8_transposed(monkeypatch):
    monkeypatch.setattr(oracle, "int8_gemm_exact", lambda a, b: ogemm.int8_gemm_exact(a, b[:, ::-1]))
    return pin_w8a8_example


def _mut_w4_zero_dropped(monkeypatch):
    orig = ogemm.w4a16_reference
    monkeypatch.setattr(oracle, "w4a16_reference", lambda x, c, s, z, g=128: orig(x, c, s, None, g))
    return pin_w4a16_brute_force


def _mut_nvfp4_scale_not_decoded(monkeypatch):
    monkeypatch.setattr(oquant, "_block_divisor", lambda sf, g: (sf.astype(np.float32) * np.float32(g)).astype(np.float32))
    return pin_nvfp4_block


def _mut_sym_qmax(monkeypatch):
    orig = oquant.quant_sym_rows
    monkeypatch.setattr(oracle, "quant_sym_rows", lambda x, qmax: orig(x, qmax + 1))
    return pin_granularity


def _mut_fp8_scale_447(monkeypatch):
    def bad(x):
        x = np.asarray(x, dtype=np.float32)
        a = np.abs(x).max()
        s = np.float32(1.0) if a == 0 else np.float32(a / np.float32(447.0))
        return oracle.e4m3_encode(x / s), s

    monkeypatch.setattr(oracle, "quant_fp8_tensor", bad)
    return pin_fp8_per_tensor_example


def _mut_fp8_scales_swapped(monkeypatch):
    orig = ogemm.fp8_gemm_reference
    monkeypatch.setattr(oracle, "fp8_gemm_reference",
                        lambda qa, sa, qb, sb, bias=None: orig(qa, np.resize(sb, sa.shape), qb, np.resize(sa, sb.shape), bias))
    return pin_fp8_gemm_brute_force


def _mut_rmsnorm_mean_k_minus_1(monkeypatch):
    def bad(x, gamma, eps):
        x = np.asarray(x, dtype=np.float32)
        k = x.shape[1]
        ms = ((x * x).sum(axis=1, dtype=np.float32) / np.float32(k - 1)).astype(np.float32)
        inv = (np.float32(1.0) / np.sqrt(ms + np.float32(eps))).astype(np.float32)
        return ((x * inv[:, None]) * np.asarray(gamma, dtype=np.float32)).astype(np.float32)

    monkeypatch.setattr(oracle, "rmsnorm_rows", bad)
    return pin_rmsnorm_formula


def _mut_rmsnorm_arc_gamma_reordered(monkeypatch):
    def bad(x, gamma, eps, perm, s_res, g):
        y = oquant.rmsnorm_rows(x, np.ones_like(gamma), eps)[:, perm] * np.asarray(gamma, dtype=np.float32)
        return oquant.arc_quantize_activation(y.astype(np.float32), None, s_res, g)

    monkeypatch.setattr(oracle, "rmsnorm_arc_quantize_activation", bad)
    return pin_rmsnorm_arc_unit_rms


def _mut_act_order_ignores_g_idx(monkeypatch):
    monkeypatch.setattr(oracle, "w4a16_act_order_reference",
                        lambda x, c, s, z, g_idx, group=128: ogemm.w4a16_reference(x, c, s, z, group))
    return pin_act_order


def _mut_hadamard_outputs_swapped(monkeypatch):
    orig = oquant_had._rotate_groups

    def bad(g, n, kind):
        y = orig(g, n, kind)
        return np.concatenate([y[:, 1:2], y[:, :1], y[:, 2:]], axis=1)   # two outputs swapped
    monkeypatch.setattr(oquant_had, "_rotate_groups", bad)
    return pin_hadamard_dense


def _mut_asym_add_then_round(monkeypatch):
    def bad(x):
        x = np.asarray(x, dtype=np.float32)
        mn = np.minimum(x.min(axis=1), F32(0.0))
        mx = np.maximum(x.max(axis=1), F32(0.0))
        s = (np.maximum(mx - mn, F32(1e-5)) / F32(255.0)).astype(np.float32)
        z = (-128 - np.rint(mn / s).astype(np.int64)).astype(np.int32)
        q = np.clip(np.rint((x / s[:, None]).astype(np.float64) + z[:, None]), -128, 127).astype(np.int8)
        return q, s, z

    monkeypatch.setattr(oracle, "quant_int8_asym", bad)
    return pin_zero_point_added_after_rounding


def _mut_w4_add_then_round(monkeypatch):
    def bad(w, group=128):
        w = np.asarray(w, dtype=np.float32)
        n, k = w.shape
        g = w.reshape(n, k // group, group)
        s16 = (np.maximum(g.max(axis=2) - g.min(axis=2), F32(1e-5)) / F32(15.0)).astype(np.float16)
        s = s16.astype(np.float32)
        z = np.clip(np.rint(-g.min(axis=2) / s), 0, 15)
        q = np.clip(np.rint((g / s[:, :, None]).astype(np.float64) + z[:, :, None]), 0, 15)
        return q.reshape(n, k).astype(np.uint8), s16, z.astype(np.uint8)

    monkeypatch.setattr(oracle, "quant_w4_g128", bad)
    return pin_zero_point_added_after_rounding


def _mut_sum_squares_float32_left_to_right(monkeypatch):
    def bad(x):
        x = np.asarray(x, dtype=np.float32)
        out = np.zeros(x.shape[0], dtype=np.float32)
        for j in range(x.shape[1]):
            with np.errstate(over="ignore", invalid="ignore"):
                out = (out + (x[:, j] * x[:, j]).astype(np.float32)).astype(np.float32)
        return out

    monkeypatch.setattr(oracle, "sum_squares_f32", bad)
    return pin_sum_squares_exact


def _mut_mx_emax_e4m3_7(monkeypatch):
    monkeypatch.setitem(oquant_mx.MX_EMAX, "e4m3", 7)
    return pin_mx_page_examples


def _mut_mx_scales_swapped(monkeypatch):
    orig = oquant_mx.mx_gemm_reference
    monkeypatch.setattr(oracle, "mx_gemm_reference",
                        lambda qa, sfa, qb, sfb, fmt: orig(qa, np.resize(sfb, sfa.shape), qb, np.resize(sfa, sfb.shape), fmt))
    return pin_mx_gemm_brute_force


MUTATIONS = [_mut_e2m1_ties_odd, _mut_azp_sign, _mut_azp_adj_axis, _mut_residual_sign,
             _mut_w8a8_transposed, _mut_w4_zero_dropped, _mut_nvfp4_scale_not_decoded, _mut_sym_qmax,
             _mut_fp8_scale_447, _mut_fp8_scales_swapped, _mut_rmsnorm_mean_k_minus_1,
             _mut_rmsnorm_arc_gamma_reordered, _mut_mx_emax_e4m3_7, _mut_mx_scales_swapped,
             _mut_act_order_ignores_g_idx, _mut_hadamard_outputs_swapped,
             _mut_asym_add_then_round, _mut_w4_add_then_round, _mut_sum_squares_float32_left_to_right]


@pytest.mark.parametrize("mutation", MUTATIONS, ids=[m.__name__ for m in MUTATIONS])
def test_planted_mistake_is_caught(monkeypatch, mutation):
    pin = mutation(monkeypatch)
    with pytest.raises(AssertionError):
        pin()
