"""W8A8 on the GPU against the CPU oracle: the int32 accumulator bit for bit
(including adversarial extremes that bring each exact fp32 chunk to its
2^24 bound), the four fused epilogues within the bf16/fp16 tolerance, and
the two full-size workloads through the device quantizers.  Every GEMM test
runs with the weights as int8 codes (qlin_w8a8_gemm), as the same codes in
fp16 (qlin_int8_to_f16 + qlin_w8a8_gemm_f16b), and with both operands' codes
in fp16 (qlin_w8a8_gemm_f16; on the full-size workloads the activation codes
come from qlin_quant_act_int8_f16)."""

import numpy as np
import pytest
import torch

import oracle
from quantized_linear_layer_gb300 import inputs
from conftest import assert_within_tolerance

pytestmark = pytest.mark.gpu


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


BFORMS = ["i8", "f16", "f16ab"]


def _f16(q, codes):
    c16 = torch.empty(codes.shape, dtype=torch.float16, device="cuda")
    q.qlin_int8_to_f16(codes, c16)
    return c16


def _gemm(q, bform, a, b, sa, sb, out, a16=None, **kw):
    """qlin_w8a8_gemm on int8 codes; qlin_w8a8_gemm_f16b on the weights'
    exact fp16 copy (qlin_int8_to_f16); or qlin_w8a8_gemm_f16 on fp16 copies
    of both (a16: the activation codes already in fp16, e.g. from
    qlin_quant_act_int8_f16)."""
    if bform == "i8":
        q.qlin_w8a8_gemm(a, b, sa, sb, out, **kw)
    elif bform == "f16":
        q.qlin_w8a8_gemm_f16b(a, _f16(q, b), sa, sb, out, **kw)
    else:
        q.qlin_w8a8_gemm_f16(_f16(q, a) if a16 is None else a16, _f16(q, b), sa, sb, out, **kw)


def _raw(q, a, b, bform="i8"):
    out = torch.empty((a.shape[0], b.shape[0]), dtype=torch.int32, device="cuda")
    _gemm(q, bform, _dev(a), _dev(b), None, None, out)
    torch.cuda.synchronize()
    assert q.qlin_get_device_error() == 0
    return out.cpu().numpy()


def test_int8_to_f16_exact(qlin_gpu):
    """Every code, in a count that is not a multiple of 16."""
    src = np.tile(np.arange(-128, 128, dtype=np.int16).astype(np.int8), 5)[:1277]
    dst = torch.empty(src.shape, dtype=torch.float16, device="cuda")
    qlin_gpu.qlin_int8_to_f16(_dev(src), dst)
    torch.cuda.synchronize()
    assert np.array_equal(dst.cpu().numpy().astype(np.float64), src.astype(np.float64))


@pytest.mark.parametrize("bform", BFORMS)
@pytest.mark.parametrize("T,N,K", [(128, 128, 64), (200, 136, 1040), (1, 8, 16), (130, 264, 2064),
                                   (257, 384, 4096), (64, 1000, 3072)])
def test_accumulator_bit_exact(qlin_gpu, T, N, K, bform):
    rng = np.random.default_rng(T * 7 + N + K)
    a = rng.integers(-128, 128, size=(T, K), dtype=np.int8)
    b = rng.integers(-127, 128, size=(N, K), dtype=np.int8)
    assert np.array_equal(_raw(qlin_gpu, a, b, bform), oracle.int8_gemm_exact(a, b))


@pytest.mark.parametrize("bform", BFORMS)
@pytest.mark.parametrize("K", [1024, 2048, 4096, 5120])
def test_accumulator_extremes(qlin_gpu, K, bform):
    """All-extreme codes drive every 1024-wide fp32 chunk to +-1024*128*127."""
    T, N = 128, 128
    a = np.full((T, K), -128, dtype=np.int8)
    a[1::2] = 127
    a[2] = -127
    b = np.full((N, K), 127, dtype=np.int8)
    b[1::2] = -127
    b[5] = -128
    b[7, ::3] = 0
    got = _raw(qlin_gpu, a, b, bform)
    ref = oracle.int8_gemm_exact(a, b)
    assert np.array_equal(got, ref)
    assert np.abs(ref).max() >= (K // 1024) * 1024 * 127 * 127


def _epilogue_case(rng, T, N, K):
    x = rng.standard_normal((T, K)).astype(np.float32)
    w = (rng.standard_normal((N, K)) * 0.02).astype(np.float32)
    return x, w


@pytest.mark.parametrize("bform", BFORMS)
@pytest.mark.parametrize("form", ["scaled", "bias", "azp_tensor", "azp_token", "azp_token_nobias", "scalar_scales"])
@pytest.mark.parametrize("out_dtype", ["bf16", "f16"])
def test_epilogues(qlin_gpu, form, out_dtype, bform):
    rng = np.random.default_rng(5)
    T, N, K = 193, 264, 1552
    x, w = _epilogue_case(rng, T, N, K)
    bq, sb = oracle.quant_int8_sym(w)
    adj = oracle.azp_adj_from_weight(bq)
    bias = (rng.standard_normal(N) * 0.1).astype(np.float16)
    if form in ("azp_tensor", "azp_token", "azp_token_nobias"):
        aq, sa, za = oracle.quant_int8_asym(x + 1.0)
    else:
        aq, sa = oracle.quant_int8_sym(x)
        za = None
    d = oracle.int8_gemm_exact(aq, bq)
    kw = {}
    if form == "scaled":
        ref = oracle.w8a8_epilogue(d, sa, sb)
    elif form == "bias":
        ref = oracle.w8a8_epilogue(d, sa, sb, bias=bias)
        kw = dict(bias=_dev(bias))
    elif form == "azp_tensor":
        z = int(za[0])
        aq = np.clip(np.rint((x + 1.0) / sa[0]) + z, -128, 127).astype(np.int8)   # one zero-point for all rows
        d = oracle.int8_gemm_exact(aq, bq)
        sa = np.full(1, sa[0], dtype=np.float32)
        ref = oracle.w8a8_epilogue(d, sa, sb, azp=None, azp_adj=z * adj.astype(np.int64), bias=bias)
        kw = dict(azp_adj=_dev((z * adj.astype(np.int64)).astype(np.int32)), bias=_dev(bias))
    elif form == "azp_token":
        ref = oracle.w8a8_epilogue(d, sa, sb, azp=za, azp_adj=adj, bias=bias)
        kw = dict(azp=_dev(za), azp_adj=_dev(adj), bias=_dev(bias))
    elif form == "azp_token_nobias":
        ref = oracle.w8a8_epilogue(d, sa, sb, azp=za, azp_adj=adj)
        kw = dict(azp=_dev(za), azp_adj=_dev(adj))
    else:
        sa = np.full(1, sa.max(), dtype=np.float32)
        sb = np.full(1, sb.max(), dtype=np.float32)
        ref = oracle.w8a8_epilogue(d, sa, sb)
    tdt = torch.bfloat16 if out_dtype == "bf16" else torch.float16
    out = torch.empty((T, N), dtype=tdt, device="cuda")
    _gemm(qlin_gpu, bform, _dev(aq), _dev(bq), _dev(sa), _dev(sb), out, **kw)
    torch.cuda.synchronize()
    assert qlin_gpu.qlin_get_device_error() == 0
    assert_within_tolerance(out.float().cpu().numpy(), ref, "W8A8 %s %s %s" % (form, out_dtype, bform))


def _device_quant(q, x_np, asym):
    xt = _dev(x_np)
    t, k = x_np.shape
    aq = torch.empty((t, k), dtype=torch.int8, device="cuda")
    sa = torch.empty(t, dtype=torch.float32, device="cuda")
    za = torch.empty(t, dtype=torch.int32, device="cuda") if asym else None
    q.qlin_quant_act_int8(xt, aq, sa, za)
    return aq, sa, za


def _device_quant_f16(q, x_np, asym, aq, sa, za):
    """qlin_quant_act_int8_f16 on the same rows: its codes, scales and
    zero-points must equal qlin_quant_act_int8's exactly."""
    xt = _dev(x_np)
    t, k = x_np.shape
    a16 = torch.empty((t, k), dtype=torch.float16, device="cuda")
    sa16 = torch.empty(t, dtype=torch.float32, device="cuda")
    za16 = torch.empty(t, dtype=torch.int32, device="cuda") if asym else None
    q.qlin_quant_act_int8_f16(xt, a16, sa16, za16)
    torch.cuda.synchronize()
    assert torch.equal(a16.float(), aq.float())
    assert torch.equal(sa16, sa)
    if asym:
        assert torch.equal(za16, za)
    return a16


@pytest.mark.parametrize("bform", BFORMS)
def test_config3_symmetric_bias_bf16(qlin_gpu, bform):
    d = inputs.w8a8_sym_bias(seed=2)
    x32 = d["x"].astype(np.float32)
    aq, sa, _ = _device_quant(qlin_gpu, d["x"], asym=False)
    bq, sb, _ = _device_quant(qlin_gpu, d["w"], asym=False)
    a16 = _device_quant_f16(qlin_gpu, d["x"], False, aq, sa, None) if bform == "f16ab" else None
    raq, rsa = oracle.quant_int8_sym(x32)
    rbq, rsb = oracle.quant_int8_sym(d["w"])
    assert np.array_equal(aq.cpu().numpy(), raq) and np.array_equal(bq.cpu().numpy(), rbq)
    dh = oracle.int8_gemm_exact(raq, rbq)
    raw = torch.empty((2048, 4096), dtype=torch.int32, device="cuda")
    _gemm(qlin_gpu, bform, aq, bq, None, None, raw, a16=a16)
    assert np.array_equal(raw.cpu().numpy(), dh)
    out = torch.empty((2048, 4096), dtype=torch.bfloat16, device="cuda")
    _gemm(qlin_gpu, bform, aq, bq, sa, sb, out, a16=a16, bias=_dev(d["bias"]))
    torch.cuda.synchronize()
    assert qlin_gpu.qlin_get_device_error() == 0
    ref = oracle.w8a8_epilogue(dh, rsa, rsb, bias=d["bias"])
    assert_within_tolerance(out.float().cpu().numpy(), ref, "config 3")


@pytest.mark.parametrize("bform", BFORMS)
def test_config4_azp_per_token_f16(qlin_gpu, bform):
    d = inputs.w8a8_azp_token(seed=3)
    x32 = d["x"].astype(np.float32)
    aq, sa, za = _device_quant(qlin_gpu, d["x"], asym=True)
    bq, sb, _ = _device_quant(qlin_gpu, d["w"], asym=False)
    a16 = _device_quant_f16(qlin_gpu, d["x"], True, aq, sa, za) if bform == "f16ab" else None
    adj = torch.empty(d["w"].shape[0], dtype=torch.int32, device="cuda")
    qlin_gpu.qlin_int8_row_sum(bq, adj)
    raq, rsa, rza = oracle.quant_int8_asym(x32)
    rbq, rsb = oracle.quant_int8_sym(d["w"])
    assert np.array_equal(aq.cpu().numpy(), raq) and np.array_equal(za.cpu().numpy(), rza)
    assert np.array_equal(bq.cpu().numpy(), rbq)
    radj = oracle.azp_adj_from_weight(rbq)
    assert np.array_equal(adj.cpu().numpy(), radj)
    dh = oracle.int8_gemm_exact(raq, rbq)
    for bias in (d["bias"], None):
        out = torch.empty((4096, 14336), dtype=torch.float16, device="cuda")
        _gemm(qlin_gpu, bform, aq, bq, sa, sb, out, a16=a16, azp=za, azp_adj=adj,
              bias=None if bias is None else _dev(bias))
        torch.cuda.synchronize()
        assert qlin_gpu.qlin_get_device_error() == 0
        ref = oracle.w8a8_epilogue(dh, rsa, rsb, azp=rza, azp_adj=radj, bias=bias)
        assert_within_tolerance(out.float().cpu().numpy(), ref, "config 4 bias=%s" % (bias is not None))
    raw = torch.empty((4096, 14336), dtype=torch.int32, device="cuda")
    _gemm(qlin_gpu, bform, aq, bq, None, None, raw, a16=a16)
    assert np.array_equal(raw.cpu().numpy(), dh)


@pytest.mark.parametrize("T,N,K", [(193, 264, 1552), (1, 8, 16), (300, 520, 3088), (128, 256, 1024)])
@pytest.mark.parametrize("out_dtype", [torch.bfloat16, torch.float16])
def test_operand_forms_agree_bit_for_bit(qlin_gpu, T, N, K, out_dtype):
    """The three operand forms compute the same D^ and apply the same
    epilogue in the same order: their outputs are equal bit for bit (the
    per-token zero-point form, with bias, on ragged tiles)."""
    rng = np.random.default_rng(T + N + K)
    x, w = _epilogue_case(rng, T, N, K)
    aq, sa, za = oracle.quant_int8_asym(x + 0.5)
    bq, sb = oracle.quant_int8_sym(w)
    adj = oracle.azp_adj_from_weight(bq)
    bias = (rng.standard_normal(N) * 0.1).astype(np.float32)
    outs = []
    for bform in BFORMS:
        out = torch.empty((T, N), dtype=out_dtype, device="cuda")
        _gemm(qlin_gpu, bform, _dev(aq), _dev(bq), _dev(sa), _dev(sb), out, azp=_dev(za), azp_adj=_dev(adj),
              bias=_dev(bias))
        torch.cuda.synchronize()
        assert qlin_gpu.qlin_get_device_error() == 0
        outs.append(out.cpu())
    ref = oracle.w8a8_epilogue(oracle.int8_gemm_exact(aq, bq), sa, sb, azp=za, azp_adj=adj, bias=bias)
    assert_within_tolerance(outs[0].float().numpy(), ref, "W8A8 forms %dx%dx%d" % (T, N, K))
    for o in outs[1:]:
        assert torch.equal(o.view(torch.int16), outs[0].view(torch.int16))
