"""FP8 W8A8 on the GPU against the CPU oracle: the per-row E4M3 quantizer bit
for bit (codes and scales), and the kind::f8f6f4 GEMM with per-token /
per-channel scales and bias within the fp16 / bf16 tolerance."""

import numpy as np
import pytest
import torch

import oracle
from quantized_linear_layer_gb300 import inputs
from conftest import assert_within_tolerance, check_gemm_output, load_golden

pytestmark = pytest.mark.gpu


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def _quant(q, x):
    rows, k = x.shape
    codes = torch.empty((rows, k), dtype=torch.uint8, device="cuda")
    scale = torch.empty(rows, dtype=torch.float32, device="cuda")
    q.qlin_quant_fp8(x, codes, scale)
    torch.cuda.synchronize()
    assert q.qlin_get_device_error() == 0
    return codes, scale


def _rows_with_edges(seed, rows, k):
    d = inputs.w8a8_sym_bias(seed=seed, T=rows, K=k, N=16)
    x = d["x"].astype(np.float32)
    x[1] = 0.0                               # all-zero row: scale 1, codes 0
    x[2, :] = 1e-7                           # quotients far below the E4M3 range
    x[2, 0] = 3.0
    x[3, 5] = 60000.0                        # one huge outlier
    x[4, :] = -0.0                           # signed zeros only
    x[5, ::2] = -x[5, ::2]
    return x


@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16, torch.float32])
def test_quant_fp8_bit_exact(qlin_gpu, dtype):
    x = _rows_with_edges(31, 96, 4096 + 64)
    xt = torch.from_numpy(x).to(dtype).cuda()
    codes, scale = _quant(qlin_gpu, xt)
    ref_codes, ref_scale = oracle.quant_fp8_rows(xt.float().cpu().numpy())
    assert np.array_equal(scale.cpu().numpy().view(np.uint32), ref_scale.view(np.uint32))
    got = codes.cpu().numpy()
    bad = np.argwhere(got != ref_codes)
    assert bad.size == 0, "first mismatches (row, col): %s" % bad[:5].tolist()


def test_quant_fp8_page_example(qlin_gpu):
    g = load_golden("fp8_w8a8_example.json")
    x = np.zeros((2, 16), dtype=np.float32)
    x[0, :4] = g["x"]
    codes, scale = _quant(qlin_gpu, _dev(x.astype(np.float16)))
    dec = oracle.e4m3_decode(codes.cpu().numpy()[0, :4])
    quot = np.asarray(g["x"], dtype=np.float64) / float(scale[0])
    for printed, code in g["printed_roundings"]:
        i = int(np.argmin(np.abs(quot - printed)))
        assert abs(quot[i] - printed) <= 0.005 and dec[i] == code
    assert np.max(np.abs(dec)) == g["e4m3_max"]


def _random_codes(rng, shape):
    c = rng.integers(0, 256, size=shape).astype(np.uint8)
    c[(c & 0x7F) == 0x7F] = 0x38            # no NaN codes (0x38 = 1.0)
    return c


@pytest.mark.parametrize("T,N,K,bias_dt,out_dt", [
    (200, 136, 208, None, torch.bfloat16),          # ragged tiles; K % 128 = 80 (a half-filled MMA)
    (129, 264, 4096, torch.float16, torch.float16),
    (257, 520, 1040, torch.float32, torch.bfloat16),
    (1, 8, 16, torch.bfloat16, torch.float16),      # the smallest problem
])
def test_fp8_gemm_against_oracle(qlin_gpu, T, N, K, bias_dt, out_dt):
    rng = np.random.default_rng(T * 7 + N)
    qa, qb = _random_codes(rng, (T, K)), _random_codes(rng, (N, K))
    # scales that keep the products in a sensible range for fp16 outputs
    sa = rng.uniform(0.5, 1.5, size=T).astype(np.float32) / np.float32(64.0 * np.sqrt(K))
    sb = rng.uniform(0.5, 1.5, size=N).astype(np.float32) / np.float32(64.0)
    bias = None if bias_dt is None else rng.standard_normal(N).astype(np.float32)
    bias_t = None if bias is None else torch.from_numpy(bias).to(bias_dt).cuda()
    bias_ref = None if bias is None else bias_t.float().cpu().numpy()
    out = torch.empty((T, N), dtype=out_dt, device="cuda")
    qlin_gpu.qlin_fp8_gemm(_dev(qa), _dev(qb), _dev(sa), _dev(sb), out, bias=bias_t)
    torch.cuda.synchronize()
    assert qlin_gpu.qlin_get_device_error() == 0
    ref = oracle.fp8_gemm_reference(qa, sa, qb, sb, bias_ref)
    check_gemm_output(out.float().cpu().numpy(), ref, "fp8 GEMM %dx%dx%d" % (T, N, K), out_dt)


def test_fp8_w8a8_pipeline_sampled_rows(qlin_gpu):
    """The W8A8 workload shape (T = 2048, N = K = 4096) in FP8: activations and
    weights quantized on the device, the GEMM with bias, checked against the
    oracle on a sample of rows (the oracle quantizes those rows itself)."""
    d = inputs.w8a8_sym_bias(seed=2, T=2048, K=4096, N=4096)
    x, w, bias = d["x"], d["w"], d["bias"]
    xt = _dev(x)
    wt = _dev(w.astype(np.float16))
    qa, sa = _quant(qlin_gpu, xt)
    qb, sb = _quant(qlin_gpu, wt)
    out = torch.empty((2048, 4096), dtype=torch.bfloat16, device="cuda")
    qlin_gpu.qlin_fp8_gemm(qa, qb, sa, sb, out, bias=_dev(bias))
    torch.cuda.synchronize()
    assert qlin_gpu.qlin_get_device_error() == 0
    rows = np.unique(np.concatenate([np.arange(0, 8), np.arange(2040, 2048),
                                     np.random.default_rng(5).choice(2048, 48, replace=False)]))
    oqa, osa = oracle.quant_fp8_rows(x[rows].astype(np.float32))
    oqb, osb = oracle.quant_fp8_rows(w.astype(np.float16).astype(np.float32))
    ref = oracle.fp8_gemm_reference(oqa, osa, oqb, osb, bias.astype(np.float32))
    assert_within_tolerance(out.float().cpu().numpy()[rows], ref, "fp8 W8A8 pipeline (sampled rows)")
