"""MX block-scaled formats on the GPU against the CPU oracle: the MXFP8 /
MXFP4 quantizer bit for bit (codes and E8M0 scales, both scale layouts), and
the block-scaled GEMM (kind::mxf8f6f4 scale_vec::1X, kind::mxf4nvf4
scale_vec::2X) within the fp16 / bf16 tolerance."""

import numpy as np
import pytest
import torch

import oracle
from quantized_linear_layer_gb300 import inputs
from conftest import assert_within_tolerance, check_gemm_output, sf_rows_to_mma

pytestmark = pytest.mark.gpu

FMTS = {"mxfp8": ("e4m3", 0), "mxfp4": ("e2m1", 1)}


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def _mx_sf_mma(sf):
    """Row-major E8M0 scales [rows][K/32] -> the QLIN_SF_MMA bytes (scale groups
    of 4 padded with zeros, rows padded to 128)."""
    rows, kb = sf.shape
    pad = np.zeros((rows, (kb + 3) // 4 * 4), dtype=np.uint8)
    pad[:, :kb] = sf
    return sf_rows_to_mma(pad)


def _codes_bytes(codes, ofmt):
    return codes if ofmt == "e4m3" else oracle.pack_u4(codes)


def _quant(q, xt, fmt, layout):
    rows, k = xt.shape
    ofmt, code = FMTS[fmt]
    qb = torch.empty((rows, k if ofmt == "e4m3" else k // 2), dtype=torch.uint8, device="cuda")
    sf = torch.zeros(q.qlin_mx_sf_bytes(rows, k, layout), dtype=torch.uint8, device="cuda")
    q.qlin_quant_mx(xt, qb, sf, fmt=code, sf_layout=layout)
    torch.cuda.synchronize()
    assert q.qlin_get_device_error() == 0
    return qb, sf


def _rows_with_edges(seed, rows, k):
    rng = np.random.default_rng(seed)
    x = (rng.standard_normal((rows, k)) * np.exp(rng.uniform(-6, 6, size=(rows, 1)))).astype(np.float32)
    x[1] = 0.0                        # zero blocks: scale code 0, codes 0
    x[2, :32] = 1e-30                 # a block far below the normal range of fp16 (f32 only)
    x[3, 40] = 60000.0                # one outlier block
    x[4, ::3] = -0.0                  # signed zeros
    x[5, 64:96] = 6.0                 # a constant block (exactly at a power-of-two boundary times 1.5)
    return x


@pytest.mark.parametrize("fmt", ["mxfp8", "mxfp4"])
@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16, torch.float32])
@pytest.mark.parametrize("k", [4096 + 32, 64])
def test_quant_mx_bit_exact(qlin_gpu, fmt, dtype, k):
    rows = 133                                    # a ragged last 128-row scale tile
    x = _rows_with_edges(k + rows, rows, k)
    xt = torch.from_numpy(x).to(dtype).cuda()
    ofmt = FMTS[fmt][0]
    rq, rsf = oracle.mx_quantize(xt.float().cpu().numpy(), ofmt)
    for layout in (qlin_gpu.QLIN_SF_ROWS, qlin_gpu.QLIN_SF_MMA):
        qb, sf = _quant(qlin_gpu, xt, fmt, layout)
        want_sf = rsf.reshape(-1) if layout == qlin_gpu.QLIN_SF_ROWS else _mx_sf_mma(rsf)
        assert np.array_equal(sf.cpu().numpy(), want_sf), "scales differ (layout %d)" % layout
        got = qb.cpu().numpy()
        bad = np.argwhere(got != _codes_bytes(rq, ofmt))
        assert bad.size == 0, "first mismatches (row, byte): %s" % bad[:5].tolist()


def _random_operands(rng, rows, k, ofmt):
    if ofmt == "e4m3":
        c = rng.integers(0, 256, size=(rows, k)).astype(np.uint8)
        c[(c & 0x7F) == 0x7F] = 0x38
    else:
        c = rng.integers(0, 16, size=(rows, k)).astype(np.uint8)
    # scale ranges that keep K-long sums of products inside fp16
    lo, hi = (116, 122) if ofmt == "e4m3" else (118, 128)
    sf = rng.integers(lo, hi, size=(rows, k // 32)).astype(np.uint8)
    return c, sf


@pytest.mark.parametrize("fmt", ["mxfp8", "mxfp4"])
@pytest.mark.parametrize("T,N,K,out_dt", [
    (200, 136, 192, torch.bfloat16),     # ragged tiles; a partial stage (3 of 4 MMAs for MXFP4, 2 for MXFP8)
    (129, 264, 4096, torch.float16),
    (257, 520, 1088, torch.bfloat16),    # a partial 4-scale group at the end of K
    (1, 8, 64, torch.float16),           # the smallest problem
])
def test_mx_gemm_against_oracle(qlin_gpu, fmt, T, N, K, out_dt):
    ofmt, code = FMTS[fmt]
    rng = np.random.default_rng(T * 13 + N + K)
    qa, sfa = _random_operands(rng, T, K, ofmt)
    qb, sfb = _random_operands(rng, N, K, ofmt)
    out = torch.empty((T, N), dtype=out_dt, device="cuda")
    qlin_gpu.qlin_mx_gemm(_dev(_codes_bytes(qa, ofmt)), _dev(_mx_sf_mma(sfa)), _dev(_codes_bytes(qb, ofmt)),
                          _dev(_mx_sf_mma(sfb)), out, fmt=code)
    torch.cuda.synchronize()
    assert qlin_gpu.qlin_get_device_error() == 0
    ref = oracle.mx_gemm_reference(qa, sfa, qb, sfb, ofmt)
    check_gemm_output(out.float().cpu().numpy(), ref, "%s GEMM %dx%dx%d" % (fmt, T, N, K), out_dt)


@pytest.mark.parametrize("fmt", ["mxfp8", "mxfp4"])
def test_mx_pipeline_sampled_rows(qlin_gpu, fmt):
    """T = 2048, N = K = 4096 (the W8A8 / NVFP4 workload shape): activations and
    weights quantized on the device into the MMA scale layout, then the GEMM,
    checked on a sample of rows against the oracle's quantization and GEMM."""
    ofmt, code = FMTS[fmt]
    d = inputs.w8a8_sym_bias(seed=4, T=2048, K=4096, N=4096)
    x, w = d["x"], d["w"].astype(np.float16)
    qx, sfx = _quant(qlin_gpu, _dev(x), fmt, qlin_gpu.QLIN_SF_MMA)
    qw, sfw = _quant(qlin_gpu, _dev(w), fmt, qlin_gpu.QLIN_SF_MMA)
    out = torch.empty((2048, 4096), dtype=torch.bfloat16, device="cuda")
    qlin_gpu.qlin_mx_gemm(qx, sfx, qw, sfw, out, fmt=code)
    torch.cuda.synchronize()
    assert qlin_gpu.qlin_get_device_error() == 0
    rows = np.unique(np.concatenate([np.arange(0, 8), np.arange(2040, 2048),
                                     np.random.default_rng(6).choice(2048, 48, replace=False)]))
    oqa, osa = oracle.mx_quantize(x[rows].astype(np.float32), ofmt)
    oqb, osb = oracle.mx_quantize(w.astype(np.float32), ofmt)
    ref = oracle.mx_gemm_reference(oqa, osa, oqb, osb, ofmt)
    assert_within_tolerance(out.float().cpu().numpy()[rows], ref, "%s pipeline (sampled rows)" % fmt)


@pytest.mark.parametrize("fmt,T,N,K", [("mxfp8", 1, 8, 32), ("mxfp4", 3, 16, 64), ("mxfp8", 130, 264, 96)])
def test_mx_gemm_smallest_k(qlin_gpu, fmt, T, N, K):
    """One MMA of K (a single scale block for MXFP8, two for MXFP4), and a K of
    three MXFP8 MMAs whose scale group is partial."""
    ofmt, code = FMTS[fmt]
    rng = np.random.default_rng(K + T)
    qa, sfa = _random_operands(rng, T, K, ofmt)
    qb, sfb = _random_operands(rng, N, K, ofmt)
    out = torch.empty((T, N), dtype=torch.bfloat16, device="cuda")
    qlin_gpu.qlin_mx_gemm(_dev(_codes_bytes(qa, ofmt)), _dev(_mx_sf_mma(sfa)), _dev(_codes_bytes(qb, ofmt)),
                          _dev(_mx_sf_mma(sfb)), out, fmt=code)
    torch.cuda.synchronize()
    assert qlin_gpu.qlin_get_device_error() == 0
    ref = oracle.mx_gemm_reference(qa, sfa, qb, sfb, ofmt)
    check_gemm_output(out.float().cpu().numpy(), ref, "%s GEMM %dx%dx%d" % (fmt, T, N, K), torch.bfloat16)
