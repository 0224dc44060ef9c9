"""RMSNorm fused with the per-token quantizers on the GPU against the CPU
oracle: codes and scales bit for bit, int8 and E4M3 outputs, 16-bit and
float32 inputs, rows held in registers and rows read twice; and the NVFP4 /
ARCQuant form (codes and block scales bit for bit).

The oracle's mean of squares is the exact sum of squares rounded once to
float32; the rows below include sums that a float32 sum in any fixed order
would round differently (a tie between two float32 values broken by a far
smaller square), rows whose squares span most of the float32 range, sums
that underflow to zero or overflow to infinity, and subnormal elements."""

import numpy as np
import pytest
import torch

import oracle
from quantized_linear_layer_gb300 import inputs
from conftest import sf_rows_to_mma

pytestmark = pytest.mark.gpu


def _rows(seed, rows, k, dtype=torch.float16):
    d = inputs.w8a8_sym_bias(seed=seed, T=rows, K=k, N=16)
    x = d["x"].astype(np.float32)
    x[1] = 0.0                 # all-zero row: y = 0, scale 1
    x[2] = 0.5                 # constant row
    x[3, 7] = 3000.0           # one outlier channel
    x[4] *= np.float32(1e-4)   # small magnitudes (the mean of squares near eps)
    if k >= 8:
        # the exact sum 1 + 2^-24 is halfway between two float32 values (ties
        # to even: 1); with 2^-20 (2^-40 squared) it lies above halfway
        x[5] = 0.0
        x[5, :2] = [1.0, 2.0 ** -12]
        x[6] = 0.0
        x[6, :3] = [1.0, 2.0 ** -12, 2.0 ** -20]
        x[6, 3:] = 2.0 ** -24          # the smallest fp16 subnormal, on every other channel
        x[6, 4::2] = 0.0
    if dtype != torch.float16:
        # squares spanning much of the float32 range; a sum above it (+inf:
        # y = 0); squares below the float32 range (a sum that rounds to 0)
        x[7] = x[0] * np.float32(1e-25)
        x[7, :4] = [1e18, -3e-18, 7.0, 1e-19]
        x[8] = 0.0
        x[8, :2] = [2.0 ** 64, 1.0]
        x[9] = np.float32(1e-38)
        x[9, ::3] = np.float32(3e-39)
    return x


@pytest.mark.parametrize("fmt", ["int8", "fp8"])
@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16, torch.float32])
@pytest.mark.parametrize("k,eps", [(4096, 1e-6), (8256, 1e-5), (16, 0.0), (4160, 1e-6)])
def test_rmsnorm_quant_bit_exact(qlin_gpu, fmt, dtype, k, eps):
    rng = np.random.default_rng(k + 3)
    x = _rows(41, 48, k, dtype)
    g = rng.uniform(0.5, 1.5, size=k).astype(np.float32)
    xt = torch.from_numpy(x).to(dtype).cuda()
    gt = torch.from_numpy(g).to(dtype).cuda()
    q_fmt = qlin_gpu.QLIN_QFMT_INT8 if fmt == "int8" else qlin_gpu.QLIN_QFMT_FP8_E4M3
    q = torch.empty((48, k), dtype=torch.int8 if fmt == "int8" else torch.uint8, device="cuda")
    s = torch.empty(48, dtype=torch.float32, device="cuda")
    qlin_gpu.qlin_rmsnorm_quant(xt, gt, eps, q, s, fmt=q_fmt)
    torch.cuda.synchronize()
    assert qlin_gpu.qlin_get_device_error() == 0
    xo, go = xt.float().cpu().numpy(), gt.float().cpu().numpy()
    if fmt == "int8":
        rq, rs = oracle.rmsnorm_quant_int8(xo, go, eps)
    else:
        rq, rs = oracle.rmsnorm_quant_fp8(xo, go, eps)
    assert np.array_equal(s.cpu().numpy().view(np.uint32), rs.view(np.uint32)), \
        "scales differ in rows %s" % np.nonzero(s.cpu().numpy() != rs)[0][:5].tolist()
    got = q.cpu().numpy().view(np.uint8)
    bad = np.argwhere(got != rq.view(np.uint8))
    assert bad.size == 0, "first mismatches (row, col): %s" % bad[:5].tolist()


@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16, torch.float32])
@pytest.mark.parametrize("k,eps,S,mode,layout", [
    (4096, 1e-6, 128, 0, "rows"),
    (8192, 1e-5, 256, 0, "mma"),
    (1024, 0.0, 0, 0, "rows"),         # eps = 0 with an all-zero row; no residual channels
    (4160, 1e-6, 64, 1, "mma"),        # duplicated (weight-side) columns
])
def test_rmsnorm_quant_nvfp4_bit_exact(qlin_gpu, dtype, k, eps, S, mode, layout):
    """RMSNorm fused with the NVFP4 / ARCQuant quantizer: codes and block scales
    bit for bit, g and perm calibrated by the oracle on the normalized rows;
    47 rows (an odd last pair of staged rows)."""
    rows = 47
    rng = np.random.default_rng(k + S)
    x = _rows(43, rows, k, dtype)
    gam = rng.uniform(0.5, 1.5, size=k).astype(np.float32)
    gam[5] = 6.0                                    # one strong channel of gamma
    xt = torch.from_numpy(x).to(dtype).cuda()
    gt = torch.from_numpy(gam).to(dtype).cuda()
    xo, go = xt.float().cpu().numpy(), gt.float().cpu().numpy()
    y = oracle.rmsnorm_rows(xo, go, eps)
    g = np.float32(oracle.nvfp4_global_scale(y))
    perm = oracle.arc_perm(y)
    sf_layout = qlin_gpu.QLIN_SF_ROWS if layout == "rows" else qlin_gpu.QLIN_SF_MMA
    q = torch.empty((rows, (k + S) // 2), dtype=torch.uint8, device="cuda")
    sf = torch.zeros(qlin_gpu.qlin_nvfp4_sf_bytes(rows, k + S, sf_layout), dtype=torch.uint8, device="cuda")
    qlin_gpu.qlin_rmsnorm_quant_nvfp4(xt, gt, eps, torch.tensor([g]).cuda(), q, sf,
                                      perm=torch.from_numpy(perm).cuda(), S=S, mode=mode, sf_layout=sf_layout)
    torch.cuda.synchronize()
    assert qlin_gpu.qlin_get_device_error() == 0
    if mode == 0:
        rq, rsf = oracle.rmsnorm_arc_quantize_activation(xo, go, eps, perm, S, g)
    else:
        rq, rsf = oracle.arc_quantize_weight(y, perm, S, g)
    want_sf = rsf.reshape(-1) if layout == "rows" else sf_rows_to_mma(rsf)
    assert np.array_equal(sf.cpu().numpy(), want_sf)
    got = q.cpu().numpy()
    bad = np.argwhere(got != oracle.pack_u4(rq))
    assert bad.size == 0, "first mismatches (row, byte): %s" % bad[:5].tolist()
