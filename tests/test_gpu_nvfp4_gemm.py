"""NVFP4 block-scaled GEMM on the GPU against the CPU oracle, within the
bf16/fp16 tolerance: random operands over ragged tile and K-stage edges,
structured operands that expose the scale-factor layout, and the full
ARCQuant workload through the device quantizers."""

import numpy as np
import pytest
import torch

import oracle
import quantized_linear_layer_gb300 as qmod
from quantized_linear_layer_gb300 import inputs
from conftest import assert_within_tolerance, check_gemm_output, sf_rows_to_mma

pytestmark = pytest.mark.gpu


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def _gemm(q, qa, sfa, ga, qb, sfb, gb, out_dtype=torch.bfloat16):
    out = torch.empty((qa.shape[0], qb.shape[0]), dtype=out_dtype, device="cuda")
    q.qlin_nvfp4_gemm(_dev(oracle.pack_u4(qa)), _dev(sf_rows_to_mma(sfa)), _dev(oracle.pack_u4(qb)),
                      _dev(sf_rows_to_mma(sfb)),
                      _dev(np.array([ga], np.float32)), _dev(np.array([gb], np.float32)), out)
    torch.cuda.synchronize()
    assert q.qlin_get_device_error() == 0
    return out.float().cpu().numpy()


def _rand(rng, rows, k):
    codes = rng.integers(0, 16, size=(rows, k), dtype=np.uint8)
    sf = rng.integers(0x28, 0x48, size=(rows, k // 16), dtype=np.uint8)   # scales ~0.3 .. 4
    return codes, sf


@pytest.mark.parametrize("T,N,K", [(128, 128, 256), (130, 136, 320), (1, 8, 64), (200, 264, 4224), (300, 128, 1088),
                                   (129, 384, 192), (1300, 4480, 320)])
@pytest.mark.parametrize("out_dtype", [torch.bfloat16, torch.float16])
def test_random_operands(qlin_gpu, T, N, K, out_dtype):
    rng = np.random.default_rng(T + N + K)
    qa, sfa = _rand(rng, T, K)
    qb, sfb = _rand(rng, N, K)
    ga, gb = np.float32(0.05), np.float32(0.02)
    ref = oracle.nvfp4_gemm_reference(qa, sfa, ga, qb, sfb, gb)
    y = _gemm(qlin_gpu, qa, sfa, ga, qb, sfb, gb, out_dtype)
    check_gemm_output(y, ref, "nvfp4 %dx%dx%d" % (T, N, K), out_dtype)


def test_many_tiles_per_cta_pair(qlin_gpu):
    """18 M tiles x 24 N tiles (432 tiles): every persistent CTA walks about
    three tiles, so each stage slot is refilled across tile boundaries and
    the accumulator is handed to the epilogue several times."""
    T, N, K = 2304, 6144, 512
    rng = np.random.default_rng(77)
    qa, sfa = _rand(rng, T, K)
    qb, sfb = _rand(rng, N, K)
    ga, gb = np.float32(0.05), np.float32(0.02)
    ref = oracle.nvfp4_gemm_reference(qa, sfa, ga, qb, sfb, gb)
    y = _gemm(qlin_gpu, qa, sfa, ga, qb, sfb, gb, torch.bfloat16)
    check_gemm_output(y, ref, "nvfp4 %dx%dx%d" % (T, N, K), torch.bfloat16)


@pytest.mark.parametrize("T,N", [(128, 128), (128, 256), (256, 384)])
def test_scale_factor_layout(qlin_gpu, T, N):
    """Every element 1.0 and one non-unit block scale per row of A (and of B)
    at a row- and block-dependent position: any misplaced scale factor shows
    up as a wrong output.  N spans one, two and three 128-row scale blocks of
    B, so both halves of a 256-column tile are exercised."""
    K = 512
    qa = np.full((T, K), 2, dtype=np.uint8)           # E2M1 code 2 = 1.0
    qb = np.full((N, K), 2, dtype=np.uint8)
    one = 0x38                                         # E4M3 1.0
    sfa = np.full((T, K // 16), one, dtype=np.uint8)
    sfb = np.full((N, K // 16), one, dtype=np.uint8)
    for r in range(T):
        sfa[r, (r * 7) % (K // 16)] = 0x40             # 2.0
    for r in range(N):
        sfb[r, (r * 5 + 3) % (K // 16)] = 0x48         # 4.0
    ref = oracle.nvfp4_gemm_reference(qa, sfa, np.float32(1), qb, sfb, np.float32(1))
    y = _gemm(qlin_gpu, qa, sfa, 1.0, qb, sfb, 1.0, torch.bfloat16)
    assert np.array_equal(y, ref.astype(np.float32)) or np.allclose(y, ref, rtol=4e-3, atol=0)


def test_config5_arcquant(qlin_gpu):
    d = inputs.nvfp4_arc(seed=4)
    S = d["S"]
    x32 = d["x"].astype(np.float32)
    T, K = x32.shape
    N = d["w"].shape[0]
    xt, wt = _dev(d["x"]), _dev(d["w"])
    gx = torch.empty(1, dtype=torch.float32, device="cuda")
    gw = torch.empty(1, dtype=torch.float32, device="cuda")
    perm = torch.empty(K, dtype=torch.int32, device="cuda")
    qlin_gpu.qlin_nvfp4_global_scale(xt, gx)
    qlin_gpu.qlin_nvfp4_global_scale(wt, gw)
    qlin_gpu.qlin_arc_perm(xt, perm)
    qx = torch.empty((T, (K + S) // 2), dtype=torch.uint8, device="cuda")
    sfx = torch.empty((T, (K + S) // 16), dtype=torch.uint8, device="cuda")
    qw = torch.empty((N, (K + S) // 2), dtype=torch.uint8, device="cuda")
    sfw = torch.empty((N, (K + S) // 16), dtype=torch.uint8, device="cuda")
    qlin_gpu.qlin_quant_nvfp4(xt, gx, qx, sfx, perm=perm, S=S, mode=qmod.QLIN_NVFP4_RESIDUAL)
    qlin_gpu.qlin_quant_nvfp4(wt, gw, qw, sfw, perm=perm, S=S, mode=qmod.QLIN_NVFP4_DUPLICATE)
    # the GEMM reads the scales in the MMA layout, written directly by the quantizer
    sfx_m = torch.empty(qlin_gpu.qlin_nvfp4_sf_bytes(T, K + S, qmod.QLIN_SF_MMA), dtype=torch.uint8, device="cuda")
    sfw_m = torch.empty(qlin_gpu.qlin_nvfp4_sf_bytes(N, K + S, qmod.QLIN_SF_MMA), dtype=torch.uint8, device="cuda")
    qlin_gpu.qlin_quant_nvfp4(xt, gx, qx, sfx_m, perm=perm, S=S, mode=qmod.QLIN_NVFP4_RESIDUAL,
                              sf_layout=qmod.QLIN_SF_MMA)
    qlin_gpu.qlin_quant_nvfp4(wt, gw, qw, sfw_m, perm=perm, S=S, mode=qmod.QLIN_NVFP4_DUPLICATE,
                              sf_layout=qmod.QLIN_SF_MMA)
    out = torch.empty((T, N), dtype=torch.bfloat16, device="cuda")
    qlin_gpu.qlin_nvfp4_gemm(qx, sfx_m, qw, sfw_m, gx, gw, out)
    torch.cuda.synchronize()
    assert qlin_gpu.qlin_get_device_error() == 0
    rperm = oracle.arc_perm(x32)
    rgx, rgw = oracle.nvfp4_global_scale(x32), oracle.nvfp4_global_scale(d["w"])
    rqa, rsfa = oracle.arc_quantize_activation(x32, rperm, S, rgx)
    rqb, rsfb = oracle.arc_quantize_weight(d["w"], rperm, S, rgw)
    assert np.array_equal(qx.cpu().numpy(), oracle.pack_u4(rqa)) and np.array_equal(sfx.cpu().numpy(), rsfa)
    assert np.array_equal(qw.cpu().numpy(), oracle.pack_u4(rqb)) and np.array_equal(sfw.cpu().numpy(), rsfb)
    assert np.array_equal(sfx_m.cpu().numpy(), sf_rows_to_mma(rsfa))
    assert np.array_equal(sfw_m.cpu().numpy(), sf_rows_to_mma(rsfb))
    ref = oracle.nvfp4_gemm_reference(rqa, rsfa, rgx, rqb, rsfb, rgw)
    y = out.float().cpu().numpy()
    assert_within_tolerance(y, ref, "config 5")
    # the residual channels bring the product closer to the exact X W^T
    exact = x32.astype(np.float64) @ d["w"].astype(np.float64).T
    rq0, rs0 = oracle.arc_quantize_activation(x32, rperm, 0, rgx)
    wq0, ws0 = oracle.arc_quantize_weight(d["w"], rperm, 0, rgw)
    rtn = oracle.nvfp4_gemm_reference(rq0, rs0, rgx, wq0, ws0, rgw)
    assert np.linalg.norm(y - exact) < np.linalg.norm(rtn - exact)


@pytest.mark.parametrize("rows,K", [(128, 256), (130, 4224), (1, 64), (300, 1088)])
def test_sf_to_mma_conversion(qlin_gpu, rows, K):
    rng = np.random.default_rng(rows + K)
    sf = rng.integers(0, 0x7E, size=(rows, K // 16), dtype=np.uint8)
    out = torch.full((qlin_gpu.qlin_nvfp4_sf_bytes(rows, K, qmod.QLIN_SF_MMA),), 0xAB, dtype=torch.uint8, device="cuda")
    qlin_gpu.qlin_nvfp4_sf_to_mma(_dev(sf), out)
    torch.cuda.synchronize()
    assert np.array_equal(out.cpu().numpy(), sf_rows_to_mma(sf))
