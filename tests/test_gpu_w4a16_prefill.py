"""W4A16 beyond decode (more than 64 tokens): the tcgen05 prefill GEMM on the
GPU against the CPU oracle within the fp16 tolerance, with ragged token and
weight-row tiles, symmetric and asymmetric zero-points, activation outliers,
the grouped entry point, and the Llama-2-7B layer shapes at 2048 tokens on
sampled rows."""

import numpy as np
import pytest
import torch

import oracle
from quantized_linear_layer_gb300 import inputs
from conftest import assert_within_tolerance

pytestmark = pytest.mark.gpu


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def _gemm(q, x, wq, sc, zp):
    y = torch.empty((x.shape[0], wq.shape[0]), dtype=torch.float16, device="cuda")
    q.qlin_w4a16_gemm(x, wq, sc, zp, y)
    torch.cuda.synchronize()
    assert q.qlin_get_device_error() == 0
    return y.cpu().numpy()


@pytest.mark.parametrize("T,N,K", [
    (65, 200, 640),        # one ragged token tile, ragged weight rows, odd group count (5)
    (300, 136, 1152),      # three token tiles (the last 44 tokens), 9 groups
    (129, 4096, 256),      # many weight-row tiles, two groups
    (513, 520, 4096),      # a longer K
])
def test_prefill_against_oracle(qlin_gpu, T, N, K):
    d = inputs.w4a16_decode(seed=T + N, T=T, N=N, K=K)
    codes, s16, z = oracle.quant_w4_g128(d["w"])
    ref = oracle.w4a16_reference(d["x"], codes, s16, z)
    y = _gemm(qlin_gpu, _dev(d["x"]), _dev(oracle.pack_u4(codes)), _dev(s16), _dev(oracle.pack_u4(z)))
    assert_within_tolerance(y, ref, "W4A16 prefill T=%d N=%d K=%d" % (T, N, K))


def test_prefill_symmetric_and_outliers(qlin_gpu):
    """NULL zero-points (z = 8) and activations with outlier channels."""
    T, N, K = 200, 384, 1024
    rng = np.random.default_rng(7)
    x = rng.standard_normal((T, K)).astype(np.float32)
    x[:, rng.choice(K, 10, replace=False)] *= 30.0
    x = x.astype(np.float16)
    codes = rng.integers(0, 16, size=(N, K)).astype(np.uint8)
    s16 = (rng.uniform(0.001, 0.01, size=(N, K // 128))).astype(np.float16)
    ref = oracle.w4a16_reference(x, codes, s16, None)
    y = _gemm(qlin_gpu, _dev(x), _dev(oracle.pack_u4(codes)), _dev(s16), None)
    assert_within_tolerance(y, ref, "W4A16 prefill, symmetric")


def test_prefill_all_codes_and_zero_points_exact(qlin_gpu):
    """Every (code, zero-point) pair with one-hot activations: each output is
    s . (q - z) itself, exact in fp16 for s = 0.25."""
    n, k, t = 256, 128, 128
    codes = np.tile(np.arange(16, dtype=np.uint8), (n, k // 16))
    zeros = (np.arange(n, dtype=np.uint8) % 16).reshape(n, 1)
    scales = np.full((n, 1), 0.25, dtype=np.float16)
    x = np.zeros((t, k), dtype=np.float16)
    x[np.arange(t), np.arange(t) % k] = 1.0
    y = _gemm(qlin_gpu, _dev(x), _dev(oracle.pack_u4(codes)), _dev(scales), _dev(oracle.pack_u4(zeros)))
    want = (codes[:, np.arange(t) % k].T.astype(np.float64) - zeros.T.astype(np.float64)) * 0.25
    assert np.array_equal(y.astype(np.float64), want)


def test_prefill_grouped_equals_separate(qlin_gpu):
    T, K = 160, 512
    shapes = [256, 384, 128]
    x = _dev(inputs.w4a16_decode(seed=61, T=T, N=8, K=K)["x"])
    mats = []
    for i, n in enumerate(shapes):
        codes, s16, z = oracle.quant_w4_g128(inputs.w4a16_decode(seed=70 + i, T=1, N=n, K=K)["w"])
        mats.append((_dev(oracle.pack_u4(codes)), _dev(s16), _dev(oracle.pack_u4(z))))
    ys = [torch.empty((T, n), dtype=torch.float16, device="cuda") for n in shapes]
    qlin_gpu.qlin_w4a16_gemm_grouped(x, [m[0] for m in mats], [m[1] for m in mats], [m[2] for m in mats], ys)
    torch.cuda.synchronize()
    for (wq, sc, zp), yg in zip(mats, ys):
        assert np.array_equal(_gemm(qlin_gpu, x, wq, sc, zp), yg.cpu().numpy())


@pytest.mark.parametrize("N,K", inputs.LLAMA2_7B_LAYERS)
def test_prefill_llama_layers_sampled_rows(qlin_gpu, N, K):
    """2048 tokens through each Llama-2-7B linear shape; the oracle checks a
    sample of token rows (its GEMM on all 2048 rows would take minutes)."""
    T = 2048
    d = inputs.w4a16_decode(seed=N + K, T=T, N=N, K=K)
    codes, s16, z = oracle.quant_w4_g128(d["w"])
    y = _gemm(qlin_gpu, _dev(d["x"]), _dev(oracle.pack_u4(codes)), _dev(s16), _dev(oracle.pack_u4(z)))
    rows = np.unique(np.concatenate([np.arange(0, 4), np.arange(T - 4, T),
                                     np.random.default_rng(N).choice(T, 24, replace=False)]))
    ref = oracle.w4a16_reference(d["x"][rows], codes, s16, z)
    assert_within_tolerance(y[rows], ref, "W4A16 prefill %dx%dx%d (sampled rows)" % (T, N, K))


@pytest.mark.parametrize("T,N,K", [
    (33, 8, 128),       # the smallest prefill: one tile, one K stage (no split)
    (257, 128, 256),    # three 128-token tiles, two K stages: a CTA pair splits K one stage each
    (64, 256, 384),     # an odd stage count split 1 + 2
    (100, 4096, 1024),  # 32 tiles, each shared by a cluster of four CTAs (two K stages each)
    (256, 11008, 512),  # 172 tiles of 128 tokens on persistent CTAs (some take two)
    (1000, 520, 256),   # eight token tiles, the last of 104 tokens, CTA pairs
])
def test_prefill_edge_shapes(qlin_gpu, T, N, K):
    d = inputs.w4a16_decode(seed=T * 3 + K, T=T, N=N, K=K)
    codes, s16, z = oracle.quant_w4_g128(d["w"])
    ref = oracle.w4a16_reference(d["x"], codes, s16, z)
    y = _gemm(qlin_gpu, _dev(d["x"]), _dev(oracle.pack_u4(codes)), _dev(s16), _dev(oracle.pack_u4(z)))
    assert_within_tolerance(y, ref, "W4A16 prefill edge T=%d N=%d K=%d" % (T, N, K))
