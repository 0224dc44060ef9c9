"""W4A16 with act-order (g_idx) on the GPU against the CPU oracle: the
offline preparation bit for bit (the group-sorted column order and the
reordered packed codes), and the run-time gather + GEMM within the fp16
tolerance for decode, skinny and prefill token counts; uneven groups are
reported through the device error word."""

import numpy as np
import pytest
import torch

import oracle
from conftest import assert_within_tolerance

pytestmark = pytest.mark.gpu


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def _case(seed, n, k):
    rng = np.random.default_rng(seed)
    g = k // 128
    g_idx = rng.permutation(np.repeat(np.arange(g), 128)).astype(np.int32)
    codes = rng.integers(0, 16, size=(n, k)).astype(np.uint8)
    scales = rng.uniform(0.001, 0.02, size=(n, g)).astype(np.float16)
    zeros = rng.integers(0, 16, size=(n, g)).astype(np.uint8)
    return g_idx, codes, scales, zeros


def _prepare(q, g_idx, wq):
    perm = torch.empty(g_idx.shape[0], dtype=torch.int32, device="cuda")
    wq_sorted = torch.empty_like(wq)
    q.qlin_w4a16_act_order_prepare(_dev(g_idx), wq, perm, wq_sorted)
    torch.cuda.synchronize()
    return perm, wq_sorted


@pytest.mark.parametrize("n,k", [(200, 640), (4096, 11008)])
def test_act_order_prepare_bit_exact(qlin_gpu, n, k):
    g_idx, codes, _, _ = _case(n + k, n, k)
    perm, wq_sorted = _prepare(qlin_gpu, g_idx, _dev(oracle.pack_u4(codes)))
    assert qlin_gpu.qlin_get_device_error() == 0
    ref_perm = oracle.act_order_perm(g_idx)
    assert np.array_equal(perm.cpu().numpy(), ref_perm)
    assert np.array_equal(wq_sorted.cpu().numpy(), oracle.pack_u4(codes[:, ref_perm]))


@pytest.mark.parametrize("T", [1, 5, 16, 33, 300])
def test_act_order_gemm_against_oracle(qlin_gpu, T):
    n, k = 520, 1152
    g_idx, codes, scales, zeros = _case(T, n, k)
    x = np.random.default_rng(T + 1).standard_normal((T, k)).astype(np.float16)
    perm, wq_sorted = _prepare(qlin_gpu, g_idx, _dev(oracle.pack_u4(codes)))
    y = torch.empty((T, n), dtype=torch.float16, device="cuda")
    qlin_gpu.qlin_w4a16_gemm_act_order(_dev(x), perm, wq_sorted, _dev(scales), _dev(oracle.pack_u4(zeros)), y)
    torch.cuda.synchronize()
    assert qlin_gpu.qlin_get_device_error() == 0
    ref = oracle.w4a16_act_order_reference(x, codes, scales, zeros, g_idx)
    assert_within_tolerance(y.cpu().numpy(), ref, "W4A16 act-order T=%d" % T)


def test_act_order_uneven_groups_reported(qlin_gpu):
    """A group holding 127 columns and another 129: the preparation records a
    device error (the gathers stay in bounds); a later valid call is clean."""
    n, k = 64, 512
    g_idx, codes, _, _ = _case(5, n, k)
    g_idx = g_idx.copy()
    g_idx[np.nonzero(g_idx == 0)[0][0]] = 1
    wq = _dev(oracle.pack_u4(codes))
    perm = torch.zeros(k, dtype=torch.int32, device="cuda")
    wq_sorted = torch.empty_like(wq)
    qlin_gpu.qlin_w4a16_act_order_prepare(_dev(g_idx), wq, perm, wq_sorted)
    torch.cuda.synchronize()
    assert qlin_gpu.qlin_get_device_error() != 0
    g_ok, _, _, _ = _case(5, n, k)
    _prepare(qlin_gpu, g_ok, wq)
    assert qlin_gpu.qlin_get_device_error() == 0
