"""The C ABI on the CPU: the library loads, exports every entry point that
include/qlin.h declares, and rejects bad arguments before touching the GPU."""

import ctypes
import os
import re
import subprocess

import pytest

import quantized_linear_layer_gb300 as q
from quantized_linear_layer_gb300 import buildlib as qbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    src = open(os.path.join(ROOT, "include", "qlin.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(qlin_[a-z0-9_]+)\s*\(", src)))


@pytest.fixture(scope="module")
def built():
    qbuild.build()
    return q.lib()


def test_exports_every_declared_symbol(built):
    names = _declared()
    assert "qlin_w8a8_gemm" in names and "qlin_nvfp4_gemm" in names
    out = subprocess.run(["nm", "-D", "--defined-only", qbuild.LIB_PATH], capture_output=True, text=True).stdout
    exported = set(re.findall(r"\b(qlin_[a-z0-9_]+)\b", out))
    missing = [n for n in names if n not in exported]
    assert not missing, missing
    for n in names:
        assert hasattr(built, n)


def test_status_strings(built):
    built.qlin_status_string.restype = ctypes.c_char_p
    assert built.qlin_status_string(0) == b"QLIN_OK"
    assert built.qlin_status_string(5) == b"QLIN_ERR_TIMEOUT"
    assert built.qlin_version() >= 100


def test_rejects_bad_arguments_without_gpu(built):
    L = built
    P = ctypes.c_void_p
    # W4A16: group 64 is not built; T out of range; K not a multiple of the group
    assert L.qlin_w4a16_gemm(P(16), 1, 16, 256, P(16), P(16), None, 64, P(16), None) == 3
    assert L.qlin_w4a16_gemm(P(16), 1 << 31, 16, 256, P(16), P(16), None, 128, P(16), None) == 1
    assert L.qlin_w4a16_gemm(P(16), 1, 16, 200, P(16), P(16), None, 128, P(16), None) == 1
    assert L.qlin_w4a16_gemm(P(8), 1, 16, 256, P(16), P(16), None, 128, P(16), None) == 2
    # int8 quant: K not a multiple of 16, bad dtype, misaligned x
    assert L.qlin_quant_act_int8(P(16), 0, 4, 40, P(16), P(16), None, None) == 2
    assert L.qlin_quant_act_int8(P(16), 3, 4, 64, P(16), P(16), None, None) == 1
    assert L.qlin_quant_act_int8(P(24), 0, 4, 64, P(16), P(16), None, None) == 2
    # W8A8: scale numel, azp without azp_adj, bad out dtype
    assert L.qlin_w8a8_gemm(P(16), P(16), 4, 8, 64, P(16), 3, P(16), 8, None, None, None, 0, P(16), 0, None) == 1
    assert L.qlin_w8a8_gemm(P(16), P(16), 4, 8, 64, P(16), 4, P(16), 8, P(16), None, None, 0, P(16), 0, None) == 1
    assert L.qlin_w8a8_gemm(P(16), P(16), 4, 8, 64, P(16), 4, P(16), 8, None, None, None, 0, P(16), 2, None) == 1
    # the fp16-code forms take the same checks, and their own alignment
    assert L.qlin_quant_act_int8_f16(P(16), 0, 4, 40, P(16), P(16), None, None) == 2
    assert L.qlin_quant_act_int8_f16(P(16), 0, 4, 64, P(24), P(16), None, None) == 2
    assert L.qlin_w8a8_gemm_f16(P(16), P(16), 4, 8, 64, P(16), 3, P(16), 8, None, None, None, 0, P(16), 0, None) == 1
    assert L.qlin_w8a8_gemm_f16(P(16), P(16), 4, 8, 40, P(16), 4, P(16), 8, None, None, None, 0, P(16), 0, None) == 2
    assert L.qlin_w8a8_gemm_f16(P(24), P(16), 4, 8, 64, P(16), 4, P(16), 8, None, None, None, 0, P(16), 0, None) == 2
    # NVFP4: S not a multiple of 16, K+S not a multiple of 32, GEMM K not a multiple of 64
    assert L.qlin_quant_nvfp4(P(16), 0, 4, 64, None, 8, 0, P(16), P(16), P(16), 0, None) == 1
    assert L.qlin_quant_nvfp4(P(16), 0, 4, 64, None, 16, 0, P(16), P(16), P(16), 0, None) == 2
    # the MMA scale layout needs K+S to be a multiple of 64
    assert L.qlin_quant_nvfp4(P(16), 0, 4, 96, None, 0, 0, P(16), P(16), P(16), 1, None) == 1
    assert L.qlin_nvfp4_sf_bytes(130, 4224, 1) == 2 * 66 * 512
    assert L.qlin_nvfp4_sf_bytes(130, 4224, 0) == 130 * 264
    assert L.qlin_nvfp4_sf_bytes(130, 4208, 1) == -1
    assert L.qlin_nvfp4_gemm(P(16), P(16), P(16), P(16), 4, 8, 96, P(16), P(16), P(16), 1, None) == 1
    # grouped W4A16: count outside [1, 4], null host arrays, K not a multiple of the group
    n2 = (ctypes.c_int64 * 2)(16, 16)
    ptrs = (ctypes.c_void_p * 2)(16, 16)
    assert L.qlin_w4a16_gemm_grouped(P(16), 1, 256, 0, n2, ptrs, ptrs, ptrs, 128, ptrs, None) == 1
    assert L.qlin_w4a16_gemm_grouped(P(16), 1, 256, 5, n2, ptrs, ptrs, ptrs, 128, ptrs, None) == 1
    assert L.qlin_w4a16_gemm_grouped(P(16), 1, 256, 2, None, ptrs, ptrs, ptrs, 128, ptrs, None) == 1
    assert L.qlin_w4a16_gemm_grouped(P(16), 1, 200, 2, n2, ptrs, ptrs, ptrs, 128, ptrs, None) == 1
    assert L.qlin_w4a16_gemm_grouped(P(16), 1, 256, 2, n2, ptrs, ptrs, ptrs, 64, ptrs, None) == 3
    bad = (ctypes.c_void_p * 2)(16, 24)
    assert L.qlin_w4a16_gemm_grouped(P(16), 1, 256, 2, n2, bad, ptrs, ptrs, 128, ptrs, None) == 2
    # W4A16 sequence: workspace size, bad K, null workspace, bad group
    assert L.qlin_w4a16_sequence_workspace_bytes(128) == 512
    assert L.qlin_w4a16_sequence_workspace_bytes(-1) == -1

    class Step(ctypes.Structure):
        _fields_ = [("x", ctypes.c_void_p), ("K", ctypes.c_int64), ("count", ctypes.c_int),
                    ("N", ctypes.c_int64 * 4), ("wq", ctypes.c_void_p * 4), ("scales", ctypes.c_void_p * 4),
                    ("zeros", ctypes.c_void_p * 4), ("y", ctypes.c_void_p * 4)]
    assert ctypes.sizeof(Step) == 184
    st = (Step * 1)()
    st[0].x, st[0].K, st[0].count = 16, 200, 1
    st[0].N[0], st[0].wq[0], st[0].scales[0], st[0].y[0] = 16, 16, 16, 16
    sp = ctypes.cast(st, ctypes.c_void_p)
    assert L.qlin_w4a16_gemv_sequence(sp, 1, 128, P(16), None) == 1      # K not a multiple of 128
    st[0].K = 256
    assert L.qlin_w4a16_gemv_sequence(sp, 1, 128, None, None) == 1       # null workspace
    assert L.qlin_w4a16_gemv_sequence(sp, 1, 64, P(16), None) == 3       # group 64 not built
    st[0].K = 12416
    assert L.qlin_w4a16_gemv_sequence(sp, 1, 128, P(16), None) == 3      # K above 12288
    st[0].K, st[0].count = 256, 5
    assert L.qlin_w4a16_gemv_sequence(sp, 1, 128, P(16), None) == 1      # count above 4
    assert L.qlin_w4a16_gemv_sequence(None, 0, 128, None, None) == 0     # empty sequence
    # W4A16 decode plan: workspace size; tokens outside 1 .. 16, null steps, no steps, null or
    # misaligned workspace, K not a multiple of 128 (all before the device is touched)
    assert L.qlin_w4a16_decode_workspace_bytes(-1) == -1
    assert L.qlin_w4a16_decode_workspace_bytes(224) >= 224 * (4 * 128 + 4)
    st[0].K, st[0].count = 256, 1
    assert L.qlin_w4a16_decode_prepare(sp, 1, 17, 128, P(256), None) == 3
    assert L.qlin_w4a16_decode_prepare(sp, 1, 0, 128, P(256), None) == 3
    assert L.qlin_w4a16_decode_prepare(None, 1, 4, 128, P(256), None) == 1
    assert L.qlin_w4a16_decode_prepare(sp, 0, 4, 128, P(256), None) == 1
    assert L.qlin_w4a16_decode_prepare(sp, 1, 4, 128, None, None) == 1
    assert L.qlin_w4a16_decode_prepare(sp, 1, 4, 128, P(272), None) == 2
    st[0].K = 200
    assert L.qlin_w4a16_decode_prepare(sp, 1, 4, 128, P(256), None) == 1
    st[0].K = 256
    assert L.qlin_w4a16_decode_prepare(sp, 1, 4, 64, P(256), None) == 3
    assert L.qlin_w4a16_decode_run(P(256), 0, 4, None) == 1
    assert L.qlin_w4a16_decode_run(P(256), 1, 17, None) == 3
    assert L.qlin_w4a16_decode_run(P(272), 1, 4, None) == 2
    assert L.qlin_w4a16_decode_run(None, 1, 4, None) == 1
    # FP8: K not a multiple of 16, bad dtype, misaligned x; GEMM out dtype, bias dtype,
    # misaligned b, out row pitch (N = 12: 24 bytes)
    assert L.qlin_quant_fp8(P(16), 0, 4, 40, P(16), P(16), None) == 2
    assert L.qlin_quant_fp8(P(16), 3, 4, 64, P(16), P(16), None) == 1
    assert L.qlin_quant_fp8(P(24), 0, 4, 64, P(16), P(16), None) == 2
    assert L.qlin_fp8_gemm(P(16), P(16), 4, 8, 64, P(16), P(16), None, 0, P(16), 2, None) == 1
    assert L.qlin_fp8_gemm(P(16), P(16), 4, 8, 64, P(16), P(16), P(16), 3, P(16), 0, None) == 1
    assert L.qlin_fp8_gemm(P(16), P(24), 4, 8, 64, P(16), P(16), None, 0, P(16), 0, None) == 2
    assert L.qlin_fp8_gemm(P(16), P(16), 4, 12, 64, P(16), P(16), None, 0, P(16), 0, None) == 2
    assert L.qlin_fp8_gemm(P(16), P(16), 4, 8, 72, P(16), P(16), None, 0, P(16), 0, None) == 2
    # fused RMSNorm + quant: unknown format, negative eps, K not a multiple of 16, misaligned gamma
    F = ctypes.c_float
    assert L.qlin_rmsnorm_quant(P(16), 0, 4, 64, P(16), F(1e-6), 2, P(16), P(16), None) == 1
    assert L.qlin_rmsnorm_quant(P(16), 0, 4, 64, P(16), F(-1.0), 0, P(16), P(16), None) == 1
    assert L.qlin_rmsnorm_quant(P(16), 0, 4, 40, P(16), F(1e-6), 0, P(16), P(16), None) == 2
    assert L.qlin_rmsnorm_quant(P(16), 0, 4, 64, P(24), F(1e-6), 1, P(16), P(16), None) == 2
    assert L.qlin_rmsnorm_quant(None, 0, 0, 64, None, F(1e-6), 0, None, None, None) == 0
    # fused RMSNorm + NVFP4: null gamma, negative eps, misaligned gamma, S not a multiple
    # of 16, a row above 96 KB; an empty problem needs no pointers
    assert L.qlin_rmsnorm_quant_nvfp4(P(16), 0, 4, 64, None, F(1e-6), None, 0, 0, P(16), P(16), P(16), 0, None) == 1
    assert L.qlin_rmsnorm_quant_nvfp4(P(16), 0, 4, 64, P(16), F(-1.0), None, 0, 0, P(16), P(16), P(16), 0, None) == 1
    assert L.qlin_rmsnorm_quant_nvfp4(P(16), 0, 4, 64, P(24), F(1e-6), None, 0, 0, P(16), P(16), P(16), 0, None) == 2
    assert L.qlin_rmsnorm_quant_nvfp4(P(16), 2, 4, 24608, P(16), F(1e-6), None, 0, 0, P(16), P(16), P(16), 0,
                                      None) == 3
    assert L.qlin_rmsnorm_quant_nvfp4(P(16), 0, 4, 64, P(16), F(1e-6), None, 8, 0, P(16), P(16), P(16), 0, None) == 1
    assert L.qlin_rmsnorm_quant_nvfp4(None, 0, 0, 64, None, F(1e-6), None, 0, 0, None, None, None, 0, None) == 0
    # Hadamard: unknown kind, n not a power of two, regular n = 8, n above 8192, K not a
    # multiple of n, misaligned signs; an empty problem
    assert L.qlin_hadamard(P(16), 0, 4, 256, 2, 256, None, P(16), None) == 1
    assert L.qlin_hadamard(P(16), 0, 4, 384, 0, 48, None, P(16), None) == 1
    assert L.qlin_hadamard(P(16), 0, 4, 256, 1, 8, None, P(16), None) == 1
    assert L.qlin_hadamard(P(16), 0, 4, 16384, 0, 16384, None, P(16), None) == 1
    assert L.qlin_hadamard(P(16), 0, 4, 320, 0, 256, None, P(16), None) == 1
    assert L.qlin_hadamard(P(16), 0, 4, 256, 0, 256, P(12), P(16), None) == 2
    assert L.qlin_hadamard(None, 0, 0, 256, 0, 256, None, None, None) == 0
    # act-order: group 64 not built, K not a multiple of 128, misaligned perm, wq_sorted
    # aliasing wq; GEMM: x_work missing or aliasing x, misaligned x_work; empty problems
    assert L.qlin_w4a16_act_order_prepare(P(16), 256, 64, P(16), 4, P(16), P(32), None) == 3
    assert L.qlin_w4a16_act_order_prepare(P(16), 200, 128, P(16), 4, P(16), P(32), None) == 1
    assert L.qlin_w4a16_act_order_prepare(P(16), 256, 128, P(16), 4, P(24), P(32), None) == 2
    assert L.qlin_w4a16_act_order_prepare(P(16), 256, 128, P(16), 4, P(16), P(16), None) == 1
    assert L.qlin_w4a16_gemm_act_order(P(16), 2, 8, 256, P(16), P(16), P(16), None, 128, None, P(16), None) == 1
    assert L.qlin_w4a16_gemm_act_order(P(16), 2, 8, 256, P(16), P(16), P(16), None, 128, P(16), P(16), None) == 1
    assert L.qlin_w4a16_gemm_act_order(P(16), 2, 8, 256, P(16), P(16), P(16), None, 128, P(40), P(16), None) == 2
    assert L.qlin_w4a16_gemm_act_order(None, 0, 8, 256, None, None, None, None, 128, None, None, None) == 0
    # MX: unknown format, K not a multiple of 32, misaligned x; GEMM: MXFP4 K not a
    # multiple of 64, F32 out, out row pitch (N = 12); empty problems; scale sizes
    assert L.qlin_quant_mx(P(16), 0, 4, 64, 2, P(16), P(16), 0, None) == 1
    assert L.qlin_quant_mx(P(16), 0, 4, 48, 0, P(16), P(16), 0, None) == 1
    assert L.qlin_quant_mx(P(24), 0, 4, 64, 1, P(16), P(16), 1, None) == 2
    assert L.qlin_quant_mx(None, 0, 0, 64, 0, None, None, 0, None) == 0
    assert L.qlin_mx_gemm(P(16), P(16), P(16), P(16), 4, 8, 96, 1, P(16), 0, None) == 1
    assert L.qlin_mx_gemm(P(16), P(16), P(16), P(16), 4, 8, 96, 0, P(16), 2, None) == 1
    assert L.qlin_mx_gemm(P(16), P(16), P(16), P(16), 4, 12, 96, 0, P(16), 0, None) == 2
    assert L.qlin_mx_gemm(None, None, None, None, 0, 8, 96, 0, None, 0, None) == 0
    assert L.qlin_mx_sf_bytes(130, 160, 1) == 2 * 2 * 512 and L.qlin_mx_sf_bytes(3, 96, 0) == 9
    assert L.qlin_mx_sf_bytes(3, 100, 0) == -1
    # perm K limit
    assert L.qlin_arc_perm(P(16), 0, 4, 32768, P(16), None) == 1
    msg = L.qlin_last_error_message()
    assert b"16384" in msg


def test_empty_problems_launch_nothing(built):
    L = built
    P = ctypes.c_void_p
    assert L.qlin_w4a16_gemm(None, 0, 16, 256, None, None, None, 128, None, None) == 0
    n0 = (ctypes.c_int64 * 2)(0, 0)
    nul = (ctypes.c_void_p * 2)(None, None)
    assert L.qlin_w4a16_gemm_grouped(None, 1, 256, 2, n0, nul, nul, nul, 128, nul, None) == 0
    assert L.qlin_quant_act_int8(None, 0, 0, 64, None, None, None, None) == 0
    assert L.qlin_w8a8_gemm(None, None, 0, 8, 64, None, 1, None, 1, None, None, None, 0, None, 0, None) == 0
    assert L.qlin_w8a8_gemm_f16(None, None, 0, 8, 64, None, 1, None, 1, None, None, None, 0, None, 0, None) == 0
    assert L.qlin_quant_act_int8_f16(None, 0, 0, 64, None, None, None, None) == 0
    assert L.qlin_nvfp4_gemm(None, None, None, None, 4, 0, 64, None, None, None, 1, None) == 0
    assert L.qlin_quant_fp8(None, 0, 0, 64, None, None, None) == 0
    assert L.qlin_fp8_gemm(None, None, 0, 8, 64, None, None, None, 0, None, 0, None) == 0


def test_chain_checks_every_step_before_launching(built):
    """qlin_w4a16_chain rejects a bad step anywhere in the chain on the host,
    before any launch (no GPU is touched here)."""
    L = built
    steps = (q.qlin_w4a16_step * 2)()
    for st in steps:
        st.x, st.K, st.count = 16, 256, 1
        st.N[0], st.wq[0], st.scales[0], st.y[0] = 8, 32, 64, 96
    arr = ctypes.cast(steps, ctypes.c_void_p)
    assert L.qlin_w4a16_chain(arr, 2, 1, 64, None) == 3            # group 64 is not built
    steps[1].x = 24                                                 # step 1: x not 16-byte aligned
    assert L.qlin_w4a16_chain(arr, 2, 1, 128, None) == 2
    assert b"step 1" in L.qlin_last_error_message()
    steps[1].x, steps[1].count = 16, 0                              # step 1: no matrix
    assert L.qlin_w4a16_chain(arr, 2, 1, 128, None) == 1
    steps[1].count, steps[1].K = 1, 200                             # K not a multiple of 128
    assert L.qlin_w4a16_chain(arr, 2, 4, 128, None) == 1
    assert L.qlin_w4a16_chain(arr, 0, 4, 128, None) == 0            # nothing to do
    assert L.qlin_w4a16_chain(None, 2, 4, 128, None) == 1
