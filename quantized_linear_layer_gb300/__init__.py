"""GB300-native quantized linear layer: thin Python binding of libqlin.so.

Every function here has the name of a C entry point declared in
include/qlin.h and does argument marshalling only: it reads sizes, dtypes
and device pointers from torch tensors, passes them with the current CUDA
stream, and raises QlinError on a non-OK status.  All computation happens in
the library's CUDA kernels; there is no CPU or PyTorch fallback.  If the
library has not been built, the first call raises.

Outputs are caller-allocated tensors, exactly as in the C ABI.
"""

import ctypes
import os

from .buildlib import LIB_PATH, build  # noqa: F401

__all__ = [
    "QlinError", "lib", "build",
    "QLIN_F16", "QLIN_BF16", "QLIN_F32", "QLIN_I32", "QLIN_NVFP4_RESIDUAL", "QLIN_NVFP4_DUPLICATE",
    "QLIN_SF_ROWS", "QLIN_SF_MMA", "qlin_nvfp4_sf_bytes", "qlin_nvfp4_sf_to_mma",
    "qlin_version", "qlin_get_device_error",
    "qlin_quant_w4_g128", "qlin_w4a16_gemm", "qlin_w4a16_gemm_grouped", "qlin_w4a16_gemv_launch_info",
    "qlin_w4a16_step",
    "qlin_w4a16_sequence_workspace_bytes", "qlin_w4a16_gemv_sequence", "qlin_w4a16_gemv_sequence_noalloc",
    "qlin_w4a16_chain", "qlin_w4a16_decode_workspace_bytes", "qlin_w4a16_decode_prepare", "qlin_w4a16_decode_run",
    "qlin_quant_act_int8", "qlin_int8_row_sum", "qlin_w8a8_gemm", "qlin_int8_to_f16", "qlin_w8a8_gemm_f16b",
    "qlin_quant_act_int8_f16", "qlin_w8a8_gemm_f16",
    "qlin_nvfp4_global_scale", "qlin_arc_perm", "qlin_quant_nvfp4", "qlin_nvfp4_gemm",
    "QLIN_QFMT_INT8", "QLIN_QFMT_FP8_E4M3", "qlin_quant_fp8", "qlin_fp8_gemm", "qlin_rmsnorm_quant",
    "qlin_rmsnorm_quant_nvfp4", "QLIN_MX_FP8_E4M3", "QLIN_MX_FP4_E2M1", "qlin_mx_sf_bytes", "qlin_quant_mx",
    "qlin_mx_gemm", "QLIN_HADAMARD_SYLVESTER", "QLIN_HADAMARD_REGULAR", "qlin_hadamard",
    "qlin_w4a16_act_order_prepare", "qlin_w4a16_gemm_act_order",
]

QLIN_F16, QLIN_BF16, QLIN_F32, QLIN_I32 = 0, 1, 2, 3
QLIN_NVFP4_RESIDUAL, QLIN_NVFP4_DUPLICATE = 0, 1
QLIN_SF_ROWS, QLIN_SF_MMA = 0, 1
QLIN_QFMT_INT8, QLIN_QFMT_FP8_E4M3 = 0, 1
QLIN_MX_FP8_E4M3, QLIN_MX_FP4_E2M1 = 0, 1
QLIN_HADAMARD_SYLVESTER, QLIN_HADAMARD_REGULAR = 0, 1

_STATUS = {0: "QLIN_OK", 1: "QLIN_ERR_INVALID_ARG", 2: "QLIN_ERR_ALIGNMENT", 3: "QLIN_ERR_UNSUPPORTED",
           4: "QLIN_ERR_CUDA", 5: "QLIN_ERR_TIMEOUT"}


class QlinError(RuntimeError):
    def __init__(self, status, fn, message):
        self.status = status
        super().__init__("%s failed: %s (%s)" % (fn, _STATUS.get(status, status), message))


_P = ctypes.c_void_p
_I64 = ctypes.c_int64
_I32 = ctypes.c_int
_SIGS = {
    "qlin_version": ([], ctypes.c_int),
    "qlin_status_string": ([_I32], ctypes.c_char_p),
    "qlin_last_error_message": ([], ctypes.c_char_p),
    "qlin_get_device_error": ([_P, _P], _I32),
    "qlin_w4a16_gemv_launch_info": ([_P, _P], _I32),
    "qlin_quant_w4_g128": ([_P, _I32, _I64, _I64, _I64, _P, _P, _P, _P], _I32),
    "qlin_w4a16_gemm": ([_P, _I64, _I64, _I64, _P, _P, _P, _I64, _P, _P], _I32),
    "qlin_w4a16_gemm_grouped": ([_P, _I64, _I64, _I32, _P, _P, _P, _P, _I64, _P, _P], _I32),
    "qlin_w4a16_sequence_workspace_bytes": ([_I64], _I64),
    "qlin_w4a16_gemv_sequence": ([_P, _I32, _I64, _P, _P], _I32),
    "qlin_w4a16_gemv_sequence_noalloc": ([_P, _I32, _I64, _P], _I32),
    "qlin_w4a16_chain": ([_P, _I32, _I64, _I64, _P], _I32),
    "qlin_w4a16_decode_workspace_bytes": ([_I64], _I64),
    "qlin_w4a16_decode_prepare": ([_P, _I32, _I64, _I64, _P, _P], _I32),
    "qlin_w4a16_decode_run": ([_P, _I32, _I64, _P], _I32),
    "qlin_quant_act_int8": ([_P, _I32, _I64, _I64, _P, _P, _P, _P], _I32),
    "qlin_int8_row_sum": ([_P, _I64, _I64, _P, _P], _I32),
    "qlin_w8a8_gemm": ([_P, _P, _I64, _I64, _I64, _P, _I64, _P, _I64, _P, _P, _P, _I32, _P, _I32, _P], _I32),
    "qlin_w8a8_gemm_f16b": ([_P, _P, _I64, _I64, _I64, _P, _I64, _P, _I64, _P, _P, _P, _I32, _P, _I32, _P], _I32),
    "qlin_int8_to_f16": ([_P, _I64, _P, _P], _I32),
    "qlin_quant_act_int8_f16": ([_P, _I32, _I64, _I64, _P, _P, _P, _P], _I32),
    "qlin_w8a8_gemm_f16": ([_P, _P, _I64, _I64, _I64, _P, _I64, _P, _I64, _P, _P, _P, _I32, _P, _I32, _P], _I32),
    "qlin_nvfp4_global_scale": ([_P, _I32, _I64, _I64, _P, _P], _I32),
    "qlin_arc_perm": ([_P, _I32, _I64, _I64, _P, _P], _I32),
    "qlin_quant_nvfp4": ([_P, _I32, _I64, _I64, _P, _I64, _I32, _P, _P, _P, _I32, _P], _I32),
    "qlin_nvfp4_sf_bytes": ([_I64, _I64, _I32], _I64),
    "qlin_mx_sf_bytes": ([_I64, _I64, _I32], _I64),
    "qlin_hadamard": ([_P, _I32, _I64, _I64, _I32, _I64, _P, _P, _P], _I32),
    "qlin_w4a16_act_order_prepare": ([_P, _I64, _I64, _P, _I64, _P, _P, _P], _I32),
    "qlin_w4a16_gemm_act_order": ([_P, _I64, _I64, _I64, _P, _P, _P, _P, _I64, _P, _P, _P], _I32),
    "qlin_quant_mx": ([_P, _I32, _I64, _I64, _I32, _P, _P, _I32, _P], _I32),
    "qlin_mx_gemm": ([_P, _P, _P, _P, _I64, _I64, _I64, _I32, _P, _I32, _P], _I32),
    "qlin_nvfp4_sf_to_mma": ([_P, _I64, _I64, _P, _P], _I32),
    "qlin_nvfp4_gemm": ([_P, _P, _P, _P, _I64, _I64, _I64, _P, _P, _P, _I32, _P], _I32),
    "qlin_quant_fp8": ([_P, _I32, _I64, _I64, _P, _P, _P], _I32),
    "qlin_fp8_gemm": ([_P, _P, _I64, _I64, _I64, _P, _P, _P, _I32, _P, _I32, _P], _I32),
    "qlin_rmsnorm_quant": ([_P, _I32, _I64, _I64, _P, ctypes.c_float, _I32, _P, _P, _P], _I32),
    "qlin_rmsnorm_quant_nvfp4": ([_P, _I32, _I64, _I64, _P, ctypes.c_float, _P, _I64, _I32, _P, _P, _P, _I32, _P],
                                 _I32),
}

_lib = None


def lib():
    """The loaded libqlin.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError("libqlin.so is not built (run quantized_linear_layer_gb300.build())")
        h = ctypes.CDLL(LIB_PATH)
        for name, (args, res) in _SIGS.items():
            fn = getattr(h, name)
            fn.argtypes = args
            fn.restype = res
        _lib = h
    return _lib


def _torch():
    import torch
    return torch


def _dtype_code(t):
    torch = _torch()
    return {torch.float16: QLIN_F16, torch.bfloat16: QLIN_BF16, torch.float32: QLIN_F32,
            torch.int32: QLIN_I32}[t.dtype]


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    torch = _torch()
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _check(fn, status):
    if status != 0:
        msg = lib().qlin_last_error_message().decode(errors="replace")
        raise QlinError(status, fn, msg)


def _need(t, *dtypes, contiguous=True, name="tensor"):
    if t is None:
        return
    if t.dtype not in dtypes:
        raise TypeError("%s has dtype %s, expected one of %s" % (name, t.dtype, dtypes))
    if contiguous and not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    if not t.is_cuda:
        raise ValueError("%s must be a CUDA tensor" % name)


def qlin_version():
    return lib().qlin_version()


def qlin_get_device_error(stream=None):
    """Reads and clears the device error word; returns the raw code (0 = none)."""
    code = ctypes.c_int32(0)
    st = lib().qlin_get_device_error(_stream(stream), ctypes.byref(code))
    if st not in (0, 5):
        _check("qlin_get_device_error", st)
    return code.value


def qlin_w4a16_gemv_launch_info():
    """(alternating, registers): whether the T = 1 GEMV's two alternating launch
    shapes are in use on the current device, and its registers per thread."""
    alt, regs = ctypes.c_int(0), ctypes.c_int(0)
    _check("qlin_w4a16_gemv_launch_info", lib().qlin_w4a16_gemv_launch_info(ctypes.byref(alt), ctypes.byref(regs)))
    return alt.value, regs.value


def qlin_quant_w4_g128(w, wq, scales, zeros, group=128, stream=None):
    """W [N][K] -> packed codes wq uint8 [N][K/2], fp16 scales [N][K/g], packed zeros uint8 [N][ceil(K/g/2)]."""
    torch = _torch()
    _need(w, torch.float32, torch.float16, torch.bfloat16, name="w")
    _need(wq, torch.uint8, name="wq"); _need(scales, torch.float16, name="scales"); _need(zeros, torch.uint8, name="zeros")
    n, k = w.shape
    _check("qlin_quant_w4_g128", lib().qlin_quant_w4_g128(_ptr(w), _dtype_code(w), n, k, group, _ptr(wq),
                                                         _ptr(scales), _ptr(zeros), _stream(stream)))


def qlin_w4a16_gemm(x, wq, scales, zeros, y, group=128, stream=None):
    """y[T][N] = x[T][K] . dequant(wq, scales, zeros)^T (zeros None = symmetric, z = 8)."""
    torch = _torch()
    _need(x, torch.float16, name="x"); _need(wq, torch.uint8, name="wq"); _need(scales, torch.float16, name="scales")
    _need(zeros, torch.uint8, name="zeros"); _need(y, torch.float16, name="y")
    t, k = x.shape
    n = wq.shape[0]
    _check("qlin_w4a16_gemm", lib().qlin_w4a16_gemm(_ptr(x), t, n, k, _ptr(wq), _ptr(scales), _ptr(zeros), group,
                                                   _ptr(y), _stream(stream)))


def qlin_w4a16_gemm_grouped(x, wqs, scales, zeros, ys, group=128, stream=None):
    """ys[p][T][N_p] = x[T][K] . dequant(wqs[p], scales[p], zeros[p])^T for every p, in one call
    (zeros[p] None = symmetric, z = 8)."""
    torch = _torch()
    count = len(wqs)
    if not (len(scales) == len(zeros) == len(ys) == count):
        raise ValueError("wqs, scales, zeros and ys must have the same length")
    _need(x, torch.float16, name="x")
    for p in range(count):
        _need(wqs[p], torch.uint8, name="wq"); _need(scales[p], torch.float16, name="scales")
        _need(zeros[p], torch.uint8, name="zeros"); _need(ys[p], torch.float16, name="y")
    t, k = x.shape
    n_arr = (ctypes.c_int64 * count)(*[w.shape[0] for w in wqs])
    wq_arr = (ctypes.c_void_p * count)(*[w.data_ptr() for w in wqs])
    s_arr = (ctypes.c_void_p * count)(*[s.data_ptr() for s in scales])
    z_arr = (ctypes.c_void_p * count)(*[0 if z is None else z.data_ptr() for z in zeros])
    y_arr = (ctypes.c_void_p * count)(*[y.data_ptr() for y in ys])
    _check("qlin_w4a16_gemm_grouped", lib().qlin_w4a16_gemm_grouped(
        _ptr(x), t, k, count, n_arr, wq_arr, s_arr, z_arr, group, y_arr, _stream(stream)))


_MAXG = 4  # QLIN_W4A16_MAX_GROUP


class qlin_w4a16_step(ctypes.Structure):
    """One step of qlin_w4a16_gemv_sequence (the C struct of the same name)."""
    _fields_ = [("x", ctypes.c_void_p), ("K", ctypes.c_int64), ("count", ctypes.c_int),
                ("N", ctypes.c_int64 * _MAXG), ("wq", ctypes.c_void_p * _MAXG), ("scales", ctypes.c_void_p * _MAXG),
                ("zeros", ctypes.c_void_p * _MAXG), ("y", ctypes.c_void_p * _MAXG)]


def qlin_w4a16_sequence_workspace_bytes(nsteps):
    return lib().qlin_w4a16_sequence_workspace_bytes(nsteps)


def _w4a16_steps(steps):
    torch = _torch()
    arr = (qlin_w4a16_step * max(1, len(steps)))()
    for i, (x, wqs, scales, zeros, ys) in enumerate(steps):
        _need(x, torch.float16, name="x")
        count = len(wqs)
        if not (1 <= count <= _MAXG and len(scales) == len(zeros) == len(ys) == count):
            raise ValueError("step %d: 1..%d matrices with matching lists expected" % (i, _MAXG))
        st = arr[i]
        st.x = x.data_ptr()
        st.K = x.shape[-1]
        st.count = count
        for p in range(count):
            _need(wqs[p], torch.uint8, name="wq"); _need(scales[p], torch.float16, name="scales")
            _need(zeros[p], torch.uint8, name="zeros"); _need(ys[p], torch.float16, name="y")
            st.N[p] = wqs[p].shape[0]
            st.wq[p] = wqs[p].data_ptr()
            st.scales[p] = scales[p].data_ptr()
            st.zeros[p] = 0 if zeros[p] is None else zeros[p].data_ptr()
            st.y[p] = ys[p].data_ptr()
    return arr


def qlin_w4a16_gemv_sequence(steps, workspace, group=128, stream=None):
    """Run decode steps in order in one persistent launch (T = 1).

    steps: list of (x, wqs, scales, zeros, ys) with x fp16 [1][K] (or [K]) and per-matrix lists as in
    qlin_w4a16_gemm_grouped; workspace: uint8 CUDA tensor of qlin_w4a16_sequence_workspace_bytes(len(steps))
    bytes or more."""
    torch = _torch()
    _need(workspace, torch.uint8, name="workspace")
    arr = _w4a16_steps(steps)
    need = qlin_w4a16_sequence_workspace_bytes(len(steps))
    if workspace.numel() < need:
        raise ValueError("workspace has %d bytes, %d needed" % (workspace.numel(), need))
    _check("qlin_w4a16_gemv_sequence", lib().qlin_w4a16_gemv_sequence(
        ctypes.cast(arr, ctypes.c_void_p), len(steps), group, _ptr(workspace), _stream(stream)))


def qlin_w4a16_gemv_sequence_noalloc(steps, group=128, stream=None):
    """qlin_w4a16_gemv_sequence with the library's own barrier counters (one call in flight per device)."""
    arr = _w4a16_steps(steps)
    _check("qlin_w4a16_gemv_sequence_noalloc", lib().qlin_w4a16_gemv_sequence_noalloc(
        ctypes.cast(arr, ctypes.c_void_p), len(steps), group, _stream(stream)))


def qlin_w4a16_chain(steps, group=128, stream=None):
    """Run W4A16 steps in order at T = x.shape[0] tokens in one call, one launch per step.

    steps: list of (x, wqs, scales, zeros, ys) with x fp16 [T][K] and per-matrix lists as in
    qlin_w4a16_gemm_grouped (ys[p] fp16 [T][N_p])."""
    if not steps:
        return
    t = steps[0][0].shape[0]
    for i, st in enumerate(steps):
        if st[0].dim() != 2 or st[0].shape[0] != t or any(y.shape[0] != t for y in st[4]):
            raise ValueError("step %d: every x and y must be [T][...] with the same T" % i)
    arr = _w4a16_steps(steps)
    _check("qlin_w4a16_chain", lib().qlin_w4a16_chain(ctypes.cast(arr, ctypes.c_void_p), len(steps), t, group,
                                                     _stream(stream)))


class W4A16Chain:
    """The steps of qlin_w4a16_chain marshalled once: run() makes the one C
    call with the stored argument array (no per-call checks or conversions
    in Python).  The array holds the tensors' device pointers, so it is valid
    while they are; the object keeps the tensors referenced."""

    def __init__(self, steps, group=128):
        if not steps:
            raise ValueError("at least one step")
        self._t = _chain_tokens(steps)
        self._arr = _w4a16_steps(steps)
        self._n = len(steps)
        self._group = group
        self._steps = steps

    def run(self, stream=None):
        _check("qlin_w4a16_chain", lib().qlin_w4a16_chain(ctypes.cast(self._arr, ctypes.c_void_p), self._n, self._t,
                                                         self._group, _stream(stream)))


def qlin_w4a16_chain_prepare(steps, group=128):
    """qlin_w4a16_chain's argument array built once, for repeated runs (W4A16Chain.run)."""
    return W4A16Chain(steps, group)


def qlin_w4a16_decode_workspace_bytes(nsteps):
    return lib().qlin_w4a16_decode_workspace_bytes(nsteps)


def _chain_tokens(steps):
    t = steps[0][0].shape[0]
    for i, st in enumerate(steps):
        if st[0].dim() != 2 or st[0].shape[0] != t or any(y.shape[0] != t for y in st[4]):
            raise ValueError("step %d: every x and y must be [T][...] with the same T" % i)
    return t


def qlin_w4a16_decode_prepare(steps, workspace, group=128, stream=None):
    """Write the decode plan of `steps` (as for qlin_w4a16_chain, T = x.shape[0] <= 16) into `workspace`
    (uint8 CUDA tensor of qlin_w4a16_decode_workspace_bytes(len(steps)) bytes or more, 256-byte aligned).
    Returns (nsteps, T) for qlin_w4a16_decode_run."""
    torch = _torch()
    _need(workspace, torch.uint8, name="workspace")
    if not steps:
        raise ValueError("at least one step")
    t = _chain_tokens(steps)
    need = qlin_w4a16_decode_workspace_bytes(len(steps))
    if workspace.numel() < need:
        raise ValueError("workspace has %d bytes, %d needed" % (workspace.numel(), need))
    arr = _w4a16_steps(steps)
    _check("qlin_w4a16_decode_prepare", lib().qlin_w4a16_decode_prepare(
        ctypes.cast(arr, ctypes.c_void_p), len(steps), t, group, _ptr(workspace), _stream(stream)))
    return len(steps), t


def qlin_w4a16_decode_run(workspace, nsteps, T, stream=None):
    """Run a plan written by qlin_w4a16_decode_prepare (nsteps and T as it returned)."""
    _check("qlin_w4a16_decode_run", lib().qlin_w4a16_decode_run(_ptr(workspace), nsteps, T, _stream(stream)))


def qlin_quant_act_int8(x, q, scale, azp=None, stream=None):
    """Per-row int8 quantization of x [T][K]; azp None = symmetric."""
    torch = _torch()
    _need(x, torch.float16, torch.bfloat16, torch.float32, name="x"); _need(q, torch.int8, name="q")
    _need(scale, torch.float32, name="scale"); _need(azp, torch.int32, name="azp")
    t, k = x.shape
    _check("qlin_quant_act_int8", lib().qlin_quant_act_int8(_ptr(x), _dtype_code(x), t, k, _ptr(q), _ptr(scale),
                                                           _ptr(azp), _stream(stream)))


def qlin_quant_act_int8_f16(x, q16, scale, azp=None, stream=None):
    """qlin_quant_act_int8 writing each code as the fp16 number of the same value, q16 [T][K]."""
    torch = _torch()
    _need(x, torch.float16, torch.bfloat16, torch.float32, name="x"); _need(q16, torch.float16, name="q16")
    _need(scale, torch.float32, name="scale"); _need(azp, torch.int32, name="azp")
    t, k = x.shape
    _check("qlin_quant_act_int8_f16", lib().qlin_quant_act_int8_f16(_ptr(x), _dtype_code(x), t, k, _ptr(q16),
                                                                   _ptr(scale), _ptr(azp), _stream(stream)))


def qlin_int8_row_sum(b, azp_adj, stream=None):
    """azp_adj[n] = sum_k b[n, k] for int8 b [N][K]."""
    torch = _torch()
    _need(b, torch.int8, name="b"); _need(azp_adj, torch.int32, name="azp_adj")
    n, k = b.shape
    _check("qlin_int8_row_sum", lib().qlin_int8_row_sum(_ptr(b), n, k, _ptr(azp_adj), _stream(stream)))


def qlin_w8a8_gemm(a, b, scale_a, scale_b, out, azp=None, azp_adj=None, bias=None, stream=None):
    """out = s_a s_b (a . b^T - azp azp_adj) + bias; out int32 gives the raw accumulator."""
    torch = _torch()
    _need(a, torch.int8, name="a"); _need(b, torch.int8, name="b")
    _need(scale_a, torch.float32, name="scale_a"); _need(scale_b, torch.float32, name="scale_b")
    _need(azp, torch.int32, name="azp"); _need(azp_adj, torch.int32, name="azp_adj")
    _need(bias, torch.float16, torch.bfloat16, torch.float32, name="bias")
    _need(out, torch.float16, torch.bfloat16, torch.int32, name="out")
    t, k = a.shape
    n = b.shape[0]
    sa_n = 0 if scale_a is None else scale_a.numel()
    sb_n = 0 if scale_b is None else scale_b.numel()
    bias_dt = QLIN_F16 if bias is None else _dtype_code(bias)
    _check("qlin_w8a8_gemm", lib().qlin_w8a8_gemm(_ptr(a), _ptr(b), t, n, k, _ptr(scale_a), sa_n, _ptr(scale_b), sb_n,
                                                 _ptr(azp), _ptr(azp_adj), _ptr(bias), bias_dt, _ptr(out),
                                                 _dtype_code(out), _stream(stream)))


def qlin_int8_to_f16(src, dst, stream=None):
    """dst = the int8 codes of src as exact fp16 values (the same number of elements)."""
    torch = _torch()
    _need(src, torch.int8, name="src"); _need(dst, torch.float16, name="dst")
    if src.numel() != dst.numel():
        raise ValueError("src and dst must have the same number of elements")
    _check("qlin_int8_to_f16", lib().qlin_int8_to_f16(_ptr(src), src.numel(), _ptr(dst), _stream(stream)))


def qlin_w8a8_gemm_f16b(a, b16, scale_a, scale_b, out, azp=None, azp_adj=None, bias=None, stream=None):
    """qlin_w8a8_gemm with the weight codes as exact fp16 values b16 [N][K] (qlin_int8_to_f16)."""
    torch = _torch()
    _need(a, torch.int8, name="a"); _need(b16, torch.float16, name="b16")
    _need(scale_a, torch.float32, name="scale_a"); _need(scale_b, torch.float32, name="scale_b")
    _need(azp, torch.int32, name="azp"); _need(azp_adj, torch.int32, name="azp_adj")
    _need(bias, torch.float16, torch.bfloat16, torch.float32, name="bias")
    _need(out, torch.float16, torch.bfloat16, torch.int32, name="out")
    t, k = a.shape
    n = b16.shape[0]
    sa_n = 0 if scale_a is None else scale_a.numel()
    sb_n = 0 if scale_b is None else scale_b.numel()
    bias_dt = QLIN_F16 if bias is None else _dtype_code(bias)
    _check("qlin_w8a8_gemm_f16b", lib().qlin_w8a8_gemm_f16b(_ptr(a), _ptr(b16), t, n, k, _ptr(scale_a), sa_n,
                                                           _ptr(scale_b), sb_n, _ptr(azp), _ptr(azp_adj), _ptr(bias),
                                                           bias_dt, _ptr(out), _dtype_code(out), _stream(stream)))


def qlin_w8a8_gemm_f16(a16, b16, scale_a, scale_b, out, azp=None, azp_adj=None, bias=None, stream=None):
    """qlin_w8a8_gemm with both operands' codes as exact fp16 values: a16 [T][K]
    (qlin_quant_act_int8_f16) and b16 [N][K] (qlin_int8_to_f16)."""
    torch = _torch()
    _need(a16, torch.float16, name="a16"); _need(b16, torch.float16, name="b16")
    _need(scale_a, torch.float32, name="scale_a"); _need(scale_b, torch.float32, name="scale_b")
    _need(azp, torch.int32, name="azp"); _need(azp_adj, torch.int32, name="azp_adj")
    _need(bias, torch.float16, torch.bfloat16, torch.float32, name="bias")
    _need(out, torch.float16, torch.bfloat16, torch.int32, name="out")
    t, k = a16.shape
    n = b16.shape[0]
    sa_n = 0 if scale_a is None else scale_a.numel()
    sb_n = 0 if scale_b is None else scale_b.numel()
    bias_dt = QLIN_F16 if bias is None else _dtype_code(bias)
    _check("qlin_w8a8_gemm_f16", lib().qlin_w8a8_gemm_f16(_ptr(a16), _ptr(b16), t, n, k, _ptr(scale_a), sa_n,
                                                         _ptr(scale_b), sb_n, _ptr(azp), _ptr(azp_adj), _ptr(bias),
                                                         bias_dt, _ptr(out), _dtype_code(out), _stream(stream)))


def qlin_nvfp4_global_scale(x, g, stream=None):
    """g[0] = max|x| / (6 * 448)."""
    torch = _torch()
    _need(x, torch.float16, torch.bfloat16, torch.float32, name="x"); _need(g, torch.float32, name="g")
    rows, k = x.shape
    _check("qlin_nvfp4_global_scale", lib().qlin_nvfp4_global_scale(_ptr(x), _dtype_code(x), rows, k, _ptr(g),
                                                                   _stream(stream)))


def qlin_arc_perm(x, perm, stream=None):
    """perm = channels by descending max|x| over rows (ties: lower index first)."""
    torch = _torch()
    _need(x, torch.float16, torch.bfloat16, torch.float32, name="x"); _need(perm, torch.int32, name="perm")
    rows, k = x.shape
    _check("qlin_arc_perm", lib().qlin_arc_perm(_ptr(x), _dtype_code(x), rows, k, _ptr(perm), _stream(stream)))


def qlin_nvfp4_sf_bytes(rows, K, sf_layout=QLIN_SF_ROWS):
    """Bytes of an E4M3 scale buffer for rows x K elements in the given layout."""
    return lib().qlin_nvfp4_sf_bytes(rows, K, sf_layout)


def qlin_nvfp4_sf_to_mma(sf_rows, sf_mma, stream=None):
    """Row-major scales uint8 [rows][K/16] -> the QLIN_SF_MMA layout (1-D uint8)."""
    torch = _torch()
    _need(sf_rows, torch.uint8, name="sf_rows"); _need(sf_mma, torch.uint8, name="sf_mma")
    rows, kb = sf_rows.shape
    if sf_mma.numel() < qlin_nvfp4_sf_bytes(rows, kb * 16, QLIN_SF_MMA):
        raise ValueError("sf_mma buffer too small")
    _check("qlin_nvfp4_sf_to_mma", lib().qlin_nvfp4_sf_to_mma(_ptr(sf_rows), rows, kb * 16, _ptr(sf_mma),
                                                             _stream(stream)))


def qlin_quant_nvfp4(x, g, q, sf, perm=None, S=0, mode=QLIN_NVFP4_RESIDUAL, sf_layout=QLIN_SF_ROWS, stream=None):
    """NVFP4 codes q uint8 [rows][(K+S)/2] and E4M3 scales sf (uint8 [rows][(K+S)/16]
    for QLIN_SF_ROWS, or a 1-D buffer of qlin_nvfp4_sf_bytes(rows, K+S, QLIN_SF_MMA))."""
    torch = _torch()
    _need(x, torch.float16, torch.bfloat16, torch.float32, name="x"); _need(g, torch.float32, name="g")
    _need(q, torch.uint8, name="q"); _need(sf, torch.uint8, name="sf"); _need(perm, torch.int32, name="perm")
    rows, k = x.shape
    if sf.numel() < qlin_nvfp4_sf_bytes(rows, k + S, sf_layout):
        raise ValueError("sf buffer too small")
    _check("qlin_quant_nvfp4", lib().qlin_quant_nvfp4(_ptr(x), _dtype_code(x), rows, k, _ptr(perm), S, mode, _ptr(g),
                                                     _ptr(q), _ptr(sf), sf_layout, _stream(stream)))


def qlin_nvfp4_gemm(a, sfa, b, sfb, g_a, g_b, out, stream=None):
    """out[T][N] = g_a g_b (dequant(a, sfa) . dequant(b, sfb)^T); sfa, sfb in the QLIN_SF_MMA layout."""
    torch = _torch()
    for t_, nm in ((a, "a"), (sfa, "sfa"), (b, "b"), (sfb, "sfb")):
        _need(t_, torch.uint8, name=nm)
    _need(g_a, torch.float32, name="g_a"); _need(g_b, torch.float32, name="g_b")
    _need(out, torch.bfloat16, torch.float16, name="out")
    t = a.shape[0]
    k = a.shape[1] * 2
    n = b.shape[0]
    _check("qlin_nvfp4_gemm", lib().qlin_nvfp4_gemm(_ptr(a), _ptr(sfa), _ptr(b), _ptr(sfb), t, n, k, _ptr(g_a),
                                                   _ptr(g_b), _ptr(out), _dtype_code(out), _stream(stream)))


def qlin_quant_fp8(x, q, scale, stream=None):
    """Per-row FP8 E4M3 quantization of x [rows][K]: q uint8 [rows][K] (E4M3-FN
    codes), scale float32 [rows] = max|x| / 448 per row."""
    torch = _torch()
    _need(x, torch.float16, torch.bfloat16, torch.float32, name="x"); _need(q, torch.uint8, name="q")
    _need(scale, torch.float32, name="scale")
    rows, k = x.shape
    _check("qlin_quant_fp8", lib().qlin_quant_fp8(_ptr(x), _dtype_code(x), rows, k, _ptr(q), _ptr(scale),
                                                 _stream(stream)))


def qlin_fp8_gemm(a, b, scale_a, scale_b, out, bias=None, stream=None):
    """out [T][N] = scale_a[t] scale_b[n] (dec(a) . dec(b)^T) + bias for E4M3 codes
    a uint8 [T][K], b uint8 [N][K]; out fp16 or bf16."""
    torch = _torch()
    _need(a, torch.uint8, name="a"); _need(b, torch.uint8, name="b")
    _need(scale_a, torch.float32, name="scale_a"); _need(scale_b, torch.float32, name="scale_b")
    _need(bias, torch.float16, torch.bfloat16, torch.float32, name="bias")
    _need(out, torch.float16, torch.bfloat16, name="out")
    t, k = a.shape
    n = b.shape[0]
    bias_dt = QLIN_F16 if bias is None else _dtype_code(bias)
    _check("qlin_fp8_gemm", lib().qlin_fp8_gemm(_ptr(a), _ptr(b), t, n, k, _ptr(scale_a), _ptr(scale_b), _ptr(bias),
                                               bias_dt, _ptr(out), _dtype_code(out), _stream(stream)))


def qlin_rmsnorm_quant(x, gamma, eps, q, scale, fmt=QLIN_QFMT_INT8, stream=None):
    """y = (x . (1 / sqrt(mean(x^2) + eps))) . gamma per row of x [rows][K], quantized
    per token: q int8 (QLIN_QFMT_INT8) or uint8 E4M3 codes (QLIN_QFMT_FP8_E4M3)
    [rows][K], scale float32 [rows]."""
    torch = _torch()
    _need(x, torch.float16, torch.bfloat16, torch.float32, name="x")
    _need(gamma, x.dtype, name="gamma")
    _need(q, torch.int8 if fmt == QLIN_QFMT_INT8 else torch.uint8, name="q")
    _need(scale, torch.float32, name="scale")
    rows, k = x.shape
    _check("qlin_rmsnorm_quant", lib().qlin_rmsnorm_quant(_ptr(x), _dtype_code(x), rows, k, _ptr(gamma), float(eps),
                                                         fmt, _ptr(q), _ptr(scale), _stream(stream)))


def qlin_rmsnorm_quant_nvfp4(x, gamma, eps, g, q, sf, perm=None, S=0, mode=QLIN_NVFP4_RESIDUAL,
                             sf_layout=QLIN_SF_ROWS, stream=None):
    """y = (x . (1 / sqrt(mean(x^2) + eps))) . gamma per row of x [rows][K], then the
    NVFP4 quantization of y as qlin_quant_nvfp4 does it (g and perm calibrated on y)."""
    torch = _torch()
    _need(x, torch.float16, torch.bfloat16, torch.float32, name="x")
    _need(gamma, x.dtype, name="gamma"); _need(g, torch.float32, name="g")
    _need(q, torch.uint8, name="q"); _need(sf, torch.uint8, name="sf"); _need(perm, torch.int32, name="perm")
    rows, k = x.shape
    if sf.numel() < qlin_nvfp4_sf_bytes(rows, k + S, sf_layout):
        raise ValueError("sf buffer too small")
    _check("qlin_rmsnorm_quant_nvfp4",
           lib().qlin_rmsnorm_quant_nvfp4(_ptr(x), _dtype_code(x), rows, k, _ptr(gamma), float(eps), _ptr(perm), S,
                                          mode, _ptr(g), _ptr(q), _ptr(sf), sf_layout, _stream(stream)))


def qlin_mx_sf_bytes(rows, K, sf_layout=QLIN_SF_ROWS):
    """Bytes of an MX (E8M0) scale buffer for `rows` rows of K elements, -1 if K % 32."""
    return lib().qlin_mx_sf_bytes(rows, K, sf_layout)


def qlin_quant_mx(x, q, sf, fmt=QLIN_MX_FP8_E4M3, sf_layout=QLIN_SF_ROWS, stream=None):
    """MXFP8 / MXFP4 quantization of x [rows][K]: q uint8 [rows][K] (E4M3) or
    [rows][K/2] (packed E2M1), sf uint8 E8M0 scales (one per 32 elements) in sf_layout."""
    torch = _torch()
    _need(x, torch.float16, torch.bfloat16, torch.float32, name="x")
    _need(q, torch.uint8, name="q"); _need(sf, torch.uint8, name="sf")
    rows, k = x.shape
    if q.numel() < rows * (k if fmt == QLIN_MX_FP8_E4M3 else k // 2):
        raise ValueError("q buffer too small")
    if sf.numel() < qlin_mx_sf_bytes(rows, k, sf_layout):
        raise ValueError("sf buffer too small")
    _check("qlin_quant_mx", lib().qlin_quant_mx(_ptr(x), _dtype_code(x), rows, k, fmt, _ptr(q), _ptr(sf), sf_layout,
                                               _stream(stream)))


def qlin_mx_gemm(a, sfa, b, sfb, out, fmt=QLIN_MX_FP8_E4M3, stream=None):
    """out[T][N] = dequant(a, sfa) . dequant(b, sfb)^T for MX codes a [T][..], b [N][..]
    and E8M0 scales in the QLIN_SF_MMA layout; out fp16 or bf16."""
    torch = _torch()
    for t_, nm in ((a, "a"), (sfa, "sfa"), (b, "b"), (sfb, "sfb")):
        _need(t_, torch.uint8, name=nm)
    _need(out, torch.bfloat16, torch.float16, name="out")
    t, n = a.shape[0], b.shape[0]
    k = a.shape[1] * (1 if fmt == QLIN_MX_FP8_E4M3 else 2)
    if b.shape[1] != a.shape[1]:
        raise ValueError("a and b must have the same K")
    if sfa.numel() < qlin_mx_sf_bytes(t, k, QLIN_SF_MMA) or sfb.numel() < qlin_mx_sf_bytes(n, k, QLIN_SF_MMA):
        raise ValueError("scale buffers too small for the QLIN_SF_MMA layout")
    if out.shape[0] != t or out.shape[1] != n:
        raise ValueError("out must be [T][N]")
    _check("qlin_mx_gemm", lib().qlin_mx_gemm(_ptr(a), _ptr(sfa), _ptr(b), _ptr(sfb), t, n, k, fmt, _ptr(out),
                                             _dtype_code(out), _stream(stream)))


def qlin_w4a16_act_order_prepare(g_idx, wq, perm, wq_sorted, group=128, stream=None):
    """Offline act-order preparation: perm int32 [K] (the columns in group order)
    and wq_sorted uint8 [N][K/2] (the packed codes in that order) from g_idx
    int32 [K] and wq uint8 [N][K/2]."""
    torch = _torch()
    _need(g_idx, torch.int32, name="g_idx"); _need(wq, torch.uint8, name="wq")
    _need(perm, torch.int32, name="perm"); _need(wq_sorted, torch.uint8, name="wq_sorted")
    k = g_idx.numel()
    n = wq.shape[0]
    if perm.numel() != k or tuple(wq_sorted.shape) != tuple(wq.shape) or wq.shape[1] * 2 != k:
        raise ValueError("shape mismatch between g_idx, wq, perm and wq_sorted")
    _check("qlin_w4a16_act_order_prepare",
           lib().qlin_w4a16_act_order_prepare(_ptr(g_idx), k, group, _ptr(wq), n, _ptr(perm), _ptr(wq_sorted),
                                              _stream(stream)))


def qlin_w4a16_gemm_act_order(x, perm, wq_sorted, scales, zeros, y, x_work=None, group=128, stream=None):
    """y [T][N] = x . dequant(W)^T for act-order weights prepared by
    qlin_w4a16_act_order_prepare; x_work fp16 [T][K] workspace (allocated here if None)."""
    torch = _torch()
    _need(x, torch.float16, name="x"); _need(perm, torch.int32, name="perm")
    _need(wq_sorted, torch.uint8, name="wq_sorted"); _need(scales, torch.float16, name="scales")
    _need(zeros, torch.uint8, name="zeros"); _need(y, torch.float16, name="y")
    if x_work is None:
        x_work = torch.empty_like(x)
    _need(x_work, torch.float16, name="x_work")
    t, k = x.shape
    n = wq_sorted.shape[0]
    if x_work.shape != x.shape or perm.numel() != k or wq_sorted.shape[1] * 2 != k or tuple(y.shape) != (t, n):
        raise ValueError("shape mismatch")
    _check("qlin_w4a16_gemm_act_order",
           lib().qlin_w4a16_gemm_act_order(_ptr(x), t, n, k, _ptr(perm), _ptr(wq_sorted), _ptr(scales), _ptr(zeros),
                                           group, _ptr(x_work), _ptr(y), _stream(stream)))


def qlin_hadamard(x, n, y=None, kind=QLIN_HADAMARD_SYLVESTER, signs=None, stream=None):
    """Rotates every group of n consecutive elements of the rows of x [rows][K]
    (Sylvester fast Walsh-Hadamard or the regular Hadamard of order 4^k), scaled by
    1/sqrt(n) and multiplied by signs (int8 [K] of +-1) if given; y defaults to a new
    tensor (y = x rotates in place)."""
    torch = _torch()
    _need(x, torch.float16, torch.bfloat16, torch.float32, name="x"); _need(signs, torch.int8, name="signs")
    if y is None:
        y = torch.empty_like(x)
    _need(y, x.dtype, name="y")
    rows, k = x.shape
    if y.shape != x.shape or (signs is not None and signs.numel() != k):
        raise ValueError("shape mismatch")
    _check("qlin_hadamard", lib().qlin_hadamard(_ptr(x), _dtype_code(x), rows, k, kind, n, _ptr(signs), _ptr(y),
                                               _stream(stream)))
    return y
