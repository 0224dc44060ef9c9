"""The W4A16 decode sequence entry point that allocates nothing.

Some callers cannot allocate device memory where they run the decoder: an
inference runtime that loads this library as a plugin and gives it neither an
allocator nor a workspace, or a serving engine that reserved almost all of
HBM up front and lets nothing else call cudaMalloc.  For them the library
keeps the grid barrier's counters in a fixed static device array, and
qlin_w4a16_gemv_sequence_noalloc takes only the inputs and outputs.

This file is collected last on purpose: if it fails, a run that stops at the
first failure has already run every other test.  It passes on its own in a
fresh process as well as after the other tests (the first call on a device
looks up the array's address; later calls reuse it)."""

import numpy as np
import pytest
import torch

import oracle
from quantized_linear_layer_gb300 import inputs
from conftest import assert_within_tolerance

pytestmark = pytest.mark.gpu

WIDTH = 1408          # K = N: 11 groups of 128, rows that do not fill a stage evenly
STEPS = 140           # longer than one launch (128 steps): the counters are reused


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def _chain(seed0):
    mats = []
    for i in range(STEPS):
        d = inputs.w4a16_decode(seed=seed0 + i, T=1, N=WIDTH, K=WIDTH)
        mats.append(oracle.quant_w4_g128(d["w"]))
    x0 = inputs.w4a16_decode(seed=seed0 - 1, T=1, N=8, K=WIDTH)["x"]
    return mats, x0


def _run(q, dev_mats, x0, entry):
    """The chain on ping-pong buffers: step i reads buffer i % 2 and writes
    the other; returns the last output."""
    bufs = [_dev(x0), torch.empty((1, WIDTH), dtype=torch.float16, device="cuda")]
    steps = [(bufs[i % 2], [wq], [sc], [zp], [bufs[(i + 1) % 2]]) for i, (wq, sc, zp) in enumerate(dev_mats)]
    entry(steps)
    torch.cuda.synchronize()
    assert q.qlin_get_device_error() == 0
    return bufs[len(dev_mats) % 2].cpu().numpy()


def test_noalloc_sequence_matches_workspace_entry_point(qlin_gpu):
    q = qlin_gpu
    mats, x0 = _chain(seed0=400)
    dev_mats = [(_dev(oracle.pack_u4(c)), _dev(s), _dev(oracle.pack_u4(z))) for (c, s, z) in mats]

    def with_workspace(steps):
        ws = torch.zeros(q.qlin_w4a16_sequence_workspace_bytes(len(steps)), dtype=torch.uint8, device="cuda")
        q.qlin_w4a16_gemv_sequence(steps, ws)

    ref = _run(q, dev_mats, x0, with_workspace)

    # two calls in a row: the second finds the counters the first one left
    # behind and must zero them before use
    for call in range(2):
        y = _run(q, dev_mats, x0, q.qlin_w4a16_gemv_sequence_noalloc)
        assert_within_tolerance(y, ref.astype(np.float64), "no-alloc call %d vs workspace entry point" % call)
        assert np.array_equal(y, ref), "call %d: outputs differ from the workspace entry point" % call

    # two steps against the oracle, so that the comparison above is anchored
    # to the definition and not only to the other entry point: step 2 reads
    # step 1's output (buffer 1) and writes buffer 0
    bufs = [_dev(x0), torch.empty((1, WIDTH), dtype=torch.float16, device="cuda")]
    steps = [(bufs[i % 2], [wq], [sc], [zp], [bufs[(i + 1) % 2]]) for i, (wq, sc, zp) in enumerate(dev_mats[:2])]
    q.qlin_w4a16_gemv_sequence_noalloc(steps)
    torch.cuda.synchronize()
    assert q.qlin_get_device_error() == 0
    c, s16, z = mats[1]
    ref2 = oracle.w4a16_reference(bufs[1].cpu().numpy(), c, s16, z)
    assert_within_tolerance(bufs[0].cpu().numpy(), ref2, "no-alloc step 2 vs oracle")
