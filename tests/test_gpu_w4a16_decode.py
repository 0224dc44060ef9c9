"""The W4A16 decode plan (qlin_w4a16_decode_prepare / _run: a chain of
decode steps at 1 .. 16 tokens in one persistent launch) against the CPU
oracle.  Every step writes its own buffers, so each step's output is checked
against the oracle on the input that step actually read (the previous
step's fp16 output, read back from the GPU): max |err| <= 1e-2 (1 + |ref|)
and relative Frobenius error <= 2e-3 per step."""

import numpy as np
import pytest
import torch

import oracle
from quantized_linear_layer_gb300 import inputs
from conftest import assert_within_tolerance

pytestmark = pytest.mark.gpu


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def _quantized(seed, n, k):
    d = inputs.w4a16_decode(seed=seed, T=1, N=n, K=k)
    return oracle.quant_w4_g128(d["w"])


def _dev_mat(m, symmetric=False):
    codes, s16, z = m
    return (_dev(oracle.pack_u4(codes)), _dev(s16), None if symmetric else _dev(oracle.pack_u4(z)))


def _workspace(q, nsteps):
    return torch.zeros(q.qlin_w4a16_decode_workspace_bytes(nsteps), dtype=torch.uint8, device="cuda")


def _run(q, steps, runs=1):
    ws = _workspace(q, len(steps))
    n, t = q.qlin_w4a16_decode_prepare(steps, ws)
    for _ in range(runs):
        q.qlin_w4a16_decode_run(ws, n, t)
    torch.cuda.synchronize()
    assert q.qlin_get_device_error() == 0
    return ws


def _check_steps(steps, mats, what):
    """Each step's outputs against the oracle on the step's own (GPU) input."""
    for i, ((x, _w, _s, _z, ys), ms) in enumerate(zip(steps, mats)):
        xin = x.cpu().numpy()
        for p, (y, (codes, s16, z, sym)) in enumerate(zip(ys, ms)):
            zz = np.full_like(z, 8) if sym else z
            ref = oracle.w4a16_reference(xin, codes, s16, zz)
            assert_within_tolerance(y.cpu().numpy(), ref, "%s step %d matrix %d" % (what, i, p))


def _decoder_steps(T, hid, inter, kv, nblocks, seed, symmetric_v=False):
    """nblocks decoder blocks with their dependencies (q,k,v on the block
    input; o on v; gate,up on o; down on up; the next block on down), every
    output in a buffer of its own (filled with NaN first)."""
    x0 = inputs.w4a16_decode(seed=seed, T=T, N=8, K=hid)["x"]
    h = _dev(x0)
    steps, mats = [], []
    for b in range(nblocks):
        blk = {}
        for name, (n, k) in (("q", (hid, hid)), ("k", (kv, hid)), ("v", (kv, hid)), ("o", (hid, kv)),
                             ("gate", (inter, hid)), ("up", (inter, hid)), ("down", (hid, inter))):
            blk[name] = _quantized(seed + 1, n, k)
            seed += 1
        sym = {n: (symmetric_v and b == 0 and n == "v") for n in blk}
        dev = {n: _dev_mat(blk[n], sym[n]) for n in blk}
        out = {n: torch.full((T, blk[n][0].shape[0]), float("nan"), dtype=torch.float16, device="cuda") for n in blk}
        groups = [("q", "k", "v"), ("o",), ("gate", "up"), ("down",)]
        inputs_of = {("q", "k", "v"): h, ("o",): out["v"], ("gate", "up"): out["o"], ("down",): out["up"]}
        for grp in groups:
            steps.append((inputs_of[grp], [dev[n][0] for n in grp], [dev[n][1] for n in grp], [dev[n][2] for n in grp],
                          [out[n] for n in grp]))
            mats.append([(*blk[n], sym[n]) for n in grp])
        h = out["down"]
    return steps, mats


@pytest.mark.parametrize("T", [1, 2, 3, 8, 9, 16])
def test_decoder_blocks_small(qlin_gpu, T):
    """Two small decoder blocks (hidden 1024: one K chunk with half the warps
    idle; intermediate 2816: two chunks, the second of 6 groups; k and v of
    256 rows), the first block's v symmetric (no zero-points)."""
    steps, mats = _decoder_steps(T, 1024, 2816, 256, 2, 500 + T, symmetric_v=True)
    _run(qlin_gpu, steps)
    _check_steps(steps, mats, "T=%d" % T)


@pytest.mark.parametrize("T", [1, 4, 16])
def test_llama_block_full_size(qlin_gpu, T):
    """One Llama-2-7B-shaped block (4096 / 11008, the bench's layer shapes and
    launch configuration) at the bench's token counts, every output checked."""
    steps, mats = _decoder_steps(T, 4096, 11008, 4096, 1, 900 + T)
    _run(qlin_gpu, steps)
    _check_steps(steps, mats, "llama T=%d" % T)


@pytest.mark.parametrize("T", [1, 5, 16])
def test_ragged_shapes(qlin_gpu, T):
    """Heights that are not multiples of the 32-row unit (200, 5 and 48 rows)
    with an empty matrix in the group, K = 2176 (a second chunk holding a
    single group), then a step of one row with K = 128 (one group) and no
    zero-points; most CTAs have no rows in these steps."""
    x0 = inputs.w4a16_decode(seed=40 + T, T=T, N=8, K=2176)["x"]
    ms = [_quantized(41, 200, 2176), _quantized(42, 5, 2176), _quantized(43, 48, 2176)]
    dev = [_dev_mat(m) for m in ms]
    ys = [torch.full((T, m[0].shape[0]), float("nan"), dtype=torch.float16, device="cuda") for m in ms]
    e_wq = torch.empty((0, 2176 // 2), dtype=torch.uint8, device="cuda")
    e_sc = torch.empty((0, 17), dtype=torch.float16, device="cuda")
    e_zp = torch.empty((0, 9), dtype=torch.uint8, device="cuda")
    y_empty = torch.empty((T, 0), dtype=torch.float16, device="cuda")
    x = _dev(x0)
    step0 = (x, [dev[0][0], e_wq, dev[1][0], dev[2][0]], [dev[0][1], e_sc, dev[1][1], dev[2][1]],
             [dev[0][2], e_zp, dev[1][2], dev[2][2]], [ys[0], y_empty, ys[1], ys[2]])
    m3 = _quantized(45, 1, 128)
    d3 = _dev_mat(m3, symmetric=True)
    y3 = torch.full((T, 1), float("nan"), dtype=torch.float16, device="cuda")
    x3 = _dev(inputs.w4a16_decode(seed=46, T=T, N=8, K=128)["x"])
    _run(qlin_gpu, [step0, (x3, [d3[0]], [d3[1]], [d3[2]], [y3])])
    _check_steps([(x, None, None, None, ys)], [[(*m, False) for m in ms]], "ragged T=%d" % T)
    _check_steps([(x3, None, None, None, [y3])], [[(*m3, True)]], "K=128 T=%d" % T)


def test_runs_repeat_bit_for_bit(qlin_gpu):
    """A plan runs any number of times (its counters return to zero after
    every run) and gives the same bits each time, also after it is prepared
    again."""
    steps, mats = _decoder_steps(4, 1024, 2816, 256, 2, 610)
    ws = _run(qlin_gpu, steps)
    first = [y.clone() for st in steps for y in st[4]]
    for _ in range(3):
        qlin_gpu.qlin_w4a16_decode_run(ws, len(steps), 4)
    torch.cuda.synchronize()
    assert qlin_gpu.qlin_get_device_error() == 0
    assert all(torch.equal(a, y) for a, y in zip(first, [y for st in steps for y in st[4]]))
    _run(qlin_gpu, steps, runs=2)
    assert all(torch.equal(a, y) for a, y in zip(first, [y for st in steps for y in st[4]]))
    _check_steps(steps, mats, "repeat")


def test_many_steps_ping_pong(qlin_gpu):
    """150 chained steps, K = 1408 (11 groups: scale rows not 16-byte
    aligned), scales raised so that the activations keep their size along the
    chain.  Run once with a buffer per step (every step against the oracle on
    its GPU input) and once on two ping-pong buffers, where each step also
    overwrites what the step before it read: the last output must be the
    same bits."""
    T, width, n_steps = 2, 1408, 150
    mats = []
    for i in range(n_steps):
        codes, s16, z = _quantized(300 + i, width, width)
        mats.append((codes, (s16.astype(np.float32) * 1.33).astype(np.float16), z))
    dev = [_dev_mat(m) for m in mats]
    x0 = _dev(inputs.w4a16_decode(seed=299, T=T, N=8, K=width)["x"])
    outs = [torch.full((T, width), float("nan"), dtype=torch.float16, device="cuda") for _ in range(n_steps)]
    steps = [((x0 if i == 0 else outs[i - 1]), [d[0]], [d[1]], [d[2]], [outs[i]]) for i, d in enumerate(dev)]
    _run(qlin_gpu, steps)
    mag = [float(o.float().abs().mean()) for o in (outs[0], outs[-1])]
    assert 0.1 < mag[1] / mag[0] < 10, mag
    _check_steps(steps, [[(*m, False)] for m in mats], "150 steps")
    bufs = [x0.clone(), torch.empty((T, width), dtype=torch.float16, device="cuda")]
    pp = [(bufs[i % 2], [d[0]], [d[1]], [d[2]], [bufs[(i + 1) % 2]]) for i, d in enumerate(dev)]
    _run(qlin_gpu, pp)
    assert torch.equal(bufs[n_steps % 2], outs[-1])


@pytest.mark.parametrize("scale", [1e3, 3e4])
def test_activation_outliers(qlin_gpu, scale):
    """Activations with a few channels scaled by 1e3 and 3e4 (fp16 stays
    finite): the exact fp16 (q - z) MMA path keeps every product exact."""
    T = 9
    d = inputs.w4a16_decode(seed=77, T=T, N=8, K=4096)
    x = d["x"].astype(np.float32)
    idx = np.random.default_rng(5).choice(4096, 41, replace=False)
    x[:, idx] *= scale
    x = np.clip(x, -60000, 60000).astype(np.float16)
    m = _quantized(78, 4096, 4096)
    dm = _dev_mat(m)
    y = torch.full((T, 4096), float("nan"), dtype=torch.float16, device="cuda")
    steps = [(_dev(x), [dm[0]], [dm[1]], [dm[2]], [y])]
    _run(qlin_gpu, steps)
    _check_steps(steps, [[(*m, False)]], "outliers x%g" % scale)


def test_rejects_unsupported(qlin_gpu):
    steps, _ = _decoder_steps(1, 512, 1024, 128, 1, 5)
    ws = _workspace(qlin_gpu, len(steps))
    # 17 tokens
    x17 = torch.zeros((17, 512), dtype=torch.float16, device="cuda")
    y17 = torch.zeros((17, 512), dtype=torch.float16, device="cuda")
    bad = [(x17, steps[0][1][:1], steps[0][2][:1], steps[0][3][:1], [y17])]
    with pytest.raises(qlin_gpu.QlinError):
        qlin_gpu.qlin_w4a16_decode_prepare(bad, ws)
    # a misaligned workspace
    big = torch.zeros(ws.numel() + 256, dtype=torch.uint8, device="cuda")
    with pytest.raises(qlin_gpu.QlinError):
        qlin_gpu.qlin_w4a16_decode_prepare(steps, big[16:])
