"""W4A16 on the GPU against the CPU oracle: the a0 weight quantizer bit for
bit, and the fused dequant GEMV / skinny GEMM within the fp16 tolerance, on
the tiny symmetric workload and on the Llama-2-7B-shaped decode layers."""

import numpy as np
import pytest
import torch

import oracle
from quantized_linear_layer_gb300 import inputs
from conftest import assert_within_tolerance

pytestmark = pytest.mark.gpu


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def _gpu_quant_w4(q, w):
    n, k = w.shape
    wq = torch.empty((n, k // 2), dtype=torch.uint8, device="cuda")
    sc = torch.empty((n, k // 128), dtype=torch.float16, device="cuda")
    zp = torch.empty((n, (k // 128 + 1) // 2), dtype=torch.uint8, device="cuda")
    q.qlin_quant_w4_g128(_dev(w), wq, sc, zp)
    return wq, sc, zp


def _gemm(q, x, wq, sc, zp):
    y = torch.empty((x.shape[0], wq.shape[0]), dtype=torch.float16, device="cuda")
    q.qlin_w4a16_gemm(x, wq, sc, zp, y)
    torch.cuda.synchronize()
    assert q.qlin_get_device_error() == 0
    return y.cpu().numpy()


def test_tiny_symmetric(qlin_gpu):
    d = inputs.tiny_w4a16(seed=0)
    ref = oracle.w4a16_reference(d["x"], d["codes"], d["scales"], None)
    y = _gemm(qlin_gpu, _dev(d["x"]), _dev(oracle.pack_u4(d["codes"])), _dev(d["scales"]), None)
    assert_within_tolerance(y, ref, "tiny W4A16")


@pytest.mark.parametrize("T", [1, 2, 5, 8, 9, 16, 24, 33, 64])
def test_token_counts_ragged_rows(qlin_gpu, T):
    # N = 200 is not a multiple of the 16-row tile; every code and zero-point occurs
    d = inputs.w4a16_decode(seed=17, T=T, N=200, K=640)
    codes, s16, z = oracle.quant_w4_g128(d["w"])
    ref = oracle.w4a16_reference(d["x"], codes, s16, z)
    y = _gemm(qlin_gpu, _dev(d["x"]), _dev(oracle.pack_u4(codes)), _dev(s16), _dev(oracle.pack_u4(z)))
    assert_within_tolerance(y, ref, "W4A16 T=%d" % T)


def test_all_codes_and_zero_points_exact(qlin_gpu):
    """Every (code, zero-point) pair: with one-hot activations the GEMV
    returns s * (q - z) itself, which is exact in fp16 for these scales."""
    n, k = 256, 128
    codes = np.tile(np.arange(16, dtype=np.uint8), (n, k // 16))
    zeros = (np.arange(n, dtype=np.uint8) % 16).reshape(n, 1)
    scales = np.full((n, 1), 0.25, dtype=np.float16)
    wq, sc, zp = _dev(oracle.pack_u4(codes)), _dev(scales), _dev(oracle.pack_u4(zeros))
    for kk in range(0, 16):
        x = np.zeros((1, k), dtype=np.float16)
        x[0, kk] = 1.0
        y = _gemm(qlin_gpu, _dev(x), wq, sc, zp)
        expect = 0.25 * (kk - zeros[:, 0].astype(np.float64))
        assert np.array_equal(y[0].astype(np.float64), expect)


def test_weight_quantizer_bit_exact(qlin_gpu):
    d = inputs.w4a16_decode(seed=3, T=1, N=300, K=1152)   # odd group count (9)
    w = d["w"].copy()
    w[5, :128] = 0.0                                        # a flat group: range floor
    w[7, 128:256] = np.abs(w[7, 128:256])                   # a group that does not straddle 0
    codes, s16, z = oracle.quant_w4_g128(w)
    wq, sc, zp = _gpu_quant_w4(qlin_gpu, w)
    assert np.array_equal(wq.cpu().numpy(), oracle.pack_u4(codes))
    assert np.array_equal(sc.cpu().numpy().view(np.uint16), s16.view(np.uint16))
    assert np.array_equal(zp.cpu().numpy(), oracle.pack_u4(z))


@pytest.mark.parametrize("N,K", inputs.LLAMA2_7B_LAYERS)
def test_llama_decode_layers(qlin_gpu, N, K):
    d = inputs.w4a16_decode(seed=1, T=16, N=N, K=K)
    codes, s16, z = oracle.quant_w4_g128(d["w"])
    wq, sc, zp = _gpu_quant_w4(qlin_gpu, d["w"])
    assert np.array_equal(wq.cpu().numpy(), oracle.pack_u4(codes))
    assert np.array_equal(sc.cpu().numpy().view(np.uint16), s16.view(np.uint16))
    assert np.array_equal(zp.cpu().numpy(), oracle.pack_u4(z))
    for T in (1, 4, 16):
        x = d["x"][:T]
        ref = oracle.w4a16_reference(x, codes, s16, z)
        y = _gemm(qlin_gpu, _dev(x), wq, sc, zp)
        assert_within_tolerance(y, ref, "W4A16 N=%d K=%d T=%d" % (N, K, T))


@pytest.mark.parametrize("scale", [1e3, 3e4])
def test_decode_activation_outliers(qlin_gpu, scale):
    """Large activation outliers next to ordinary ones in the same 32-element
    chunk; in half of the rows the outlier channels carry code = zero-point,
    so those outputs come from the ordinary activations alone."""
    d = inputs.w4a16_decode(seed=23, T=1, N=512, K=4096)
    x = d["x"].astype(np.float32)
    idx = np.random.default_rng(5).choice(4096, 16, replace=False)
    x[0, idx] *= scale
    x = np.clip(x, -60000.0, 60000.0).astype(np.float16)
    codes, s16, z = oracle.quant_w4_g128(d["w"])
    codes[:256, idx] = z[:256, idx // 128]
    ref = oracle.w4a16_reference(x, codes, s16, z)
    y = _gemm(qlin_gpu, _dev(x), _dev(oracle.pack_u4(codes)), _dev(s16), _dev(oracle.pack_u4(z)))
    assert_within_tolerance(y, ref, "W4A16 outliers x%g" % scale)


def _plane_bound(x, codes, s16, z):
    """Per-output error bound of the T = 1 GEMV's fixed-point activations.
    Each 32-element chunk c is represented as x_fix . sx_c with
    sx_c = max|x_c| / (127 . 2^15) and |x_fix - x / sx_c| <= 0.75 (the
    rounded quotient), so every element is off by at most 0.75 . sx_c.  The
    dot product of those errors with |s (q - z)|, plus the final fp16
    rounding (2^-11 relative) and slack for the fp32 combination of the
    plane sums, bounds |y - y_exact|."""
    xf = x.astype(np.float64).reshape(-1)
    k = xf.size
    amax = np.abs(xf.reshape(k // 32, 32)).max(axis=1)
    e = np.repeat(0.75 * amax / (127.0 * 2 ** 15), 32)
    n = codes.shape[0]
    w = np.abs((codes.reshape(n, k // 128, 128).astype(np.float64) - z[:, :, None]) * s16.astype(np.float64)[:, :, None])
    w = w.reshape(n, k)
    ref = oracle.w4a16_reference(x, codes, s16, z)[0]
    return w @ e + 2.0 ** -11 * np.abs(ref) + 1e-6 * (w @ np.abs(xf)), ref


@pytest.mark.parametrize("ratio", [16.0, 64.0, 1024.0])
def test_decode_fixed_point_activations(qlin_gpu, ratio):
    """The T = 1 GEMV rounds each 32-element chunk of x to fixed point on its
    largest |x|.  Here every chunk has one element `ratio` times the mean |x|
    of the other 31 (random signs), outputs are large (|ref| >> 1, so the
    relative part of the tolerance is what bites), and in half of the rows
    the large element's code equals the zero-point, so those outputs come
    from the small elements alone, where the fixed point is coarsest
    relative to the value.  Every output must lie within the error bound of
    the representation (_plane_bound) and within the parity tolerance."""
    rng = np.random.default_rng(71)
    n, k = 512, 4096
    small = rng.uniform(8.0, 24.0, size=(k // 32, 31)) * rng.choice([-1.0, 1.0], size=(k // 32, 31))
    big = np.minimum(ratio * np.abs(small).mean(axis=1), 60000.0)
    chunks = np.concatenate([big[:, None] * rng.choice([-1.0, 1.0], size=(k // 32, 1)), small], axis=1)
    perm = rng.permuted(np.tile(np.arange(32), (k // 32, 1)), axis=1)
    chunks = np.take_along_axis(chunks, perm, axis=1)
    x = chunks.reshape(1, k).astype(np.float16)
    xf = x.astype(np.float64).reshape(k // 32, 32)
    d = inputs.w4a16_decode(seed=72, T=1, N=n, K=k)
    # weights scaled so that the outputs are large but stay within fp16
    codes, s16, z = oracle.quant_w4_g128(d["w"] * (50.0 if ratio <= 64 else 3.0))
    big_cols = np.argmax(np.abs(xf), axis=1) + 32 * np.arange(k // 32)
    codes[: n // 2, big_cols] = z[: n // 2, big_cols // 128]
    bound, ref = _plane_bound(x, codes, s16, z)
    assert np.abs(ref).max() < 60000.0
    assert np.median(np.abs(ref)) > 100.0
    y = _gemm(qlin_gpu, _dev(x), _dev(oracle.pack_u4(codes)), _dev(s16), _dev(oracle.pack_u4(z)))[0].astype(np.float64)
    err = np.abs(y - ref)
    worst = int(np.argmax(err - bound))
    assert (err <= bound).all(), "row %d: err %g > bound %g (ref %g)" % (worst, err[worst], bound[worst], ref[worst])
    assert_within_tolerance(y[None, :], ref[None, :], "W4A16 T=1 fixed point, ratio %g" % ratio)


def test_decode_band_split_shapes(qlin_gpu):
    """Row counts that split unevenly over the CTAs and K with a partial last
    warp of 32-code chunks (K = 1408: 44 chunks)."""
    for (n, k) in ((763, 4096), (1000, 1408), (1, 128), (3, 384)):
        d = inputs.w4a16_decode(seed=29, T=1, N=n, K=k)
        codes, s16, z = oracle.quant_w4_g128(d["w"])
        ref = oracle.w4a16_reference(d["x"], codes, s16, z)
        y = _gemm(qlin_gpu, _dev(d["x"]), _dev(oracle.pack_u4(codes)), _dev(s16), _dev(oracle.pack_u4(z)))
        assert_within_tolerance(y, ref, "W4A16 N=%d K=%d" % (n, k))


def test_gemv_alternating_launch_shapes_in_use(qlin_gpu):
    """The T = 1 GEMV places each layer's CTAs one per SM beside the previous
    layer's by alternating two launch shapes, which are derived from the
    device's limits and the kernel's register count; when they cannot be met
    every launch silently keeps the plain shape (same results, a slower
    stack).  Pin that the two shapes are in use here, so that a change of
    the kernel's registers that breaks the plan fails this test."""
    alternating, registers = qlin_gpu.qlin_w4a16_gemv_launch_info()
    assert 0 < registers <= 72, "GEMV kernel uses %d registers per thread" % registers
    assert alternating == 1, "the GEMV's alternating launch shapes are not in use (%d registers)" % registers


@pytest.mark.parametrize("T", [1, 4])
def test_decode_chain_ping_pong(qlin_gpu, T):
    """Six layers launched back to back on one stream, each reading the
    previous layer's output from a ping-pong buffer pair (the kernels overlap
    through programmatic dependent launch); the oracle runs the same chain,
    rounding each layer's output to fp16 as the kernels do."""
    n = 2048
    layers = []
    for i in range(6):
        d = inputs.w4a16_decode(seed=40 + i, T=T, N=n, K=n)
        codes, s16, z = oracle.quant_w4_g128(d["w"])  # gain about 1 per layer: magnitudes stay O(1)
        layers.append((codes, s16, z))
    x0 = inputs.w4a16_decode(seed=39, T=T, N=n, K=n)["x"]
    bufs = [_dev(x0), torch.empty((T, n), dtype=torch.float16, device="cuda")]
    dev_w = [(_dev(oracle.pack_u4(c)), _dev(s), _dev(oracle.pack_u4(z))) for (c, s, z) in layers]
    for i, (wq, sc, zp) in enumerate(dev_w):
        qlin_gpu.qlin_w4a16_gemm(bufs[i % 2], wq, sc, zp, bufs[(i + 1) % 2])
    torch.cuda.synchronize()
    assert qlin_gpu.qlin_get_device_error() == 0
    y = bufs[len(dev_w) % 2].cpu().numpy()
    ref = x0
    for (c, s, z) in layers:
        ref = oracle.w4a16_reference(ref, c, s, z).astype(np.float16)
    assert_within_tolerance(y, ref.astype(np.float64), "W4A16 chain T=%d" % T)


def _quantized(seed, n, k):
    d = inputs.w4a16_decode(seed=seed, T=1, N=n, K=k)
    codes, s16, z = oracle.quant_w4_g128(d["w"])
    return codes, s16, z


@pytest.mark.parametrize("T,shapes", [(1, ((4096, 4096), (1024, 4096), (1024, 4096))),
                                      (1, ((763, 1408), (8, 1408), (5, 1408), (1000, 1408))),
                                      (1, ((0, 512), (300, 512), (1, 512))),
                                      (4, ((256, 1024), (100, 1024)))])
def test_grouped_equals_separate(qlin_gpu, T, shapes):
    """One grouped call over matrices of different heights (a GQA-like q/k/v
    set, ragged heights whose boundaries fall inside a shared-memory stage,
    an empty matrix) gives every output bit for bit equal to a separate
    qlin_w4a16_gemm call, and within tolerance of the oracle; one matrix is
    symmetric (no zero-points)."""
    k = shapes[0][1]
    x = inputs.w4a16_decode(seed=60, T=T, N=8, K=k)["x"]
    xt = _dev(x)
    mats = [_quantized(61 + i, n, k) for i, (n, _) in enumerate(shapes)]
    wqs = [_dev(oracle.pack_u4(c)) for (c, _, _) in mats]
    scs = [_dev(s) for (_, s, _) in mats]
    zps = [_dev(oracle.pack_u4(z)) for (_, _, z) in mats]
    zps[-1] = None
    ys = [torch.empty((T, n), dtype=torch.float16, device="cuda") for (n, _) in shapes]
    qlin_gpu.qlin_w4a16_gemm_grouped(xt, wqs, scs, zps, ys)
    torch.cuda.synchronize()
    assert qlin_gpu.qlin_get_device_error() == 0
    for i, (n, _) in enumerate(shapes):
        if n == 0:
            continue
        sep = torch.empty((T, n), dtype=torch.float16, device="cuda")
        qlin_gpu.qlin_w4a16_gemm(xt, wqs[i], scs[i], zps[i], sep)
        torch.cuda.synchronize()
        assert torch.equal(ys[i], sep), "matrix %d" % i
        codes, s16, z = mats[i]
        if zps[i] is None:
            z = np.full_like(z, 8)
        ref = oracle.w4a16_reference(x, codes, s16, z)
        assert_within_tolerance(ys[i].cpu().numpy(), ref, "grouped matrix %d (N=%d)" % (i, n))


def test_grouped_decoder_block_chain(qlin_gpu):
    """Two decoder blocks at decode (T = 1) with the block's dependency
    structure: q, k, v in one grouped call on h; o on v; gate and up in one
    grouped call on o's output; down on up; the next block starts from down's
    output.  The kernels overlap through programmatic dependent launch; the
    oracle runs the same chain, rounding every output to fp16."""
    hid, inter = 1024, 2816
    blocks = []
    seed = 80
    for _ in range(2):
        blk = {}
        for name, (n, k) in (("q", (hid, hid)), ("k", (hid, hid)), ("v", (hid, hid)), ("o", (hid, hid)),
                             ("gate", (inter, hid)), ("up", (inter, hid)), ("down", (hid, inter))):
            blk[name] = _quantized(seed, n, k)
            seed += 1
        blocks.append(blk)
    x0 = inputs.w4a16_decode(seed=79, T=1, N=8, K=hid)["x"]
    dev = [{n: (_dev(oracle.pack_u4(c)), _dev(s), _dev(oracle.pack_u4(z))) for n, (c, s, z) in b.items()}
           for b in blocks]
    h = _dev(x0)
    out = {}
    for b in dev:
        out = {n: torch.empty((1, b[n][0].shape[0]), dtype=torch.float16, device="cuda") for n in b}
        qlin_gpu.qlin_w4a16_gemm_grouped(h, [b[n][0] for n in "qkv"], [b[n][1] for n in "qkv"],
                                         [b[n][2] for n in "qkv"], [out[n] for n in "qkv"])
        qlin_gpu.qlin_w4a16_gemm(out["v"], *b["o"], out["o"])
        qlin_gpu.qlin_w4a16_gemm_grouped(out["o"], [b[n][0] for n in ("gate", "up")], [b[n][1] for n in ("gate", "up")],
                                         [b[n][2] for n in ("gate", "up")], [out[n] for n in ("gate", "up")])
        qlin_gpu.qlin_w4a16_gemm(out["up"], *b["down"], out["down"])
        h = out["down"]
    torch.cuda.synchronize()
    assert qlin_gpu.qlin_get_device_error() == 0
    ref = x0
    refs = {}
    for blk in blocks:
        refs = {}
        for n in "qkv":
            refs[n] = oracle.w4a16_reference(ref, *blk[n]).astype(np.float16)
        refs["o"] = oracle.w4a16_reference(refs["v"], *blk["o"]).astype(np.float16)
        for n in ("gate", "up"):
            refs[n] = oracle.w4a16_reference(refs["o"], *blk[n]).astype(np.float16)
        refs["down"] = oracle.w4a16_reference(refs["up"], *blk["down"]).astype(np.float16)
        ref = refs["down"]
    for n in ("q", "k", "gate", "down"):
        assert_within_tolerance(out[n].cpu().numpy(), refs[n].astype(np.float64), "block chain %s" % n)


def _dev_mats(mats, symmetric_last=False):
    wqs = [_dev(oracle.pack_u4(c)) for (c, _, _) in mats]
    scs = [_dev(s) for (_, s, _) in mats]
    zps = [_dev(oracle.pack_u4(z)) for (_, _, z) in mats]
    if symmetric_last:
        zps[-1] = None
    return wqs, scs, zps


def _run_sequence(q, steps):
    ws = torch.zeros(q.qlin_w4a16_sequence_workspace_bytes(len(steps)), dtype=torch.uint8, device="cuda")
    q.qlin_w4a16_gemv_sequence(steps, ws)
    torch.cuda.synchronize()
    assert q.qlin_get_device_error() == 0


@pytest.mark.parametrize("hid,inter", [(1024, 2816), (4096, 11008)])
def test_sequence_decoder_blocks_equal_single_launches(qlin_gpu, hid, inter):
    """Two decoder blocks as one persistent sequence (q,k,v grouped on the
    block input; o on v; gate,up grouped on o; down on up; the second block
    on the first block's output): every output equals the per-launch path on
    the same inputs bit for bit, and the oracle within tolerance.  The first
    block's v projection is symmetric (no zero-points)."""
    seed = 100
    blocks = []
    for _ in range(2):
        blk = {}
        for name, (n, k) in (("q", (hid, hid)), ("k", (hid // 4, hid)), ("v", (hid // 4, hid)), ("o", (hid, hid // 4)),
                             ("gate", (inter, hid)), ("up", (inter, hid)), ("down", (hid, inter))):
            blk[name] = _quantized(seed, n, k)
            seed += 1
        blocks.append(blk)
    x0 = inputs.w4a16_decode(seed=99, T=1, N=8, K=hid)["x"]
    xt = _dev(x0)
    devs = []
    for bi, blk in enumerate(blocks):
        d = {}
        for name in blk:
            wq, sc, zp = _dev_mats([blk[name]], symmetric_last=(bi == 0 and name == "v"))
            d[name] = (wq[0], sc[0], zp[0])
        devs.append(d)

    def outputs():
        return [{n: torch.full((1, blocks[0][n][0].shape[0]), float("nan"), dtype=torch.float16, device="cuda")
                 for n in blocks[0]} for _ in blocks]

    seq_out, ref_out = outputs(), outputs()
    steps = []
    h = xt
    for d, o in zip(devs, seq_out):
        steps.append((h, [d[n][0] for n in "qkv"], [d[n][1] for n in "qkv"], [d[n][2] for n in "qkv"],
                      [o[n] for n in "qkv"]))
        steps.append((o["v"], [d["o"][0]], [d["o"][1]], [d["o"][2]], [o["o"]]))
        steps.append((o["o"], [d[n][0] for n in ("gate", "up")], [d[n][1] for n in ("gate", "up")],
                      [d[n][2] for n in ("gate", "up")], [o[n] for n in ("gate", "up")]))
        steps.append((o["up"], [d["down"][0]], [d["down"][1]], [d["down"][2]], [o["down"]]))
        h = o["down"]
    _run_sequence(qlin_gpu, steps)
    h = xt
    for d, o in zip(devs, ref_out):
        for n in "qkv":
            qlin_gpu.qlin_w4a16_gemm(h, *d[n], o[n])
        qlin_gpu.qlin_w4a16_gemm(o["v"], *d["o"], o["o"])
        for n in ("gate", "up"):
            qlin_gpu.qlin_w4a16_gemm(o["o"], *d[n], o[n])
        qlin_gpu.qlin_w4a16_gemm(o["up"], *d["down"], o["down"])
        h = o["down"]
    torch.cuda.synchronize()
    for bi in range(2):
        for n in blocks[0]:
            assert torch.equal(seq_out[bi][n], ref_out[bi][n]), "block %d %s" % (bi, n)
    # the oracle on the first block's q and down projections
    codes, s16, z = blocks[0]["q"]
    assert_within_tolerance(seq_out[0]["q"].cpu().numpy(), oracle.w4a16_reference(x0, codes, s16, z), "sequence q")
    codes, s16, z = blocks[0]["down"]
    up = seq_out[0]["up"].cpu().numpy()
    assert_within_tolerance(seq_out[0]["down"].cpu().numpy(), oracle.w4a16_reference(up, codes, s16, z),
                            "sequence down")


@pytest.mark.parametrize("T,hid,inter", [(1, 1024, 2816), (4, 1024, 2816), (16, 1024, 2816), (20, 512, 1408),
                                          (4, 4096, 11008)])
def test_chain_equals_grouped_calls(qlin_gpu, T, hid, inter):
    """qlin_w4a16_chain (one call, a launch per step) over two decoder blocks,
    and the same chain prepared once (qlin_w4a16_chain_prepare) and run
    twice, give every output of the same grouped calls made one by one, bit
    for bit, and the oracle within tolerance; T = 20 runs the prefill GEMM (a
    128-token tile, K shared by a CTA cluster) per step.  The first block's
    v projection is symmetric (no
    zero-points)."""
    seed = 700 + T
    blocks = []
    for _ in range(2):
        blk = {}
        for name, (n, k) in (("q", (hid, hid)), ("k", (hid // 4, hid)), ("v", (hid // 4, hid)), ("o", (hid, hid // 4)),
                             ("gate", (inter, hid)), ("up", (inter, hid)), ("down", (hid, inter))):
            blk[name] = _quantized(seed, n, k)
            seed += 1
        blocks.append(blk)
    x0 = inputs.w4a16_decode(seed=98, T=T, N=8, K=hid)["x"]
    xt = _dev(x0)
    devs = []
    for bi, blk in enumerate(blocks):
        d = {}
        for name in blk:
            wq, sc, zp = _dev_mats([blk[name]], symmetric_last=(bi == 0 and name == "v"))
            d[name] = (wq[0], sc[0], zp[0])
        devs.append(d)

    def run(mode):
        outs = [{n: torch.full((T, blocks[0][n][0].shape[0]), float("nan"), dtype=torch.float16, device="cuda")
                 for n in blocks[0]} for _ in blocks]
        steps = []
        h = xt
        for d, o in zip(devs, outs):
            steps.append((h, [d[n][0] for n in "qkv"], [d[n][1] for n in "qkv"], [d[n][2] for n in "qkv"],
                          [o[n] for n in "qkv"]))
            steps.append((o["v"], [d["o"][0]], [d["o"][1]], [d["o"][2]], [o["o"]]))
            steps.append((o["o"], [d[n][0] for n in ("gate", "up")], [d[n][1] for n in ("gate", "up")],
                          [d[n][2] for n in ("gate", "up")], [o[n] for n in ("gate", "up")]))
            steps.append((o["up"], [d["down"][0]], [d["down"][1]], [d["down"][2]], [o["down"]]))
            h = o["down"]
        if mode == "chain":
            qlin_gpu.qlin_w4a16_chain(steps)
        elif mode == "prepared":
            prepared = qlin_gpu.qlin_w4a16_chain_prepare(steps)
            prepared.run()
            prepared.run()  # a second run over the same buffers gives the same outputs
        else:
            for (x, wqs, scs, zps, ys) in steps:
                qlin_gpu.qlin_w4a16_gemm_grouped(x, wqs, scs, zps, ys)
        torch.cuda.synchronize()
        assert qlin_gpu.qlin_get_device_error() == 0
        return outs

    got, ref, prep = run("chain"), run("grouped"), run("prepared")
    for bi in range(2):
        for n in blocks[0]:
            assert torch.equal(got[bi][n], ref[bi][n]), "block %d %s" % (bi, n)
            assert torch.equal(prep[bi][n], ref[bi][n]), "prepared chain, block %d %s" % (bi, n)
    codes, s16, z = blocks[0]["q"]
    assert_within_tolerance(got[0]["q"].cpu().numpy(), oracle.w4a16_reference(x0, codes, s16, z), "chain q")
    codes, s16, z = blocks[1]["down"]
    up = got[1]["up"].cpu().numpy()
    assert_within_tolerance(got[1]["down"].cpu().numpy(), oracle.w4a16_reference(up, codes, s16, z), "chain down")


def test_sequence_many_small_steps(qlin_gpu):
    """130 chained steps (more than one launch holds) on two ping-pong buffers,
    with ragged heights and K values whose scale rows are not 16-byte aligned
    (K = 1408: 11 groups); equal to per-launch results bit for bit."""
    rng = np.random.default_rng(7)
    n_steps = 130
    width = 1408
    mats = []
    for i in range(n_steps):
        mats.append(_quantized(200 + i, width, width))
    dev = [_dev_mats([m]) for m in mats]
    x0 = inputs.w4a16_decode(seed=198, T=1, N=8, K=width)["x"]
    bufs = [_dev(x0), torch.empty((1, width), dtype=torch.float16, device="cuda")]
    ref_bufs = [_dev(x0), torch.empty((1, width), dtype=torch.float16, device="cuda")]
    steps = []
    for i, (wq, sc, zp) in enumerate(dev):
        steps.append((bufs[i % 2], wq, sc, zp, [bufs[(i + 1) % 2]]))
    _run_sequence(qlin_gpu, steps)
    for i, (wq, sc, zp) in enumerate(dev):
        qlin_gpu.qlin_w4a16_gemm(ref_bufs[i % 2], wq[0], sc[0], zp[0], ref_bufs[(i + 1) % 2])
    torch.cuda.synchronize()
    assert torch.equal(bufs[n_steps % 2], ref_bufs[n_steps % 2])
    assert torch.isfinite(bufs[n_steps % 2].float()).all()


def test_sequence_ragged_groups_and_outliers(qlin_gpu):
    """Grouped steps with ragged and tiny heights (763, 5, 1000 rows; an empty
    matrix) and activation outliers (the three-plane path) in the input."""
    k = 4096
    mats = [_quantized(300 + i, n, k) for i, n in enumerate((763, 5, 0, 1000))]
    wqs, scs, zps = _dev_mats([m for m in mats])
    x = inputs.w4a16_decode(seed=301, T=1, N=8, K=k)["x"].astype(np.float32)
    x[0, 17] *= 3e3
    x[0, 2049] *= -1e3
    x = x.astype(np.float16)
    xt = _dev(x)
    ys = [torch.empty((1, max(n, 1) if n else 0), dtype=torch.float16, device="cuda") for n in (763, 5, 0, 1000)]
    _run_sequence(qlin_gpu, [(xt, wqs, scs, zps, ys)])
    for i, n in enumerate((763, 5, 0, 1000)):
        if n == 0:
            continue
        ref = torch.empty((1, n), dtype=torch.float16, device="cuda")
        qlin_gpu.qlin_w4a16_gemm(xt, wqs[i], scs[i], zps[i], ref)
        torch.cuda.synchronize()
        assert torch.equal(ys[i], ref), i
        codes, s16, z = mats[i]
        assert_within_tolerance(ys[i].cpu().numpy(), oracle.w4a16_reference(x, codes, s16, z), "ragged %d" % n)


# ---- the streamed tensor-core path for a few tokens (T <= 16 per launch) ----

@pytest.mark.parametrize("T,N,K", [
    (7, 5000, 128),      # one group per row: every CTA owns full rows
    (3, 77, 1152),       # bands shorter than a stage, odd group count
    (9, 1000, 3584),     # two token tiles (one padded token), 14 warps of two groups
    (6, 1500, 4480),     # K split over two CTAs, ragged group count (35)
    (2, 2000, 8192),     # two CTAs, 16 warps of two groups
    (16, 300, 4096),     # two CTAs, two token tiles, bands of one stage
    (4, 300, 8448),      # K split over four CTAs (66 groups)
    (12, 640, 7296),     # four CTAs, two token tiles with padded tokens
    (16, 600, 11008),    # four CTAs on the down-projection K
])
def test_skinny_splits_against_oracle(qlin_gpu, T, N, K):
    d = inputs.w4a16_decode(seed=500 + T, T=T, N=N, K=K)
    codes, s16, z = oracle.quant_w4_g128(d["w"])
    ref = oracle.w4a16_reference(d["x"], codes, s16, z)
    y = _gemm(qlin_gpu, _dev(d["x"]), _dev(oracle.pack_u4(codes)), _dev(s16), _dev(oracle.pack_u4(z)))
    assert_within_tolerance(y, ref, "W4A16 skinny T=%d N=%d K=%d" % (T, N, K))


@pytest.mark.parametrize("T,N,K", [(16, 65536, 4096), (4, 90000, 4096)])
def test_skinny_several_bands_sampled_rows(qlin_gpu, T, N, K):
    """Large N: each cluster processes several bands of rows in turn (the
    receive buffers alternate between bands), or one CTA owns a band of
    hundreds of rows.  The oracle checks a sample of rows that covers both
    ends; a second run must give the same bits."""
    d = inputs.w4a16_packed_random(seed=700 + T, T=T, N=N, K=K)
    xt, wq, sc, zp = _dev(d["x"]), _dev(d["wq"]), _dev(d["scales"]), _dev(d["zeros"])
    y = _gemm(qlin_gpu, xt, wq, sc, zp)
    y2 = _gemm(qlin_gpu, xt, wq, sc, zp)
    assert np.array_equal(y.view(np.uint16), y2.view(np.uint16))
    rng = np.random.default_rng(7)
    rows = np.unique(np.concatenate([np.arange(0, 40), np.arange(N - 40, N),
                                     rng.choice(N, size=600, replace=False)]))
    ref = oracle.w4a16_reference_packed(d["x"], d["wq"][rows], d["scales"][rows], d["zeros"][rows])
    assert_within_tolerance(y[:, rows], ref, "W4A16 T=%d N=%d sampled rows" % (T, N))


@pytest.mark.parametrize("T", [2, 9, 16, 33])
def test_skinny_grouped_equals_separate(qlin_gpu, T):
    """Grouped calls over matrices whose boundaries fall inside a 16-row
    stage give the same bits as one call per matrix (the K split depends
    only on T and K), and match the oracle."""
    shapes = ((763, 1408), (8, 1408), (5, 1408), (1000, 1408))
    k = shapes[0][1]
    x = inputs.w4a16_decode(seed=800 + T, T=T, N=8, K=k)["x"]
    xt = _dev(x)
    mats = [_quantized(801 + i, n, k) for i, (n, _) in enumerate(shapes)]
    wqs = [_dev(oracle.pack_u4(c)) for (c, _, _) in mats]
    scs = [_dev(s) for (_, s, _) in mats]
    zps = [_dev(oracle.pack_u4(z)) for (_, _, z) in mats]
    ys = [torch.empty((T, n), dtype=torch.float16, device="cuda") for (n, _) in shapes]
    qlin_gpu.qlin_w4a16_gemm_grouped(xt, wqs, scs, zps, ys)
    torch.cuda.synchronize()
    assert qlin_gpu.qlin_get_device_error() == 0
    for i, (n, _) in enumerate(shapes):
        sep = torch.empty((T, n), dtype=torch.float16, device="cuda")
        qlin_gpu.qlin_w4a16_gemm(xt, wqs[i], scs[i], zps[i], sep)
        torch.cuda.synchronize()
        assert torch.equal(ys[i], sep), "matrix %d" % i
        ref = oracle.w4a16_reference(x, *mats[i])
        assert_within_tolerance(ys[i].cpu().numpy(), ref, "grouped T=%d matrix %d" % (T, i))
