"""NVFP4 quantization with ARCQuant residual channels, and its set-up helpers
(per-tensor scale, channel order), on the GPU against the CPU oracle, bit for
bit (codes, E4M3 scales, permutation, per-tensor scale)."""

import numpy as np
import pytest
import torch

import oracle
import quantized_linear_layer_gb300 as qmod
from quantized_linear_layer_gb300 import inputs
from conftest import sf_rows_to_mma

pytestmark = pytest.mark.gpu


def _global_scale(q, xt):
    g = torch.empty(1, dtype=torch.float32, device="cuda")
    q.qlin_nvfp4_global_scale(xt, g)
    return g


def _perm(q, xt):
    p = torch.empty(xt.shape[1], dtype=torch.int32, device="cuda")
    q.qlin_arc_perm(xt, p)
    return p


def _quant(q, xt, g, perm, S, mode):
    rows, k = xt.shape
    qo = torch.empty((rows, (k + S) // 2), dtype=torch.uint8, device="cuda")
    sf = torch.empty((rows, (k + S) // 16), dtype=torch.uint8, device="cuda")
    q.qlin_quant_nvfp4(xt, g, qo, sf, perm=perm, S=S, mode=mode)
    torch.cuda.synchronize()
    assert q.qlin_get_device_error() == 0
    return qo.cpu().numpy(), sf.cpu().numpy()


def test_global_scale_and_perm_bit_exact(qlin_gpu):
    d = inputs.nvfp4_arc(seed=4, T=300, K=1024)
    xt = torch.from_numpy(d["x"]).cuda()
    x32 = d["x"].astype(np.float32)
    g = _global_scale(qlin_gpu, xt).cpu().numpy()
    assert g.view(np.uint32)[0] == np.float32(oracle.nvfp4_global_scale(x32)).view(np.uint32)
    p = _perm(qlin_gpu, xt).cpu().numpy()
    assert np.array_equal(p, oracle.arc_perm(x32))


def test_perm_ties(qlin_gpu):
    x = np.zeros((4, 64), dtype=np.float16)
    x[0, ::3] = 2.0
    x[1, 5] = -2.0
    x[2, 40] = 7.0
    p = _perm(qlin_gpu, torch.from_numpy(x).cuda()).cpu().numpy()
    assert np.array_equal(p, oracle.arc_perm(x.astype(np.float32)))


@pytest.mark.parametrize("S,mode", [(0, 0), (128, 0), (128, 1), (32, 0), (1024, 0)])
def test_quant_nvfp4_modes(qlin_gpu, S, mode):
    d = inputs.nvfp4_arc(seed=4, T=130, K=1024)
    xt = torch.from_numpy(d["x"]).cuda()
    x32 = d["x"].astype(np.float32)
    g = np.float32(oracle.nvfp4_global_scale(x32))
    perm = oracle.arc_perm(x32)
    gq, gsf = _quant(qlin_gpu, xt, torch.tensor([g]).cuda(), torch.from_numpy(perm).cuda(), S, mode)
    if mode == 0:
        rq, rsf = oracle.arc_quantize_activation(x32, perm, S, g)
    else:
        rq, rsf = oracle.arc_quantize_weight(x32, perm, S, g)
    assert np.array_equal(gsf, rsf)
    assert np.array_equal(gq, oracle.pack_u4(rq))


@pytest.mark.parametrize("dtype", ["f16", "bf16", "f32"])
def test_quant_nvfp4_no_perm_dtypes(qlin_gpu, dtype):
    rng = np.random.default_rng(8)
    x = rng.standard_normal((50, 512)).astype(np.float32)
    if dtype == "f16":
        xt = torch.from_numpy(x.astype(np.float16)).cuda()
    elif dtype == "bf16":
        xt = torch.from_numpy(x).to(torch.bfloat16).cuda()
    else:
        xt = torch.from_numpy(x).cuda()
    x32 = xt.float().cpu().numpy()
    g = np.float32(oracle.nvfp4_global_scale(x32))
    gq, gsf = _quant(qlin_gpu, xt, torch.tensor([g]).cuda(), None, 0, 0)
    rq, rsf = oracle.nvfp4_quantize(x32, g)
    assert np.array_equal(gsf, rsf)
    assert np.array_equal(gq, oracle.pack_u4(rq))


def test_quant_nvfp4_edge_values(qlin_gpu):
    """E2M1 ties, negative values that round to zero, blocks of zeros, and
    tiny blocks whose E4M3 scale is subnormal or zero."""
    k = 256
    rows = []
    mids = [0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0]
    base = np.zeros(16, dtype=np.float32)
    base[0] = 6.0                                     # block scale 1 with g = 1
    for m in mids:
        b = base.copy()
        b[1:8] = [m, -m, m * 1.0000001, -0.1, 0.1, -0.0, 0.0]
        rows.append(np.tile(b, k // 16))
    rows.append(np.zeros(k, dtype=np.float32))
    tiny = np.tile(np.linspace(-1, 1, 16, dtype=np.float32), k // 16)
    for e in (-8, -10, -12, -14, -16, -20):
        rows.append(tiny * np.float32(2.0 ** e))
    x = np.stack(rows).astype(np.float32)
    xt = torch.from_numpy(x).cuda()
    for g in (np.float32(1.0), np.float32(oracle.nvfp4_global_scale(x))):
        gq, gsf = _quant(qlin_gpu, xt, torch.tensor([g]).cuda(), None, 0, 0)
        rq, rsf = oracle.nvfp4_quantize(x, g)
        assert np.array_equal(gsf, rsf), g
        assert np.array_equal(gq, oracle.pack_u4(rq)), g


@pytest.mark.parametrize("g", [1e-12, 1e-40, 5e-39, 1e20, 3e38])
@pytest.mark.parametrize("mode", [0, 1])
def test_quant_nvfp4_extreme_global_scale(qlin_gpu, g, mode):
    """Per-tensor scales far from the tensor's own: block scales saturating at
    448 with element quotients that overflow float32 (g = 1e-12 against
    values near 1e30), subnormal g and subnormal block divisors, and huge g
    that sends block scales to zero or to the subnormal E4M3 range.  Every
    code must still equal the one true float32 division gives."""
    rng = np.random.default_rng(11)
    x = rng.standard_normal((9, 512)).astype(np.float32)
    x[0] *= np.float32(1e30)
    x[1] *= np.float32(1e-30)
    x[2] *= np.float32(3e37)
    x[3, :16] = 0.0
    x[3, 16] = -0.0
    x[4] *= np.float32(1e-39)
    xt = torch.from_numpy(x).cuda()
    g32 = np.float32(g)
    perm = oracle.arc_perm(x)
    gq, gsf = _quant(qlin_gpu, xt, torch.tensor([g32]).cuda(), torch.from_numpy(perm).cuda(), 64, mode)
    with np.errstate(over="ignore", divide="ignore", invalid="ignore", under="ignore"):
        if mode == 0:
            rq, rsf = oracle.arc_quantize_activation(x, perm, 64, g32)
        else:
            rq, rsf = oracle.arc_quantize_weight(x, perm, 64, g32)
    assert np.array_equal(gsf, rsf)
    assert np.array_equal(gq, oracle.pack_u4(rq))


def test_config5_activation_and_weight(qlin_gpu):
    d = inputs.nvfp4_arc(seed=4)
    S = d["S"]
    xt = torch.from_numpy(d["x"]).cuda()
    x32 = d["x"].astype(np.float32)
    g = _global_scale(qlin_gpu, xt)
    perm = _perm(qlin_gpu, xt)
    gx = np.float32(oracle.nvfp4_global_scale(x32))
    rperm = oracle.arc_perm(x32)
    assert g.cpu().numpy().view(np.uint32)[0] == gx.view(np.uint32)
    assert np.array_equal(perm.cpu().numpy(), rperm)
    gq, gsf = _quant(qlin_gpu, xt, g, perm, S, qmod.QLIN_NVFP4_RESIDUAL)
    rq, rsf = oracle.arc_quantize_activation(x32, rperm, S, gx)
    assert np.array_equal(gsf, rsf) and np.array_equal(gq, oracle.pack_u4(rq))
    wt = torch.from_numpy(d["w"]).cuda()
    gw_t = _global_scale(qlin_gpu, wt)
    gw = np.float32(oracle.nvfp4_global_scale(d["w"]))
    assert gw_t.cpu().numpy().view(np.uint32)[0] == gw.view(np.uint32)
    wq, wsf = _quant(qlin_gpu, wt, gw_t, perm, S, qmod.QLIN_NVFP4_DUPLICATE)
    rwq, rwsf = oracle.arc_quantize_weight(d["w"], rperm, S, gw)
    assert np.array_equal(wsf, rwsf) and np.array_equal(wq, oracle.pack_u4(rwq))


@pytest.mark.parametrize("rows,S,mode", [(130, 128, 0), (128, 64, 1), (7, 0, 0)])
def test_quant_nvfp4_mma_scale_layout(qlin_gpu, rows, S, mode):
    d = inputs.nvfp4_arc(seed=6, T=rows, K=1024)
    xt = torch.from_numpy(d["x"]).cuda()
    x32 = d["x"].astype(np.float32)
    g = np.float32(oracle.nvfp4_global_scale(x32))
    perm = oracle.arc_perm(x32)
    k_aug = 1024 + S
    q1 = torch.empty((rows, k_aug // 2), dtype=torch.uint8, device="cuda")
    sf_m = torch.full((qlin_gpu.qlin_nvfp4_sf_bytes(rows, k_aug, qmod.QLIN_SF_MMA),), 0, dtype=torch.uint8,
                      device="cuda")
    qlin_gpu.qlin_quant_nvfp4(xt, torch.tensor([g]).cuda(), q1, sf_m, perm=torch.from_numpy(perm).cuda(), S=S, mode=mode,
                              sf_layout=qmod.QLIN_SF_MMA)
    torch.cuda.synchronize()
    if mode == 0:
        rq, rsf = oracle.arc_quantize_activation(x32, perm, S, g)
    else:
        rq, rsf = oracle.arc_quantize_weight(x32, perm, S, g)
    assert np.array_equal(q1.cpu().numpy(), oracle.pack_u4(rq))
    assert np.array_equal(sf_m.cpu().numpy(), sf_rows_to_mma(rsf))


@pytest.mark.parametrize("rows,K,dtype,S,with_perm", [(5, 40960, "f32", 0, False), (7, 16384, "f16", 128, True),
                                                     (601, 1024, "bf16", 64, True)])
def test_quant_nvfp4_row_staging(qlin_gpu, rows, K, dtype, S, with_perm):
    """One staged row per CTA (160 KB fp32 rows), two per CTA (32 KB fp16 rows),
    and 601 rows of two per CTA (an odd last CTA)."""
    rng = np.random.default_rng(rows + K)
    x = rng.standard_normal((rows, K)).astype(np.float32)
    if dtype == "f16":
        xt = torch.from_numpy(x.astype(np.float16)).cuda()
    elif dtype == "bf16":
        xt = torch.from_numpy(x).to(torch.bfloat16).cuda()
    else:
        xt = torch.from_numpy(x).cuda()
    x32 = xt.float().cpu().numpy()
    g = np.float32(oracle.nvfp4_global_scale(x32))
    perm = oracle.arc_perm(x32) if with_perm else None
    gq, gsf = _quant(qlin_gpu, xt, torch.tensor([g]).cuda(),
                     None if perm is None else torch.from_numpy(perm).cuda(), S, 0)
    if perm is None:
        rq, rsf = oracle.nvfp4_quantize(x32, g)
    else:
        rq, rsf = oracle.arc_quantize_activation(x32, perm, S, g)
    assert np.array_equal(gsf, rsf)
    assert np.array_equal(gq, oracle.pack_u4(rq))
