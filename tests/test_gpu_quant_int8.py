"""Per-token int8 activation quantization and the W8A8 weight-side helpers on
the GPU against the CPU oracle, bit for bit (codes, scales, zero-points)."""

import numpy as np
import pytest
import torch

import oracle
from quantized_linear_layer_gb300 import inputs

pytestmark = pytest.mark.gpu

TORCH_DT = {np.float16: torch.float16, np.float32: torch.float32}


def _run(q, x_t, asym):
    t, k = x_t.shape
    qo = torch.empty((t, k), dtype=torch.int8, device="cuda")
    s = torch.empty(t, dtype=torch.float32, device="cuda")
    z = torch.empty(t, dtype=torch.int32, device="cuda") if asym else None
    q.qlin_quant_act_int8(x_t, qo, s, z)
    torch.cuda.synchronize()
    return qo.cpu().numpy(), s.cpu().numpy(), (z.cpu().numpy() if asym else None)


def _check(q, x_t, x32, asym):
    qo, s, z = _run(q, x_t, asym)
    if asym:
        rq, rs, rz = oracle.quant_int8_asym(x32)
        assert np.array_equal(z, rz)
    else:
        rq, rs = oracle.quant_int8_sym(x32)
    assert np.array_equal(s.view(np.uint32), rs.view(np.uint32))
    assert np.array_equal(qo, rq)


@pytest.mark.parametrize("asym", [False, True])
@pytest.mark.parametrize("dtype", ["f16", "bf16", "f32"])
@pytest.mark.parametrize("K", [16, 272, 4096, 12288])
def test_quant_int8_dtypes_and_widths(qlin_gpu, asym, dtype, K):
    rng = np.random.default_rng(K)
    x = (rng.standard_normal((37, K)) * 3).astype(np.float32)
    x[1] = 0.0                                    # all-zero row
    x[2] = np.abs(x[2]) + 0.5                     # row above 0
    x[3] = -np.abs(x[3]) - 0.5                    # row below 0
    if dtype == "f16":
        xt = torch.from_numpy(x.astype(np.float16)).cuda()
    elif dtype == "bf16":
        xt = torch.from_numpy(x).to(torch.bfloat16).cuda()
    else:
        xt = torch.from_numpy(x).cuda()
    x32 = xt.float().cpu().numpy()
    _check(qlin_gpu, xt, x32, asym)


@pytest.mark.parametrize("asym", [False, True])
def test_quant_int8_rounding_ties(qlin_gpu, asym):
    """Rows built so that many quotients x / s are exact .5 ties."""
    k = 256
    x = np.zeros((8, k), dtype=np.float32)
    for r in range(8):
        x[r] = (np.arange(k) - 128 + 0.5) * (r + 1) / 8.0
        x[r, 0] = -127.0 * (r + 1) / 8.0           # absmax pins s = (r+1)/8 for the symmetric case
    xt = torch.from_numpy(x.astype(np.float16)).cuda()
    _check(qlin_gpu, xt, xt.float().cpu().numpy(), asym)


def test_config3_activations_symmetric(qlin_gpu):
    d = inputs.w8a8_sym_bias(seed=2)
    xt = torch.from_numpy(d["x"]).cuda()
    _check(qlin_gpu, xt, d["x"].astype(np.float32), asym=False)


def test_config4_activations_asymmetric(qlin_gpu):
    d = inputs.w8a8_azp_token(seed=3, N=16)
    xt = torch.from_numpy(d["x"]).cuda()
    _check(qlin_gpu, xt, d["x"].astype(np.float32), asym=True)


def test_weight_per_channel_and_row_sum(qlin_gpu):
    d = inputs.w8a8_sym_bias(seed=2, T=16, N=1000, K=4096)
    wt = torch.from_numpy(d["w"]).cuda()
    qo, s, _ = _run(qlin_gpu, wt, asym=False)
    rq, rs = oracle.quant_int8_sym(d["w"])
    assert np.array_equal(qo, rq) and np.array_equal(s.view(np.uint32), rs.view(np.uint32))
    adj = torch.empty(1000, dtype=torch.int32, device="cuda")
    qlin_gpu.qlin_int8_row_sum(torch.from_numpy(rq).cuda(), adj)
    assert np.array_equal(adj.cpu().numpy(), oracle.azp_adj_from_weight(rq))
    # extreme codes: all -128 / all 127 rows
    ext = np.zeros((4, 4096), dtype=np.int8)
    ext[0] = -128
    ext[1] = 127
    ext[2, ::2] = -128
    adj = torch.empty(4, dtype=torch.int32, device="cuda")
    qlin_gpu.qlin_int8_row_sum(torch.from_numpy(ext).cuda(), adj)
    assert np.array_equal(adj.cpu().numpy(), oracle.azp_adj_from_weight(ext))
