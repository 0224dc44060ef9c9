"""Online Hadamard rotation on the GPU against the CPU oracle's float64
definition, every n-group of a row times H_n / sqrt(n) and then the column
signs: the Sylvester transform (groups of 2 .. 8192, warp-level and through
shared memory) and the regular Hadamard of order 4^k, fp16 / bf16 / fp32
rows, in place and out of place.  Outputs are compared within the fp
tolerance (max |err| <= 1e-2 (1 + |ref|), relative Frobenius <= 2e-3)
against the exact rotation of the same input values."""

import numpy as np
import pytest
import torch

import oracle
from conftest import assert_within_tolerance

pytestmark = pytest.mark.gpu


def _rows(seed, rows, k):
    rng = np.random.default_rng(seed)
    x = (rng.standard_normal((rows, k)) * np.exp(rng.uniform(-3, 3, size=(rows, 1)))).astype(np.float32)
    if rows > 1:
        x[1] = 0.0
    if rows > 2:
        x[2, ::7] *= 100.0       # outlier channels, the case the rotation is for
    if rows > 3:
        x[3] = 2.5               # a constant row (a row outlier)
    return x


def _signs(seed, k):
    return np.where(np.random.default_rng(seed).random(k) < 0.5, -1, 1).astype(np.int8)


def _code(q, kind):
    return q.QLIN_HADAMARD_SYLVESTER if kind == "sylvester" else q.QLIN_HADAMARD_REGULAR


CASES = [("sylvester", 2, 64), ("sylvester", 8, 1024), ("sylvester", 64, 4160), ("sylvester", 256, 4096),
         ("sylvester", 512, 4096), ("sylvester", 4096, 8192), ("regular", 4, 1024), ("regular", 16, 1040),
         ("regular", 64, 4096), ("regular", 256, 11008 + 256)]


@pytest.mark.parametrize("kind,n,k", CASES)
@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16, torch.float32])
def test_hadamard_within_tolerance(qlin_gpu, kind, n, k, dtype):
    rows = 37
    xt = torch.from_numpy(_rows(n + k, rows, k)).to(dtype).cuda()
    signs = _signs(k, k) if n % 2 == 0 and (n // 2) % 2 == 0 else None
    y = qlin_gpu.qlin_hadamard(xt, n, kind=_code(qlin_gpu, kind),
                               signs=None if signs is None else torch.from_numpy(signs).cuda())
    torch.cuda.synchronize()
    assert qlin_gpu.qlin_get_device_error() == 0
    ref = oracle.hadamard_rotate(xt.double().cpu().numpy(), n, kind, signs)
    assert_within_tolerance(y.double().cpu().numpy(), ref, "%s n=%d %s" % (kind, n, dtype))


def test_hadamard_in_place(qlin_gpu):
    """Rotating a buffer onto itself gives what the out-of-place call gives."""
    x = torch.from_numpy(_rows(3, 16, 2048)).half().cuda()
    ref = oracle.hadamard_rotate(x.double().cpu().numpy(), 1024, "sylvester")
    out = qlin_gpu.qlin_hadamard(x, 1024)
    torch.cuda.synchronize()
    qlin_gpu.qlin_hadamard(x, 1024, y=x)
    torch.cuda.synchronize()
    assert torch.equal(x.cpu().view(torch.int16), out.cpu().view(torch.int16))
    assert_within_tolerance(x.double().cpu().numpy(), ref, "in place")


@pytest.mark.parametrize("kind,n,rows,k", [("sylvester", 8, 1, 8), ("regular", 4, 3, 8), ("sylvester", 8192, 2, 8192),
                                           ("regular", 256, 1, 256)])
def test_hadamard_small_and_largest(qlin_gpu, kind, n, rows, k):
    x = torch.from_numpy(np.random.default_rng(n + k).standard_normal((rows, k)).astype(np.float32)).cuda()
    y = qlin_gpu.qlin_hadamard(x, n, kind=_code(qlin_gpu, kind))
    torch.cuda.synchronize()
    ref = oracle.hadamard_rotate(x.double().cpu().numpy(), n, kind)
    # float32 rows: the float32 butterflies stay within (log2 n + 2) roundings
    # of 2^-24 times sqrt(n) max|x| of the exact rotation
    bound = (np.log2(n) + 2) * 2.0 ** -24 * np.sqrt(n) * np.abs(x.cpu().numpy()).max()
    assert np.max(np.abs(y.double().cpu().numpy() - ref)) <= bound
    assert_within_tolerance(y.double().cpu().numpy(), ref, "%s n=%d" % (kind, n))


def test_hadamard_page_example_on_gpu(qlin_gpu):
    """The page's 8-element token rotated by H_8 / sqrt(8) (QuaRot section),
    in float32, to the printed three decimals."""
    from conftest import load_golden
    ex = load_golden("hadamard_examples.json")["sylvester_h8"]
    x = torch.tensor([ex["x"]], dtype=torch.float32).cuda()
    y = qlin_gpu.qlin_hadamard(x, 8)
    torch.cuda.synchronize()
    assert np.all(np.abs(y.cpu().numpy()[0] - np.array(ex["xH_printed"])) <= 1e-3)


def _ulp_bound(ref, dtype):
    """One unit in the last place of the output dtype at each reference value."""
    bits = 10 if dtype == torch.float16 else 7
    mag = np.maximum(np.abs(ref), 2.0 ** (-14 if dtype == torch.float16 else -126))
    return 2.0 ** (np.floor(np.log2(mag)) - bits)


@pytest.mark.parametrize("kind,n,rows,k", [("sylvester", 256, 5, 256), ("regular", 256, 5, 768),
                                           ("sylvester", 256, 37, 4096 + 256), ("regular", 256, 64, 4096),
                                           ("sylvester", 4096, 1, 4096), ("sylvester", 4096, 3, 8192),
                                           ("sylvester", 4096, 40, 4096), ("sylvester", 512, 3, 1536),
                                           ("sylvester", 1024, 5, 2048), ("sylvester", 2048, 3, 2048),
                                           ("sylvester", 512, 16, 4096), ("sylvester", 512, 15, 512),
                                           ("sylvester", 1024, 3, 1024)])
@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16])
def test_hadamard_tensor_core_within_one_ulp(qlin_gpu, kind, n, rows, k, dtype):
    """Groups of 256 (both matrices) and Sylvester groups of 512 .. 4096 in
    fp16 / bf16 run as 16 x 16 products on the tensor cores, the intermediates kept
    to 16 significant bits (relative error 2^-17 each): every output is
    within one ulp of the output type of the exact rotation, plus 2^-14 of
    the row's largest output for the intermediates (the rotation is
    orthogonal, so that is far above their error and far below any wrong
    element), with and without column signs, ragged group counts (5, 15, 1, 6
    groups) included.  For n < 4096 the groups after the buffer's last whole
    block of 4096 elements run through the float32 butterflies: one, two,
    one and seven such groups here (after 1, 2, 1, 1 blocks), and a buffer
    smaller than one block (three groups of 1024)."""
    x = torch.from_numpy(_rows(7 * n + k, rows, k)).to(dtype).cuda()
    for signs in (None, _signs(k + 1, k)):
        y = qlin_gpu.qlin_hadamard(x, n, kind=_code(qlin_gpu, kind),
                                   signs=None if signs is None else torch.from_numpy(signs).cuda())
        torch.cuda.synchronize()
        assert qlin_gpu.qlin_get_device_error() == 0
        ref = oracle.hadamard_rotate(x.double().cpu().numpy(), n, kind, signs)
        got = y.double().cpu().numpy()
        slack = 2.0 ** -14 * np.abs(ref).max(axis=1, keepdims=True)
        assert np.all(np.abs(got - ref) <= _ulp_bound(ref, dtype) * 1.0001 + slack), (kind, n, dtype)
        assert_within_tolerance(got, ref, "%s n=%d %s" % (kind, n, dtype))


@pytest.mark.parametrize("n", [256, 4096])
def test_hadamard_tensor_core_in_place(qlin_gpu, n):
    """The tensor-core paths rotate a buffer onto itself exactly as out of place."""
    x = torch.from_numpy(_rows(11, 24, 8192)).half().cuda()
    out = qlin_gpu.qlin_hadamard(x, n)
    torch.cuda.synchronize()
    qlin_gpu.qlin_hadamard(x, n, y=x)
    torch.cuda.synchronize()
    assert torch.equal(x.cpu().view(torch.int16), out.cpu().view(torch.int16))
