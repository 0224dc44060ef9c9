"""Online Hadamard rotation on the GPU against the CPU oracle, bit for bit:
the Sylvester fast Walsh-Hadamard transform (groups of 2 .. 4096, warp-level
and through shared memory) and the regular Hadamard of order 4^k, with and
without column signs, fp16 / bf16 / fp32 rows, in place."""

import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.gpu


def _rows(seed, rows, k):
    rng = np.random.default_rng(seed)
    x = (rng.standard_normal((rows, k)) * np.exp(rng.uniform(-3, 3, size=(rows, 1)))).astype(np.float32)
    x[1] = 0.0
    x[2, ::7] *= 100.0           # outlier channels, the case the rotation is for
    return x


def _signs(seed, k):
    return np.where(np.random.default_rng(seed).random(k) < 0.5, -1, 1).astype(np.int8)


def _expected(x32, n, kind, signs, dtype):
    y = oracle.hadamard_rotate(x32, n, kind, None if signs is None else signs.astype(np.float32))
    return torch.from_numpy(y).to(dtype)   # one round-to-nearest-even to the output type


CASES = [("sylvester", 2, 64), ("sylvester", 8, 1024), ("sylvester", 64, 4160), ("sylvester", 256, 4096),
         ("sylvester", 512, 4096), ("sylvester", 4096, 8192), ("regular", 4, 1024), ("regular", 16, 1040),
         ("regular", 64, 4096), ("regular", 256, 11008 + 256)]


@pytest.mark.parametrize("kind,n,k", CASES)
@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16, torch.float32])
def test_hadamard_bit_exact(qlin_gpu, kind, n, k, dtype):
    rows = 37
    x = _rows(n + k, rows, k)
    xt = torch.from_numpy(x).to(dtype).cuda()
    signs = _signs(k, k) if n % 2 == 0 and (n // 2) % 2 == 0 else None
    code = qlin_gpu.QLIN_HADAMARD_SYLVESTER if kind == "sylvester" else qlin_gpu.QLIN_HADAMARD_REGULAR
    y = qlin_gpu.qlin_hadamard(xt, n, kind=code, signs=None if signs is None else torch.from_numpy(signs).cuda())
    torch.cuda.synchronize()
    want = _expected(xt.float().cpu().numpy(), n, kind, signs, dtype)
    got = y.cpu()
    same = (got.view(torch.int16 if dtype != torch.float32 else torch.int32) ==
            want.view(torch.int16 if dtype != torch.float32 else torch.int32))
    bad = torch.nonzero(~same)
    assert bad.numel() == 0, "first mismatches (row, col): %s" % bad[:5].tolist()


def test_hadamard_in_place(qlin_gpu):
    x = _rows(3, 16, 2048)
    xt = torch.from_numpy(x).half().cuda()
    want = _expected(xt.float().cpu().numpy(), 1024, "sylvester", None, torch.float16)
    qlin_gpu.qlin_hadamard(xt, 1024, y=xt)
    torch.cuda.synchronize()
    assert torch.equal(xt.cpu().view(torch.int16), want.view(torch.int16))


@pytest.mark.parametrize("kind,n,rows,k", [("sylvester", 8, 1, 8), ("regular", 4, 3, 8), ("sylvester", 8192, 2, 8192)])
def test_hadamard_small_and_largest(qlin_gpu, kind, n, rows, k):
    x = np.random.default_rng(n + k).standard_normal((rows, k)).astype(np.float32)
    xt = torch.from_numpy(x).cuda()
    code = qlin_gpu.QLIN_HADAMARD_SYLVESTER if kind == "sylvester" else qlin_gpu.QLIN_HADAMARD_REGULAR
    y = qlin_gpu.qlin_hadamard(xt, n, kind=code)
    torch.cuda.synchronize()
    want = oracle.hadamard_rotate(x, n, kind)
    assert np.array_equal(y.cpu().numpy().view(np.uint32), want.view(np.uint32))
