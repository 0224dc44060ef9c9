"""Online Hadamard rotation of activations before 4-bit quantization (oracle
side).  TEST INFRASTRUCTURE ONLY - see the package docstring.

Two transforms, each applied to every group of n consecutive elements of a
row along K:

* Sylvester / fast Walsh-Hadamard ("LLM and AIGC quantization", QuaRot: the
  randomized Hadamard Q = H . diag(+-1); the fast transform is log2(n)
  butterfly stages, stage h mapping the pair (a, b) at distance h to
  (a + b, a - b)).  The stages run in the order h = 1, 2, 4, ..., n/2.
* Regular Hadamard of order n = 4^k ("LLM and AIGC quantization", ConvRot:
  K is cut into groups of N0 (default 256) and every group is multiplied by
  the same regular Hadamard, the k-fold Kronecker power of the 4 x 4 matrix
  H4 = [[1,1,1,-1],[1,1,-1,1],[1,-1,1,1],[-1,1,1,1]], whose column sums are
  +-sqrt(n); the group rotation is the block-diagonal diag(H, ..., H) and stays
  orthogonal).  Computed as k radix-4 stages at strides 1, 4, 16, ...; every
  quad (x0, x1, x2, x3) at one stride becomes y_i = s - 2 x_(3-i) with
  s = (x0 + x1) + (x2 + x3) (H4 = J - 2 . antidiag).

Both are then scaled by c = the float32 nearest 1/sqrt(n) (exactly 2^-k/2 for
even powers of two), and optionally multiplied by per-column signs
(diag(+-1) of QuaRot's Q = H . diag(+-1), column k of the row).  Every step
is one float32 operation in the order written; the result is rounded once
to the output type.  This fixed order is part of the operation's
definition (the pages give the butterflies, not an order of roundings).

Pins: tests/test_oracle_pins.py (dense products with the matrices built from
their definitions in float64, the regular matrix's +-1 response to a row of
ones, orthogonality: applying a transform twice gives back x).
"""
import numpy as np

F32 = np.float32
H4 = np.array([[1, 1, 1, -1], [1, 1, -1, 1], [1, -1, 1, 1], [-1, 1, 1, 1]], dtype=np.float64)


def _is_pow(n, base):
    while n > 1 and n % base == 0:
        n //= base
    return n == 1


def hadamard_scale(n):
    """c = float32(1 / sqrt(n))."""
    return F32(1.0 / np.sqrt(float(n)))


def fwht_rows(x, n):
    """Sylvester butterflies on every n-group of the rows of x (float32), unscaled."""
    x = np.asarray(x, dtype=F32)
    rows, k = x.shape
    if not _is_pow(n, 2) or n < 2 or k % n:
        raise ValueError("n must be a power of two dividing K")
    y = x.reshape(rows * (k // n), n).copy()
    h = 1
    while h < n:
        v = y.reshape(-1, n // (2 * h), 2, h)
        a = v[:, :, 0, :].copy()
        b = v[:, :, 1, :].copy()
        v[:, :, 0, :] = (a + b).astype(F32)
        v[:, :, 1, :] = (a - b).astype(F32)
        h *= 2
    return y.reshape(rows, k)


def regular_rows(x, n):
    """Radix-4 regular-Hadamard stages on every n-group of the rows (float32), unscaled."""
    x = np.asarray(x, dtype=F32)
    rows, k = x.shape
    if not _is_pow(n, 4) or n < 4 or k % n:
        raise ValueError("n must be a power of four dividing K")
    y = x.reshape(rows * (k // n), n).copy()
    d = 1
    while d < n:
        v = y.reshape(-1, n // (4 * d), 4, d)
        q = [v[:, :, i, :].copy() for i in range(4)]
        s = ((q[0] + q[1]).astype(F32) + (q[2] + q[3]).astype(F32)).astype(F32)
        for i in range(4):
            v[:, :, i, :] = (s - F32(2.0) * q[3 - i]).astype(F32)
        d *= 4
    return y.reshape(rows, k)


def hadamard_rotate(x, n, kind="sylvester", signs=None):
    """The rotation as the kernels compute it: float32 transform, times
    c = float32(1/sqrt(n)), times signs[k] (+-1 per column, or None).  float32 out."""
    t = fwht_rows(x, n) if kind == "sylvester" else regular_rows(x, n)
    y = (t * hadamard_scale(n)).astype(F32)
    if signs is not None:
        y = (y * np.asarray(signs, dtype=F32)[None, :]).astype(F32)
    return y


def sylvester_matrix(n):
    """H_n by the Sylvester doubling [[H, H], [H, -H]], float64, unnormalized."""
    h = np.ones((1, 1))
    while h.shape[0] < n:
        h = np.block([[h, h], [h, -h]])
    return h


def regular_matrix(n):
    """The k-fold Kronecker power of H4, float64, unnormalized."""
    h = np.ones((1, 1))
    while h.shape[0] < n:
        h = np.kron(h, H4)
    return h
