"""Online Hadamard rotation of activations before 4-bit quantization (oracle
side).  TEST INFRASTRUCTURE ONLY - see the package docstring.

Every group of n consecutive elements of a row along K is multiplied by the
normalized Hadamard matrix of order n, and the result optionally by a +-1
sign per column:

    y[g] = x[g] . H_n / sqrt(n),   then   y[:, k] = y[:, k] . signs[k]

computed in float64 from the matrix itself (one matrix product per group
size), so the only rounding is float64's.  Two matrices:

* Sylvester H_n, n a power of two ("LLM and AIGC quantization", QuaRot
  section: the Sylvester construction H_2n = [[H_n, H_n], [H_n, -H_n]], the
  randomized Q = H . diag(+-1); the worked example rotates an 8-element
  token by H_8 / sqrt(8)).
* Regular H_n, n = 4^k ("LLM and AIGC quantization", ConvRot section: K is
  cut into groups of N0 and every group is multiplied by the same regular
  Hadamard, built from the 4 x 4 regular matrix H4 by Kronecker products;
  every row and column sums to +-sqrt(n)).

Readings: the signs multiply the rotated columns (Q = H . diag(+-1) applied
as x . Q); a rotation of n = 8192 is computed with one Sylvester doubling
step, [a, b] . [[H, H], [H, -H]] = [a H + b H, a H - b H], so that no dense
matrix above 4096 x 4096 is built.

Pins: tests/test_oracle_pins.py (the pages' two worked examples, matrices
built two independent ways, orthogonality, column sums, involution).
"""
import numpy as np

H4 = np.array([[1, 1, 1, -1], [1, 1, -1, 1], [1, -1, 1, 1], [-1, 1, 1, 1]], dtype=np.float64)
_DENSE_MAX = 4096


def _is_pow(n, base):
    while n > 1 and n % base == 0:
        n //= base
    return n == 1


def sylvester_matrix(n):
    """H_n by the Sylvester doubling [[H, H], [H, -H]], float64, unnormalized."""
    h = np.ones((1, 1))
    while h.shape[0] < n:
        h = np.block([[h, h], [h, -h]])
    return h


def regular_matrix(n):
    """The Kronecker power of H4 of order n = 4^k, float64, unnormalized."""
    h = np.ones((1, 1))
    while h.shape[0] < n:
        h = np.kron(h, H4)
    return h


def _rotate_groups(g, n, kind):
    """g: float64 [m][n] -> g . H_n (unnormalized)."""
    if kind == "sylvester" and n > _DENSE_MAX:
        a = _rotate_groups(g[:, : n // 2], n // 2, kind)
        b = _rotate_groups(g[:, n // 2:], n // 2, kind)
        return np.concatenate([a + b, a - b], axis=1)
    h = sylvester_matrix(n) if kind == "sylvester" else regular_matrix(n)
    return g @ h


def hadamard_rotate(x, n, kind="sylvester", signs=None):
    """x [rows][K] (K a multiple of n) -> float64 [rows][K]: every n-group
    times H_n / sqrt(n), then times signs[k] per column (or no signs)."""
    x = np.asarray(x, dtype=np.float64)
    rows, k = x.shape
    if kind == "sylvester":
        if n < 2 or not _is_pow(n, 2):
            raise ValueError("n must be a power of two")
    elif kind == "regular":
        if n < 4 or not _is_pow(n, 4):
            raise ValueError("n must be a power of four")
    else:
        raise ValueError("kind must be 'sylvester' or 'regular'")
    if k % n:
        raise ValueError("n must divide K")
    y = (_rotate_groups(x.reshape(rows * (k // n), n), n, kind) / np.sqrt(float(n))).reshape(rows, k)
    if signs is not None:
        y = y * np.asarray(signs, dtype=np.float64)[None, :]
    return y
