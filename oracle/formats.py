"""Number formats used by the quantized linear layer (oracle side).

TEST INFRASTRUCTURE ONLY - see the package docstring.

* INT4 two's complement / unsigned nibbles and their packing
  ("LLM and AIGC quantization", sections "Integers" and "W4A16: packing").
* FP4 E2M1 and FP8 E4M3-FN, encoded by table lookup: the value set is listed
  once and a real number is mapped to the nearest listed value
  ("LLM and AIGC quantization", section "Floating point"; the E4M3-FN variant
  has no infinities, only S.1111.111 is NaN, so its largest finite value is
  1.75 x 2^8 = 448).

Readings where the pages are silent (each is listed in the design notes):

* Ties between two representable values go to the code whose lowest
  mantissa bit is 0 (IEEE round-half-to-even applied to the code, the same
  rule the pages use for integers).
* Values beyond the largest finite magnitude saturate to it (the pages' 500
  -> 448 example); NaN inputs are not handled.
* The sign is kept: a negative value whose magnitude rounds to 0 encodes as
  negative zero (sign bit set).

Parity pins: tests/test_oracle_pins.py (page examples, exhaustive decode
against torch's float8_e4m3fn, RNE ties checked at every midpoint).
"""

import numpy as np

# FP4 E2M1 magnitudes for codes 0..7; bit 3 of a code is the sign.
E2M1_MAGNITUDES = (0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0)


def e4m3_finite_magnitudes():
    """The 127 non-negative finite E4M3-FN values, indexed by code 0..126.

    Code layout S.EEEE.MMM with bias 7: exponent field 0 is subnormal
    (m/8 * 2^-6), otherwise (1 + m/8) * 2^(e-7).  Code 127 (S.1111.111) is
    NaN and is not part of the table.
    """
    vals = []
    for code in range(127):
        e = code >> 3
        m = code & 7
        if e == 0:
            vals.append((m / 8.0) * 2.0 ** -6)
        else:
            vals.append((1.0 + m / 8.0) * 2.0 ** (e - 7))
    return np.array(vals, dtype=np.float64)


_E2M1 = np.array(E2M1_MAGNITUDES, dtype=np.float64)
_E4M3 = e4m3_finite_magnitudes()


def _nearest_code(mag, table):
    """Index of the nearest table entry to each magnitude (table ascending).

    A magnitude exactly halfway between entries c and c+1 takes whichever of
    the two indices is even.  Anything above the last entry takes the last
    entry (saturation).  Comparisons are exact in float64.
    """
    mag = np.asarray(mag, dtype=np.float64)
    mids = (table[:-1] + table[1:]) / 2.0          # exact: dyadic values
    below = np.searchsorted(mids, mag, side="left")  # number of midpoints < mag
    idx = below.copy()
    on_mid = below < len(mids)
    tie = np.zeros(mag.shape, dtype=bool)
    tie[on_mid] = mag[on_mid] == mids[below[on_mid]]
    # On a midpoint between `below` and `below + 1`, step up only if the upper
    # code is the even one.
    step_up = tie & (((below + 1) % 2) == 0)
    idx = idx + step_up.astype(idx.dtype)
    return np.minimum(idx, len(table) - 1)


def e2m1_encode(v):
    """float32 array -> E2M1 codes (uint8, 0..15), sign in bit 3."""
    v = np.asarray(v, dtype=np.float32)
    mag_code = _nearest_code(np.abs(v).astype(np.float64), _E2M1)
    sign = np.signbit(v).astype(np.uint8)
    return (mag_code.astype(np.uint8) | (sign << 3)).astype(np.uint8)


def e2m1_decode(codes):
    """E2M1 codes (0..15) -> float64 values."""
    codes = np.asarray(codes, dtype=np.uint8)
    mag = _E2M1[codes & 7]
    return np.where((codes & 8) != 0, -mag, mag)


def e4m3_encode(v):
    """float32 array -> E4M3-FN codes (uint8), saturating at 448, sign in bit 7."""
    v = np.asarray(v, dtype=np.float32)
    mag_code = _nearest_code(np.abs(v).astype(np.float64), _E4M3)
    sign = np.signbit(v).astype(np.uint8)
    return (mag_code.astype(np.uint8) | (sign << 7)).astype(np.uint8)


def e4m3_decode(codes):
    """E4M3-FN codes -> float64 values (code 0x7F / 0xFF, NaN, is rejected)."""
    codes = np.asarray(codes, dtype=np.uint8)
    if np.any((codes & 0x7F) == 0x7F):
        raise ValueError("E4M3 NaN code in input")
    mag = _E4M3[codes & 0x7F]
    return np.where((codes & 0x80) != 0, -mag, mag)


def int4_decode(nibble, signed):
    """A 4-bit pattern read as two's complement (signed) or unsigned."""
    n = int(nibble) & 0xF
    if signed and n >= 8:
        return n - 16
    return n


def pack_u4(codes):
    """Pack 4-bit codes along the last axis, two per byte.

    Element 2i goes to the low nibble of byte i and element 2i+1 to the high
    nibble.  Read as little-endian 32-bit words this is the "q_i << 4i"
    packing of eight codes per int32 ("LLM and AIGC quantization", W4A16
    packing).  An odd trailing element leaves the high nibble zero.
    """
    codes = np.asarray(codes, dtype=np.uint8)
    if np.any(codes > 15):
        raise ValueError("code out of 4-bit range")
    n = codes.shape[-1]
    if n % 2:
        pad = np.zeros(codes.shape[:-1] + (1,), dtype=np.uint8)
        codes = np.concatenate([codes, pad], axis=-1)
    lo = codes[..., 0::2]
    hi = codes[..., 1::2]
    return (lo | (hi << 4)).astype(np.uint8)


def unpack_u4(packed, n):
    """Inverse of pack_u4: bytes -> the first n 4-bit codes along the last axis."""
    packed = np.asarray(packed, dtype=np.uint8)
    out = np.empty(packed.shape[:-1] + (packed.shape[-1] * 2,), dtype=np.uint8)
    out[..., 0::2] = packed & 0xF
    out[..., 1::2] = packed >> 4
    return out[..., :n]
