"""Bit-level decoders of the storage formats (oracle; test infrastructure only).

Each decoder follows the published definition of its format, written out
field by field.  The Humming pages name these formats without defining them
(README "Support Matrix": FP16 e5m10, BF16 e8m7, FP8 e4m3, FP4 e2m1, INT1-8
with or without zero point; scale types BF16, FP16, E4M3, E5M2, UE8M0), so the
definitions are the standard ones:

* IEEE binary16 / bfloat16 (1 sign, 5|8 exponent, 10|7 mantissa bits)
* OCP 8-bit floating point e4m3 "fn": bias 7, no infinities, S.1111.111 = NaN
* OCP Microscaling (MX) v1.0: e2m1 elements (bias 1, one mantissa bit, no
  inf/NaN) and UE8M0 scales (2^(E-127), E = 255 is NaN)
* two's complement integers, and the little-endian nibble / 6-bit stream
  packing of the standard storage format (``synth`` module docstring).
"""
from __future__ import annotations

import numpy as np


# ---------------------------------------------------------------------------
# integer code unpacking
# ---------------------------------------------------------------------------
def unpack_nibbles(packed: np.ndarray, count: int) -> np.ndarray:
    """uint8 [..., ceil(count/2)] -> int64 [..., count]; even index = low nibble."""
    p = np.asarray(packed, dtype=np.uint8).astype(np.int64)
    lo = p & 0x0F
    hi = (p >> 4) & 0x0F
    out = np.empty(p.shape[:-1] + (2 * p.shape[-1],), dtype=np.int64)
    out[..., 0::2] = lo
    out[..., 1::2] = hi
    return out[..., :count]


def unpack_int6(packed: np.ndarray, count: int) -> np.ndarray:
    """uint8 [..., 3*ceil(count/4)] little-endian 6-bit stream -> int64 [..., count].

    Code j of a row occupies stream bits [6j, 6j+6); three bytes hold four codes.
    """
    p = np.asarray(packed, dtype=np.uint8).astype(np.int64)
    trip = p.reshape(p.shape[:-1] + (p.shape[-1] // 3, 3))
    word = trip[..., 0] | (trip[..., 1] << 8) | (trip[..., 2] << 16)   # 24-bit groups
    out = np.empty(word.shape + (4,), dtype=np.int64)
    for j in range(4):
        out[..., j] = (word >> (6 * j)) & 0x3F
    return out.reshape(p.shape[:-1] + (-1,))[..., :count]


def twos_complement(u: np.ndarray, bits: int) -> np.ndarray:
    """Interpret unsigned bits-wide codes as two's complement integers."""
    u = np.asarray(u, dtype=np.int64)
    return np.where(u >= (1 << (bits - 1)), u - (1 << bits), u)


# ---------------------------------------------------------------------------
# floating point element formats
# ---------------------------------------------------------------------------
def e2m1_to_f64(code: np.ndarray) -> np.ndarray:
    """OCP MX e2m1: bit 3 sign, bits 2..1 exponent (bias 1), bit 0 mantissa.

    exponent 0 is subnormal: value = m * 2^-1; otherwise 2^(e-1) * (1 + m/2).
    """
    c = np.asarray(code, dtype=np.int64) & 0x0F
    s = (c >> 3) & 1
    e = (c >> 1) & 3
    m = c & 1
    mag = np.where(e == 0, m * 0.5, np.exp2(e - 1.0) * (1.0 + m / 2.0))
    return np.where(s == 1, -mag, mag)


def ue8m0_to_f64(e: np.ndarray) -> np.ndarray:
    """OCP MX scale: 2^(E - 127); E = 255 encodes NaN."""
    e = np.asarray(e, dtype=np.int64)
    return np.where(e == 255, np.nan, np.exp2(e - 127.0))


def e4m3_to_f64(b: np.ndarray) -> np.ndarray:
    """OCP e4m3 'fn': 1 sign, 4 exponent (bias 7), 3 mantissa; S.1111.111 is NaN.

    exponent 0 is subnormal: (m/8) * 2^-6; otherwise 2^(e-7) * (1 + m/8).
    """
    b = np.asarray(b, dtype=np.int64) & 0xFF
    s = (b >> 7) & 1
    e = (b >> 3) & 0x0F
    m = b & 7
    mag = np.where(e == 0, (m / 8.0) * 2.0 ** -6, np.exp2(e - 7.0) * (1.0 + m / 8.0))
    mag = np.where((e == 15) & (m == 7), np.nan, mag)
    return np.where(s == 1, -mag, mag)


def _binary16_like(u: np.ndarray, ebits: int, mbits: int) -> np.ndarray:
    u = np.asarray(u, dtype=np.int64) & 0xFFFF
    bias = (1 << (ebits - 1)) - 1
    s = (u >> (ebits + mbits)) & 1
    e = (u >> mbits) & ((1 << ebits) - 1)
    m = u & ((1 << mbits) - 1)
    frac = m / float(1 << mbits)
    emax = (1 << ebits) - 1
    mag = np.where(e == 0, frac * 2.0 ** (1 - bias), np.exp2(e - float(bias)) * (1.0 + frac))
    mag = np.where(e == emax, np.where(m == 0, np.inf, np.nan), mag)
    return np.where(s == 1, -mag, mag)


def bf16_to_f64(u: np.ndarray) -> np.ndarray:
    """bfloat16 bits: 1 sign, 8 exponent (bias 127), 7 mantissa."""
    return _binary16_like(u, 8, 7)


def fp16_to_f64(u: np.ndarray) -> np.ndarray:
    """IEEE binary16 bits: 1 sign, 5 exponent (bias 15), 10 mantissa."""
    return _binary16_like(u, 5, 10)


def scale16_to_f64(u: np.ndarray, stype: str) -> np.ndarray:
    if stype == "bf16":
        return bf16_to_f64(u)
    if stype == "fp16":
        return fp16_to_f64(u)
    raise ValueError(f"16-bit scale type expected, got {stype}")
