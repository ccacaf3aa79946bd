"""W4A8-MXFP4: MXFP4 weights against activations quantised to MXFP8 on the
fly (oracle; test infrastructure only).

What is computed.  The Humming launch article ("Humming: Fast, Flexible
Kernels for Quantized Inference", paragraph "Efficient W4A8-MXFP4 inference on
existing GPUs") and the article "Ant Group's Humming Open-Sources Faster AI
Inference, Hitting 5x Gains" (section "Coverage reaches beyond standard PTX
types") pair MXFP4 weights with 8-bit floating-point activations, converting
the weights inside the kernel where the tensor cores lack MXFP4.  On a device
whose tensor cores take MX operands directly (sm_103's block-scaled MMA), both
operands of the product carry one UE8M0 exponent per 32 elements along K.
The pages do not define the activation side.  The reading here is the OCP
Microscaling (MX) v1.0 conversion to MXFP8 with e4m3 elements:

    shared exponent  Ex[m, b] = clamp(floor(log2(max_{k in b} |X[m, k]|)) - 8 + 127, 0, 254)
                     (8 = the largest exponent of a normal e4m3 value; an
                     all-zero block clamps to 0)
    elements         xq[m, k] = e4m3_rne_sat(X[m, k] / 2^(Ex[m, k // 32] - 127))
                     (round to nearest, ties to even; magnitudes above 448,
                     the largest e4m3 value, become 448; the sign of zero kept)
    product          Y[m, n] = sum_k e4m3(xq[m, k]) 2^(Ex[m, k//32] - 127)
                                   * e2m1(wq[n, k]) 2^(Ew[n, k//32] - 127)

Dividing a bf16 value by a power of two is exact, so every code decision
above is taken on the exact value; the product sums are float64.
"""
from __future__ import annotations

import numpy as np

from . import formats as F

E4M3_EMAX = 8          # largest exponent of a normal e4m3 value (448 = 1.75 * 2^8)
E4M3_MAX = 448.0
E4M3_MIN_EXP = -6      # smallest normal exponent; subnormals are multiples of 2^-9


def e4m3_encode(v: np.ndarray) -> np.ndarray:
    """float64 -> OCP e4m3 "fn" bytes: round to nearest even, saturate at 448.

    A magnitude a in binade [2^e, 2^(e+1)) (e >= -6) is a multiple of
    2^(e-3); below 2^-6 the grid is 2^-9 (subnormals).  Rounding up to the
    next binade's first value is itself on the grid, so one rounding to the
    quantum of a's binade is exact.
    """
    v = np.asarray(v, dtype=np.float64)
    a = np.minimum(np.abs(v), E4M3_MAX)
    _, ex = np.frexp(a)                                  # a = f 2^ex, f in [0.5, 1): floor(log2 a) = ex - 1
    e = np.maximum(np.where(a > 0, ex - 1, E4M3_MIN_EXP), E4M3_MIN_EXP)
    quantum = np.ldexp(1.0, (e - 3).astype(np.int32))
    r = np.round(a / quantum) * quantum                  # half to even on the binade's grid
    r = np.minimum(r, E4M3_MAX)
    # bit fields of the rounded magnitude
    _, rex = np.frexp(r)
    re = rex - 1
    normal = r >= 2.0 ** E4M3_MIN_EXP
    exp_field = np.where(normal, re + 7, 0)
    mant = np.where(normal, np.ldexp(r, (-re).astype(np.int32)) - 1.0, r / 2.0 ** -9) * np.where(normal, 8.0, 1.0)
    code = (exp_field.astype(np.int64) << 3) | np.rint(mant).astype(np.int64)
    sign = np.signbit(v).astype(np.int64) << 7
    return (sign | code).astype(np.uint8)


def mx_shared_exponent(amax: np.ndarray, emax: int) -> np.ndarray:
    """UE8M0 byte of a block: floor(log2(amax)) - emax + 127, clamped to [0, 254]."""
    amax = np.asarray(amax, dtype=np.float64)
    _, ex = np.frexp(amax)
    e = np.where(amax > 0, ex - 1 - emax + 127, 0)
    return np.clip(e, 0, 254).astype(np.uint8)


def mxfp8_quantize(x: np.ndarray):
    """Activations float64 [M, K] (K % 32 == 0) -> (e4m3 bytes [M, K], UE8M0 bytes [M, K/32])."""
    x = np.asarray(x, dtype=np.float64)
    m, k = x.shape
    xb = x.reshape(m, k // 32, 32)
    ex = mx_shared_exponent(np.abs(xb).max(axis=-1), E4M3_EMAX)
    scaled = np.ldexp(xb, (127 - ex.astype(np.int32))[..., None])
    return e4m3_encode(scaled).reshape(m, k), ex


def mxfp8_decode(codes: np.ndarray, exps: np.ndarray) -> np.ndarray:
    """(e4m3 bytes [M, K], UE8M0 bytes [M, K/32]) -> float64 [M, K]."""
    codes = np.asarray(codes)
    k = codes.shape[1]
    return F.e4m3_to_f64(codes) * F.ue8m0_to_f64(np.asarray(exps))[:, np.arange(k) // 32]


def w4a8_mxfp4_gemm(x: np.ndarray, w: np.ndarray) -> np.ndarray:
    """Y = mxfp8(x) . w^T: x float64 [M, K] (the 16-bit activations, decoded),
    w float64 [N, K] (the dequantised MXFP4 weight)."""
    xq, ex = mxfp8_quantize(x)
    return mxfp8_decode(xq, ex) @ np.asarray(w, dtype=np.float64).T
