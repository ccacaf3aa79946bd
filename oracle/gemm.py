"""Dequantisation and the dense quantized GEMM (oracle; test infrastructure only).

What is computed (Humming launch article, "Humming: Fast, Flexible Kernels for
Quantized Inference", paragraphs on the standard format and WnA16; README
usage example, which compares the layer output with ``inputs.matmul(weight.T)``):

    Y[m, n] = sum_k a[m, k] * w[n, k]

with w the dequantised weight and a the decoded activation.  Readings of the
formats (the pages name them but print no formula):

* int, symmetric:   w = q * s[n, g(k)]            q two's complement
* int, asymmetric:  w = (q - z[n, g(k)]) * s[n, g(k)]   q, z unsigned
  (the "dynamic zero point" of the README support matrix; subtract first)
* channelwise (group_k = 0): one scale (and zero) per row, g(k) = 0
* mxfp4:            w = e2m1(q) * 2^(E[n, k//32] - 127)
* nvfp4:            w = e2m1(q) * e4m3(s[n, k//16]) * g
                    (one e4m3 scale per 16 along K and a float32 tensor
                    scale g per expert: the aiwiki article's "secondary
                    scales" and "tensor scaling", section "Quantization
                    representation"; the launch article names NVFP4 beside
                    INT4, the B300 MoE results name NVFP4 and MXINT4)
* mxint4:           w = q * 2^(E[n, k//32] - 127),  q 4-bit two's complement
                    (integer codes under the MX block exponent of mxfp4)
* fp8 block:        w = e4m3(q) * s_w[n//128, k//128];
                    a = e4m3(xq) * s_x[m, k//128]
  so that Y = sum over 128-K blocks of s_x * s_w * (e4m3 dot product), the
  block-scaled form of the plain definition.

The int, mxfp4 and mxint4 dequantised values are exact in float32 (at most 12
significant bits), so dequantising in float64 here equals dequantising to
float32; an nvfp4 value (at most 6 significant bits before g, 30 after) is
exact in float64.  Products and sums are float64.
"""
from __future__ import annotations

import numpy as np

from . import formats as F


def _groups(k: int, group_k: int) -> int:
    return 1 if group_k == 0 else k // group_k


def _group_index(k: int, group_k: int) -> np.ndarray:
    """Group g(k) of every column k."""
    if group_k == 0:
        return np.zeros(k, dtype=np.int64)
    return np.arange(k) // group_k


def dequantize(wtype: str, n: int, k: int, codes: np.ndarray, scales: np.ndarray,
               zeros: np.ndarray | None = None, group_k: int = 128, signed: bool = True,
               stype: str = "bf16", num_experts: int = 1, tensor_scale=None) -> np.ndarray:
    """Standard-format weight -> float64 [E, N, K].

    ``tensor_scale``: nvfp4 only, float32 [E] (one secondary scale per expert).
    """
    e = num_experts
    codes = np.asarray(codes).reshape(e, n, -1)
    if wtype in ("int4", "int6"):
        bits = 4 if wtype == "int4" else 6
        unpack = F.unpack_nibbles if bits == 4 else F.unpack_int6
        u = unpack(codes, k)                                   # [E, N, K] unsigned
        g = _groups(k, group_k)
        gi = _group_index(k, group_k)
        s = F.scale16_to_f64(np.asarray(scales).reshape(e, n, g), stype)[:, :, gi]
        if zeros is not None:
            z = unpack(np.asarray(zeros).reshape(e, n, -1), g)[:, :, gi]
            return (u - z) * s
        q = F.twos_complement(u, bits) if signed else u
        return q * s
    if wtype == "mxfp4":
        u = F.unpack_nibbles(codes, k)
        sc = F.ue8m0_to_f64(np.asarray(scales).reshape(e, n, k // 32))[:, :, np.arange(k) // 32]
        return F.e2m1_to_f64(u) * sc
    if wtype == "nvfp4":
        u = F.unpack_nibbles(codes, k)
        sc = F.e4m3_to_f64(np.asarray(scales).reshape(e, n, k // 16))[:, :, np.arange(k) // 16]
        g = np.asarray(tensor_scale, dtype=np.float32).astype(np.float64).reshape(e, 1, 1)
        return F.e2m1_to_f64(u) * sc * g
    if wtype == "mxint4":
        q = F.twos_complement(F.unpack_nibbles(codes, k), 4)
        sc = F.ue8m0_to_f64(np.asarray(scales).reshape(e, n, k // 32))[:, :, np.arange(k) // 32]
        return q * sc
    if wtype == "fp8":
        q = F.e4m3_to_f64(codes[..., :k])
        sw = np.asarray(scales, dtype=np.float32).astype(np.float64).reshape(e, -(-n // 128), -(-k // 128))
        sw = sw[:, np.arange(n) // 128][:, :, np.arange(k) // 128]
        return q * sw
    raise ValueError(wtype)


def decode_activations(atype: str, data: np.ndarray, scales: np.ndarray | None = None) -> np.ndarray:
    """Activation storage -> float64 [M, K]."""
    if atype == "bf16":
        return F.bf16_to_f64(data)
    if atype == "fp16":
        return F.fp16_to_f64(data)
    if atype == "fp8":
        a = F.e4m3_to_f64(data)
        k = a.shape[1]
        s = np.asarray(scales, dtype=np.float32).astype(np.float64)
        return a * s[:, np.arange(k) // 128]
    raise ValueError(atype)


def gemm_dense(a: np.ndarray, w: np.ndarray) -> np.ndarray:
    """Y = a . w^T in float64; a [M, K], w [N, K] (or [1, N, K])."""
    w = np.asarray(w, dtype=np.float64)
    if w.ndim == 3:
        assert w.shape[0] == 1
        w = w[0]
    return np.asarray(a, dtype=np.float64) @ w.T


def reference(qw, acts) -> np.ndarray:
    """Convenience: oracle output for a ``synth.QuantWeight`` and ``synth.Activations``."""
    w = dequantize(qw.wtype, qw.n, qw.k, qw.codes, qw.scales, qw.zeros, qw.group_k,
                   qw.signed, qw.stype, qw.num_experts, getattr(qw, "tensor_scale", None))
    a = decode_activations(acts.atype, acts.data, acts.scales)
    return gemm_dense(a, w)
