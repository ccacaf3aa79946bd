"""Seeded synthetic inputs for the quantized GEMM workloads.

This module is shared by the CPU oracle tests, the GPU parity tests and the
benchmark.  It only *draws* inputs and encodes them into the standard storage
format (packed codes plus scales and zero points).  It holds none of the
method's arithmetic: nothing here dequantises codes or multiplies matrices, so
a mistake in an encoder here can only change *which* valid codes are drawn,
never the agreement between the oracle and the CUDA path (both decode the same
codes independently).

Standard storage format (the "standard format" of the Humming launch article,
section on representing the quantized computation, and the schema of the
aiwiki Humming article, section "Quantization representation": weights, scales,
zero points and group size as separate tensors, with an expert dimension for
MoE).  All arrays are C-contiguous numpy arrays with a leading expert axis E
(E = 1 for dense layers):

* int4   codes  uint8 [E, N, ceil(K/2)]; element k of a row sits in byte k//2,
                low nibble for even k.  Symmetric: 4-bit two's complement
                (-8..7).  Asymmetric: unsigned 0..15.
* int6   codes  uint8 [E, N, 3*K/4]; little-endian bit stream per row, code k
                occupies bits [6k, 6k+6); symmetric codes are 6-bit two's
                complement (-32..31), asymmetric codes unsigned 0..63.
* mxfp4  codes  uint8 [E, N, ceil(K/2)], nibbles as int4, each nibble an OCP
                e2m1 value (bit 3 sign, bits 2..1 exponent, bit 0 mantissa).
* fp8    codes  uint8 [E, N, K], OCP e4m3 ("fn" variant) bytes.
* nvfp4  codes  as mxfp4; scales e4m3 bytes uint8 [E, N, K/16]; plus a
                float32 tensor scale per expert, tensor_scale [E].
* mxint4 codes  as symmetric int4; scales UE8M0 bytes uint8 [E, N, K/32].
* scales        int formats: bf16/fp16 bit patterns uint16 [E, N, G] with
                G = K/group_k groups (G = 1 for channelwise, group_k = 0);
                mxfp4: UE8M0 exponent bytes uint8 [E, N, K/32];
                fp8: float32 [E, ceil(N/128), ceil(K/128)].
* zeros         int formats only, same bit packing as that format's codes,
                uint8 [E, N, packed(G)].
* activations   bf16/fp16 bit patterns uint16 [M, K], or e4m3 bytes uint8
                [M, K] with float32 per-token per-128-K-group scales
                [M, ceil(K/128)].
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import Optional

import numpy as np
import torch

__all__ = [
    "QuantWeight", "Activations", "MoeRouting",
    "to_bf16_bits", "to_fp16_bits", "to_e4m3_bytes",
    "pack_nibbles", "pack_int6",
    "quantize_int_groupwise", "quantize_fp8_block", "quantize_mxfp4", "quantize_nvfp4", "quantize_mxint4",
    "quantize_fp8_acts", "make_activations", "make_routing",
    "dense_w4a16_sym", "dense_w4a16_asym", "dense_int6_channel",
    "dense_fp8_block", "moe_mxfp4", "random_codes_weight",
]


# ---------------------------------------------------------------------------
# containers
# ---------------------------------------------------------------------------
@dataclass
class QuantWeight:
    """One quantized weight in the standard storage format (see module doc)."""
    wtype: str                 # "int4" | "int6" | "mxfp4" | "fp8" | "nvfp4" | "mxint4"
    n: int
    k: int
    num_experts: int
    group_k: int               # 0 = channelwise
    group_n: int               # 1, or 128 for fp8 block scales
    stype: str                 # "bf16" | "fp16" | "ue8m0" | "fp32" | "e4m3"
    signed: bool               # int formats: symmetric two's complement codes
    codes: np.ndarray
    scales: np.ndarray
    zeros: Optional[np.ndarray] = None
    tensor_scale: Optional[np.ndarray] = None   # nvfp4: float32 [E]

    @property
    def has_zeros(self) -> bool:
        return self.zeros is not None


@dataclass
class Activations:
    atype: str                 # "bf16" | "fp16" | "fp8"
    m: int
    k: int
    data: np.ndarray           # uint16 bits [M, K] or uint8 e4m3 [M, K]
    scales: Optional[np.ndarray] = None   # fp8 only: float32 [M, ceil(K/128)]


@dataclass
class MoeRouting:
    topk_ids: np.ndarray       # int32 [T, topk]
    topk_w: np.ndarray         # float32 [T, topk]
    extra: dict = field(default_factory=dict)


# ---------------------------------------------------------------------------
# rounding to storage types (library casts, round-to-nearest-even)
# ---------------------------------------------------------------------------
def to_bf16_bits(a: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16).copy()


def to_fp16_bits(a: np.ndarray) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.float64).astype(np.float16).view(np.uint16).copy()


def _bits16_to_f64(bits: np.ndarray, kind: str) -> np.ndarray:
    # generator-side helper used only to quantise with the *stored* scale
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16))
    t = t.view(torch.bfloat16 if kind == "bf16" else torch.float16)
    return t.double().numpy()


def to_e4m3_bytes(a: np.ndarray) -> np.ndarray:
    """Round to e4m3fn (RNE) and saturate to +-448 first (torch does not)."""
    a = np.clip(np.asarray(a, dtype=np.float32), -448.0, 448.0)
    t = torch.from_numpy(np.ascontiguousarray(a)).to(torch.float8_e4m3fn)
    return t.view(torch.uint8).numpy().copy()


def _e4m3_bytes_to_f64(b: np.ndarray) -> np.ndarray:
    return torch.from_numpy(np.ascontiguousarray(b)).view(torch.float8_e4m3fn).double().numpy()


def _rne(a: np.ndarray) -> np.ndarray:
    return np.rint(a)   # numpy rint rounds half to even


# ---------------------------------------------------------------------------
# bit packing into the standard storage format
# ---------------------------------------------------------------------------
def pack_nibbles(u: np.ndarray) -> np.ndarray:
    """uint [..., K] values 0..15 -> uint8 [..., ceil(K/2)], low nibble = even k."""
    u = np.asarray(u).astype(np.uint8) & 0x0F
    k = u.shape[-1]
    if k % 2:
        u = np.concatenate([u, np.zeros(u.shape[:-1] + (1,), np.uint8)], axis=-1)
    return (u[..., 0::2] | (u[..., 1::2] << 4)).astype(np.uint8)


def pack_int6(u: np.ndarray) -> np.ndarray:
    """uint [..., K] values 0..63 (K % 4 == 0) -> uint8 [..., 3K/4] LE bit stream."""
    u = np.asarray(u).astype(np.uint32) & 0x3F
    k = u.shape[-1]
    assert k % 4 == 0, "int6 rows must hold a multiple of 4 codes"
    q = u.reshape(u.shape[:-1] + (k // 4, 4))
    v = q[..., 0] | (q[..., 1] << 6) | (q[..., 2] << 12) | (q[..., 3] << 18)
    out = np.stack([v & 0xFF, (v >> 8) & 0xFF, (v >> 16) & 0xFF], axis=-1)
    return out.reshape(u.shape[:-1] + (3 * k // 4,)).astype(np.uint8)


def _pack_codes(wtype: str, u: np.ndarray) -> np.ndarray:
    return pack_nibbles(u) if wtype in ("int4", "mxfp4") else pack_int6(u)


# ---------------------------------------------------------------------------
# quantisers (test-side only; the oracle consumes the codes they produce)
# ---------------------------------------------------------------------------
def quantize_int_groupwise(w: np.ndarray, bits: int, group_k: int, symmetric: bool,
                           stype: str = "bf16") -> QuantWeight:
    """w float [E, N, K] -> int codes with per-group (or per-row) scales.

    symmetric:  s = round_s(absmax/qmax), q = clamp(rne(w/s), -2^(b-1), 2^(b-1)-1)
    asymmetric: s = round_s((max-min)/(2^b-1)), z = clamp(rne(-min/s), 0, 2^b-1),
                q = clamp(rne(w/s) + z, 0, 2^b-1)
    Quantisation divides by the *stored* (rounded) scale.  A zero range gives
    s = 1, z = 0.
    """
    w = np.asarray(w, dtype=np.float64)
    e, n, k = w.shape
    g = k if group_k == 0 else group_k
    assert k % g == 0
    ng = k // g
    wg = w.reshape(e, n, ng, g)
    to_bits = to_bf16_bits if stype == "bf16" else to_fp16_bits
    if symmetric:
        qmax = 2 ** (bits - 1) - 1
        amax = np.abs(wg).max(axis=-1)
        s_raw = np.where(amax > 0, amax / qmax, 1.0)
        s_bits = to_bits(s_raw)
        s = _bits16_to_f64(s_bits, stype)
        s = np.where(s > 0, s, 1.0)
        s_bits = to_bits(s)
        q = np.clip(_rne(wg / s[..., None]), -qmax - 1, qmax).astype(np.int64)
        u = (q & (2 ** bits - 1)).reshape(e, n, k)
        zeros = None
    else:
        qmax = 2 ** bits - 1
        lo = wg.min(axis=-1)
        hi = wg.max(axis=-1)
        s_raw = np.where(hi > lo, (hi - lo) / qmax, 1.0)
        s_bits = to_bits(s_raw)
        s = _bits16_to_f64(s_bits, stype)
        s = np.where(s > 0, s, 1.0)
        s_bits = to_bits(s)
        z = np.clip(_rne(-lo / s), 0, qmax).astype(np.int64)
        z = np.where(hi > lo, z, 0)
        q = np.clip(_rne(wg / s[..., None]) + z[..., None], 0, qmax).astype(np.int64)
        u = q.reshape(e, n, k)
        zeros = _pack_codes("int4" if bits == 4 else "int6", _pad_groups_for_pack(z, bits))
    wtype = "int4" if bits == 4 else "int6"
    return QuantWeight(wtype=wtype, n=n, k=k, num_experts=e, group_k=group_k, group_n=1,
                       stype=stype, signed=symmetric, codes=_pack_codes(wtype, u),
                       scales=s_bits.reshape(e, n, ng), zeros=zeros)


def _pad_groups_for_pack(z: np.ndarray, bits: int) -> np.ndarray:
    # int6 zero rows are bit streams too, so pad the group count to a multiple of 4
    if bits == 6 and z.shape[-1] % 4:
        pad = 4 - z.shape[-1] % 4
        z = np.concatenate([z, np.zeros(z.shape[:-1] + (pad,), z.dtype)], axis=-1)
    return z


def quantize_fp8_block(w: np.ndarray) -> QuantWeight:
    """w [E, N, K] -> e4m3 codes with float32 128x128 block scales absmax/448."""
    w = np.asarray(w, dtype=np.float64)
    e, n, k = w.shape
    nb, kb = -(-n // 128), -(-k // 128)
    s = np.ones((e, nb, kb), np.float32)
    codes = np.zeros((e, n, k), np.uint8)
    for bi in range(nb):
        for bj in range(kb):
            blk = w[:, bi * 128:(bi + 1) * 128, bj * 128:(bj + 1) * 128]
            amax = np.abs(blk).reshape(e, -1).max(axis=-1)
            sc = np.where(amax > 0, amax / 448.0, 1.0).astype(np.float32)
            s[:, bi, bj] = sc
            codes[:, bi * 128:(bi + 1) * 128, bj * 128:(bj + 1) * 128] = to_e4m3_bytes(
                blk / sc.astype(np.float64)[:, None, None])
    return QuantWeight(wtype="fp8", n=n, k=k, num_experts=e, group_k=128, group_n=128,
                       stype="fp32", signed=True, codes=codes, scales=s)


_E2M1_GRID = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])


def _e2m1_encode(v: np.ndarray) -> np.ndarray:
    """Round to the nearest e2m1 value (ties to the even code), saturating at 6.

    The magnitude code is the number of decision thresholds (midpoints of the
    grid 0, .5, 1, 1.5, 2, 3, 4, 6) that |v| passes; at a midpoint the
    comparison is strict or not so that the tie lands on the even code.
    """
    a = np.abs(v)
    code = (a > 0.25).view(np.uint8) + (a >= 0.75).view(np.uint8)
    for thr, strict in ((1.25, True), (1.75, False), (2.5, True), (3.5, False), (5.0, True)):
        code += (a > thr).view(np.uint8) if strict else (a >= thr).view(np.uint8)
    sign = (np.signbit(v) & (code > 0)).view(np.uint8)
    return (sign << 3) | code


def quantize_mxfp4(w: np.ndarray) -> QuantWeight:
    """w [E, N, K] -> e2m1 codes with one UE8M0 scale per 32 values along K.

    Shared exponent per block of 32 = floor(log2(absmax)) - 2 (2 is the largest
    e2m1 exponent), biased by 127 and clamped to [0, 254]; elements are
    rounded to e2m1 after division by 2^(E-127), saturating at 6.
    """
    w = np.asarray(w)
    if w.dtype not in (np.float32, np.float64):
        w = w.astype(np.float64)
    e, n, k = w.shape
    assert k % 32 == 0
    wg = w.reshape(e, n, k // 32, 32)
    amax = np.abs(wg).max(axis=-1)
    _, ex = np.frexp(amax)                       # amax = f * 2^ex, f in [0.5, 1): floor(log2) = ex - 1
    big = np.where(amax > 0, np.clip(ex - 1 - 2 + 127, 0, 254), 127).astype(np.int64)
    scaled = np.ldexp(wg, (127 - big)[..., None].astype(np.int32))
    u = _e2m1_encode(scaled).reshape(e, n, k)
    return QuantWeight(wtype="mxfp4", n=n, k=k, num_experts=e, group_k=32, group_n=1,
                       stype="ue8m0", signed=True, codes=pack_nibbles(u),
                       scales=big.astype(np.uint8).reshape(e, n, k // 32))


def quantize_nvfp4(w: np.ndarray) -> QuantWeight:
    """w [E, N, K] -> e2m1 codes, one e4m3 scale per 16 values along K and one
    float32 tensor scale per expert.

    g = float32(absmax of the expert / (6 * 448)), so that every block scale
    fits e4m3; block scale s = e4m3(absmax_16 / 6 / g) (round to nearest even,
    saturating); elements are rounded to e2m1 after division by the stored
    s * g, saturating at 6.  A block whose scale rounds to zero stores 1.0; an
    all-zero expert g = 1.
    """
    w = np.asarray(w, dtype=np.float64)
    e, n, k = w.shape
    assert k % 16 == 0
    amax_e = np.abs(w.reshape(e, -1)).max(axis=1)
    g = np.where(amax_e > 0, amax_e / (6.0 * 448.0), 1.0).astype(np.float32)
    gd = g.astype(np.float64)[:, None, None]
    wg = w.reshape(e, n, k // 16, 16)
    sb = to_e4m3_bytes(np.abs(wg).max(axis=-1) / 6.0 / gd)
    sb = np.where(_e4m3_bytes_to_f64(sb) > 0, sb, np.uint8(0x38)).astype(np.uint8)   # 0x38 = 1.0
    div = _e4m3_bytes_to_f64(sb)[..., None] * gd[..., None]
    u = _e2m1_encode(wg / div).reshape(e, n, k)
    return QuantWeight(wtype="nvfp4", n=n, k=k, num_experts=e, group_k=16, group_n=1, stype="e4m3",
                       signed=True, codes=pack_nibbles(u), scales=sb.reshape(e, n, k // 16), tensor_scale=g)


def quantize_mxint4(w: np.ndarray) -> QuantWeight:
    """w [E, N, K] -> 4-bit two's complement codes with one UE8M0 scale per 32
    values along K.

    Shared exponent per block = floor(log2(absmax)) - 2, so absmax / 2^(E-127)
    lies in [4, 8); biased by 127 and clamped to [0, 254]; q = clamp(rne(w /
    2^(E-127)), -8, 7).  A zero block takes E = 127.
    """
    w = np.asarray(w, dtype=np.float64)
    e, n, k = w.shape
    assert k % 32 == 0
    wg = w.reshape(e, n, k // 32, 32)
    amax = np.abs(wg).max(axis=-1)
    _, ex = np.frexp(amax)
    big = np.where(amax > 0, np.clip(ex - 1 - 2 + 127, 0, 254), 127).astype(np.int64)
    q = np.clip(_rne(np.ldexp(wg, (127 - big)[..., None].astype(np.int32))), -8, 7).astype(np.int64)
    return QuantWeight(wtype="mxint4", n=n, k=k, num_experts=e, group_k=32, group_n=1, stype="ue8m0",
                       signed=True, codes=pack_nibbles((q & 0xF).reshape(e, n, k)),
                       scales=big.astype(np.uint8).reshape(e, n, k // 32))


def quantize_fp8_acts(x: np.ndarray) -> Activations:
    """x [M, K] -> e4m3 bytes with float32 per-token per-128-K-group scales."""
    x = np.asarray(x, dtype=np.float64)
    m, k = x.shape
    kb = -(-k // 128)
    s = np.ones((m, kb), np.float32)
    q = np.zeros((m, k), np.uint8)
    for j in range(kb):
        blk = x[:, j * 128:(j + 1) * 128]
        amax = np.abs(blk).max(axis=-1)
        sc = np.where(amax > 0, amax / 448.0, 1.0).astype(np.float32)
        s[:, j] = sc
        q[:, j * 128:(j + 1) * 128] = to_e4m3_bytes(blk / sc.astype(np.float64)[:, None])
    return Activations(atype="fp8", m=m, k=k, data=q, scales=s)


def make_activations(rng: np.random.Generator, m: int, k: int, atype: str = "bf16",
                     std: float = 1.0) -> Activations:
    x = rng.standard_normal((m, k)) * std
    if atype == "bf16":
        return Activations("bf16", m, k, to_bf16_bits(x))
    if atype == "fp16":
        return Activations("fp16", m, k, to_fp16_bits(x))
    if atype == "fp8":
        return quantize_fp8_acts(x)
    raise ValueError(atype)


def make_routing(rng: np.random.Generator, tokens: int, num_experts: int, topk: int = 8) -> MoeRouting:
    """Top-k routing from softmax(logits + per-expert bias), both N(0,1).

    The per-expert bias makes the expert loads skewed.  The selected
    probabilities are renormalised to sum to one per token.
    """
    logits = rng.standard_normal((tokens, num_experts))
    bias = rng.standard_normal(num_experts)
    z = logits + bias
    z = z - z.max(axis=1, keepdims=True)
    p = np.exp(z)
    p /= p.sum(axis=1, keepdims=True)
    ids = np.argsort(-p, axis=1, kind="stable")[:, :topk]
    w = np.take_along_axis(p, ids, axis=1)
    w = w / w.sum(axis=1, keepdims=True)
    return MoeRouting(ids.astype(np.int32), w.astype(np.float32), {"bias": bias})


# ---------------------------------------------------------------------------
# the workloads (seeded), shaped like the benchmark configurations
# ---------------------------------------------------------------------------
def dense_w4a16_sym(seed: int, m: int, n: int, k: int, group_k: int = 128):
    """Symmetric INT4 g128 bf16 scales, bf16 activations; W~N(0,0.02), X~N(0,1)."""
    rng = np.random.default_rng(seed)
    w = rng.standard_normal((1, n, k)) * 0.02
    qw = quantize_int_groupwise(w, 4, group_k, True, "bf16")
    return qw, make_activations(rng, m, k, "bf16")


def dense_w4a16_asym(seed: int, m: int, n: int, k: int, group_k: int = 128):
    """Asymmetric INT4 g128 with uint4 zero points, bf16 scales and activations."""
    rng = np.random.default_rng(seed)
    w = rng.standard_normal((1, n, k)) * 0.02
    qw = quantize_int_groupwise(w, 4, group_k, False, "bf16")
    return qw, make_activations(rng, m, k, "bf16")


def dense_int6_channel(seed: int, m: int, n: int, k: int):
    """Symmetric INT6 channelwise (one fp16 scale per row), fp16 activations."""
    rng = np.random.default_rng(seed)
    w = rng.standard_normal((1, n, k)) * 0.02
    qw = quantize_int_groupwise(w, 6, 0, True, "fp16")
    return qw, make_activations(rng, m, k, "fp16")


def dense_fp8_block(seed: int, m: int, n: int, k: int):
    """e4m3 weights with fp32 128x128 block scales, e4m3 per-token-group activations."""
    rng = np.random.default_rng(seed)
    w = rng.standard_normal((1, n, k)) * 0.02
    qw = quantize_fp8_block(w)
    return qw, make_activations(rng, m, k, "fp8")


def moe_mxfp4(seed: int, tokens: int, num_experts: int = 128, n: int = 1536, k: int = 2048,
              topk: int = 8):
    """MoE gate+up weights in MXFP4 with bf16 activations and skewed top-k routing."""
    rng = np.random.default_rng(seed)
    codes, scales = [], []
    for e0 in range(0, num_experts, 8):          # chunks of experts bound the memory
        ne = min(8, num_experts - e0)
        part = quantize_mxfp4(rng.standard_normal((ne, n, k), dtype=np.float32) * np.float32(0.02))
        codes.append(part.codes)
        scales.append(part.scales)
    qw = QuantWeight("mxfp4", n, k, num_experts, 32, 1, "ue8m0", True, np.concatenate(codes),
                     np.concatenate(scales))
    x = make_activations(rng, tokens, k, "bf16")
    r = make_routing(rng, tokens, num_experts, topk)
    return qw, x, r


def moe_experts(seed: int, wtype: str, num_experts: int = 128, n: int = 1536, k: int = 2048) -> QuantWeight:
    """MoE expert weights W~N(0,0.02) [E, N, K] quantised to NVFP4, MXINT4 or
    MXFP4 (drawn and quantised eight experts at a time to bound memory)."""
    quant = {"nvfp4": quantize_nvfp4, "mxint4": quantize_mxint4, "mxfp4": quantize_mxfp4}[wtype]
    rng = np.random.default_rng(seed)
    parts = []
    for e0 in range(0, num_experts, 8):
        ne = min(8, num_experts - e0)
        parts.append(quant(rng.standard_normal((ne, n, k), dtype=np.float32) * np.float32(0.02)))
    q0 = parts[0]
    ts = None if q0.tensor_scale is None else np.concatenate([q.tensor_scale for q in parts])
    return QuantWeight(wtype, n, k, num_experts, q0.group_k, q0.group_n, q0.stype, q0.signed,
                       np.concatenate([q.codes for q in parts]), np.concatenate([q.scales for q in parts]),
                       None, ts)


def random_codes_weight(seed: int, wtype: str, n: int, k: int, num_experts: int = 1,
                        group_k: int = 128, signed: bool = True, has_zeros: bool = False,
                        stype: Optional[str] = None) -> QuantWeight:
    """Uniformly random codes and scales (every code value is drawn).

    Used by round-trip and edge-case tests where the weight distribution does
    not matter but every bit pattern should appear.
    """
    rng = np.random.default_rng(seed)
    e = num_experts
    if wtype in ("int4", "int6"):
        bits = 4 if wtype == "int4" else 6
        g = k if group_k == 0 else group_k
        ng = k // g
        u = rng.integers(0, 2 ** bits, size=(e, n, k))
        stype = stype or "bf16"
        to_bits = to_bf16_bits if stype == "bf16" else to_fp16_bits
        s = to_bits(np.exp2(rng.uniform(-9, -5, size=(e, n, ng))) * rng.choice([-1, 1], size=(e, n, ng)))
        zeros = None
        if has_zeros:
            z = rng.integers(0, 2 ** bits, size=(e, n, ng))
            zeros = _pack_codes(wtype, _pad_groups_for_pack(z, bits))
        return QuantWeight(wtype, n, k, e, group_k, 1, stype, signed and not has_zeros,
                           _pack_codes(wtype, u), s, zeros)
    if wtype == "mxfp4":
        u = rng.integers(0, 16, size=(e, n, k))
        sc = rng.integers(118, 124, size=(e, n, k // 32)).astype(np.uint8)
        return QuantWeight("mxfp4", n, k, e, 32, 1, "ue8m0", True, pack_nibbles(u), sc)
    if wtype == "mxint4":
        u = rng.integers(0, 16, size=(e, n, k))
        sc = rng.integers(118, 124, size=(e, n, k // 32)).astype(np.uint8)
        return QuantWeight("mxint4", n, k, e, 32, 1, "ue8m0", True, pack_nibbles(u), sc)
    if wtype == "nvfp4":
        u = rng.integers(0, 16, size=(e, n, k))
        # positive e4m3 scales with exponent fields 4..9 (2^-3 .. 2^2), every mantissa
        sc = ((rng.integers(4, 10, size=(e, n, k // 16)) << 3) | rng.integers(0, 8, size=(e, n, k // 16)))
        ts = np.exp2(rng.uniform(-8, -4, size=e)).astype(np.float32)
        return QuantWeight("nvfp4", n, k, e, 16, 1, "e4m3", True, pack_nibbles(u), sc.astype(np.uint8),
                           tensor_scale=ts)
    if wtype == "fp8":
        b = rng.integers(0, 256, size=(e, n, k)).astype(np.uint8)
        b[(b & 0x7F) == 0x7F] = 0x00        # no NaN codes
        nb, kb = -(-n // 128), -(-k // 128)
        s = np.exp2(rng.uniform(-12, -6, size=(e, nb, kb))).astype(np.float32)
        return QuantWeight("fp8", n, k, e, 128, 128, "fp32", True, b, s)
    raise ValueError(wtype)


def e2m1_grid() -> np.ndarray:
    """Non-negative e2m1 magnitudes used by the encoder (codes 0..7)."""
    return _E2M1_GRID.copy()


def ceil_div(a: int, b: int) -> int:
    return -(-a // b)


def flops(m: int, n: int, k: int) -> int:
    return 2 * m * n * k


def log2_int(x: int) -> int:
    return int(math.log2(x))
