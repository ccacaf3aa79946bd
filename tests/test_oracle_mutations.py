"""Plant plausible mistakes in the CPU oracle and check that a pin catches each.

Every mutation below is a bug someone could plausibly write into the oracle
(a swapped nibble order, a dropped zero point, a transposed operand, an
off-by-one exponent bias, an unstable scatter, ...).  The test patches it into
the oracle on the CPU, runs all pins, and requires at least one to fail.
"""
import numpy as np
import pytest

import oracle
import oracle_pins as P
from oracle import formats as F
from oracle import gemm as G
from oracle import moe as MOE
from oracle import w4a8 as W


def _swap_nibbles(packed, count):
    p = np.asarray(packed, dtype=np.uint8).astype(np.int64)
    out = np.empty(p.shape[:-1] + (2 * p.shape[-1],), dtype=np.int64)
    out[..., 0::2] = (p >> 4) & 0xF
    out[..., 1::2] = p & 0xF
    return out[..., :count]


def _int6_big_endian(packed, count):
    p = np.asarray(packed, dtype=np.uint8).astype(np.int64)
    trip = p.reshape(p.shape[:-1] + (p.shape[-1] // 3, 3))
    word = (trip[..., 0] << 16) | (trip[..., 1] << 8) | trip[..., 2]
    out = np.stack([(word >> (18 - 6 * j)) & 0x3F for j in range(4)], axis=-1)
    return out.reshape(p.shape[:-1] + (-1,))[..., :count]


def _e2m1_bias0(code):
    c = np.asarray(code, dtype=np.int64) & 0xF
    e, m = (c >> 1) & 3, c & 1
    mag = np.where(e == 0, m * 0.5, np.exp2(e) * (1.0 + m / 2.0))
    return np.where((c >> 3) & 1, -mag, mag)


def _e4m3_bias8(b):
    b = np.asarray(b, dtype=np.int64) & 0xFF
    e, m = (b >> 3) & 15, b & 7
    mag = np.where(e == 0, (m / 8.0) * 2.0 ** -7, np.exp2(e - 8.0) * (1.0 + m / 8.0))
    mag = np.where((e == 15) & (m == 7), np.nan, mag)
    return np.where((b >> 7) & 1, -mag, mag)


def _ue8m0_bias128(e):
    e = np.asarray(e, dtype=np.int64)
    return np.where(e == 255, np.nan, np.exp2(e - 128.0))


def _twos_as_unsigned(u, bits):
    return np.asarray(u, dtype=np.int64)


def _group_modulo(k, group_k):
    if group_k == 0:
        return np.zeros(k, dtype=np.int64)
    return np.arange(k) % (k // group_k)


_orig_dequant = G.dequantize


def _zero_after_scale(wtype, n, k, codes, scales, zeros=None, group_k=128, signed=True, stype="bf16",
                      num_experts=1, tensor_scale=None):
    # w = q*s - z instead of (q - z)*s
    if zeros is None or wtype not in ("int4", "int6"):
        return _orig_dequant(wtype, n, k, codes, scales, zeros, group_k, signed, stype, num_experts, tensor_scale)
    w_nz = _orig_dequant(wtype, n, k, codes, scales, None, group_k, False, stype, num_experts)
    bits = 4 if wtype == "int4" else 6
    unpack = F.unpack_nibbles if bits == 4 else F.unpack_int6
    g = 1 if group_k == 0 else k // group_k
    z = unpack(np.asarray(zeros).reshape(num_experts, n, -1), g)[:, :, G._group_index(k, group_k)]
    return w_nz - z


def _nvfp4_variant(group, use_g):
    def dq(wtype, n, k, codes, scales, zeros=None, group_k=128, signed=True, stype="bf16", num_experts=1,
           tensor_scale=None):
        if wtype != "nvfp4":
            return _orig_dequant(wtype, n, k, codes, scales, zeros, group_k, signed, stype, num_experts, tensor_scale)
        e = num_experts
        u = F.unpack_nibbles(np.asarray(codes).reshape(e, n, -1), k)
        sc = F.e4m3_to_f64(np.asarray(scales).reshape(e, n, k // 16))[:, :, np.arange(k) // group]
        g = np.asarray(tensor_scale, np.float32).astype(np.float64).reshape(e, 1, 1) if use_g else 1.0
        return F.e2m1_to_f64(u) * sc * g
    return dq


def _mxint4_unsigned(wtype, n, k, codes, scales, zeros=None, group_k=128, signed=True, stype="bf16",
                     num_experts=1, tensor_scale=None):
    if wtype != "mxint4":
        return _orig_dequant(wtype, n, k, codes, scales, zeros, group_k, signed, stype, num_experts, tensor_scale)
    u = F.unpack_nibbles(np.asarray(codes).reshape(num_experts, n, -1), k)     # codes left unsigned
    sc = F.ue8m0_to_f64(np.asarray(scales).reshape(num_experts, n, k // 32))[:, :, np.arange(k) // 32]
    return u * sc


def _gemm_transposed_weight(a, w):
    w = np.asarray(w, dtype=np.float64)
    w = w[0] if w.ndim == 3 else w
    return np.asarray(a, dtype=np.float64) @ w.reshape(w.shape[1], w.shape[0])


def _fp8_scale_transposed(atype, data, scales=None):
    if atype != "fp8":
        return _orig_decode(atype, data, scales)
    a = F.e4m3_to_f64(data)
    s = np.asarray(scales, dtype=np.float32).astype(np.float64)
    return a * s[:, :1]          # always the first K block's scale


_orig_decode = G.decode_activations


def _route_unstable(topk_ids, num_experts):
    counts, offsets, perm = _orig_route(topk_ids, num_experts)
    perm = perm.copy()
    for e in range(num_experts):                  # reverse each expert's segment
        perm[offsets[e]:offsets[e + 1]] = perm[offsets[e]:offsets[e + 1]][::-1]
    return counts, offsets, perm


_orig_route = MOE.moe_route
_orig_moe_gemm = MOE.moe_gemm


def _moe_unweighted(a, topk_ids, topk_w, w):
    return _orig_moe_gemm(a, topk_ids, np.ones_like(np.asarray(topk_w, dtype=np.float32)), w)


_orig_ranges = MOE.moe_grouped_ranges


def _ranges_masked_off_by_one(form, expert_rows, num_experts, rows):
    r = _orig_ranges(form, expert_rows, num_experts, rows)
    return [(lo, hi + 1) if form == "masked" and hi > lo else (lo, hi) for lo, hi in r]


_orig_silu = MOE.silu


def _silu_flipped(g):
    g = np.asarray(g, dtype=np.float64)
    return g / (1.0 + np.exp(g))                   # g * sigmoid(-g)


_orig_ffn = MOE.moe_ffn


def _ffn_gate_up_swapped(a, topk_ids, topk_w, w13, w2, **kw):
    get13 = w13 if callable(w13) else (lambda e, _w=np.asarray(w13, dtype=np.float64): _w[e])

    def swapped(e):
        w = np.asarray(get13(e), dtype=np.float64)
        i = w.shape[0] // 2
        return np.concatenate([w[i:], w[:i]], axis=0)
    return _orig_ffn(a, topk_ids, topk_w, swapped, w2, **kw)


def _bf16_truncate(x):
    x = np.asarray(x, dtype=np.float64)
    m, e = np.frexp(x)
    return np.ldexp(np.trunc(m * 256.0) / 256.0, e)   # toward zero instead of to nearest


def _bf16_ties_away(x):
    x = np.asarray(x, dtype=np.float64)
    m, e = np.frexp(x)
    return np.ldexp(np.sign(m) * np.floor(np.abs(m) * 256.0 + 0.5) / 256.0, e)   # halfway cases away from zero


def _ffn_unrounded(a, topk_ids, topk_w, w13, w2, **kw):
    kw["intermediate"] = None                          # H and A kept exact between the GEMMs
    return _orig_ffn(a, topk_ids, topk_w, w13, w2, **kw)


_orig_shared_exp = W.mx_shared_exponent


def _shared_exp_emax_7(amax, emax):
    return _orig_shared_exp(amax, emax - 1)             # e4m3's largest exponent taken as 7


def _e4m3_variant(rounding, saturate):
    def enc(v):
        v = np.asarray(v, dtype=np.float64)
        a = np.minimum(np.abs(v), 448.0) if saturate else np.abs(v)
        _, ex = np.frexp(a)
        e = np.maximum(np.where(a > 0, ex - 1, -6), -6)
        q = np.ldexp(1.0, (e - 3).astype(np.int32))
        r = rounding(a / q) * q
        _, rex = np.frexp(r)
        re = rex - 1
        normal = r >= 2.0 ** -6
        code = np.where(normal, ((re + 7) << 3) | np.rint((np.ldexp(r, (-re).astype(np.int32)) - 1) * 8).astype(np.int64),
                        np.rint(r / 2.0 ** -9).astype(np.int64))
        return ((np.signbit(v).astype(np.int64) << 7) | (code & 0x7F)).astype(np.uint8)
    return enc


MUTATIONS = {
    "nibble_order_swapped": [(F, "unpack_nibbles", _swap_nibbles)],
    "int6_big_endian": [(F, "unpack_int6", _int6_big_endian)],
    "e2m1_bias_0": [(F, "e2m1_to_f64", _e2m1_bias0)],
    "e4m3_bias_8": [(F, "e4m3_to_f64", _e4m3_bias8)],
    "ue8m0_bias_128": [(F, "ue8m0_to_f64", _ue8m0_bias128)],
    "signed_codes_read_unsigned": [(F, "twos_complement", _twos_as_unsigned)],
    "group_index_modulo": [(G, "_group_index", _group_modulo)],
    "zero_point_after_scale": [(G, "dequantize", _zero_after_scale), (oracle, "dequantize", _zero_after_scale)],
    "weight_transposed": [(G, "gemm_dense", _gemm_transposed_weight), (oracle, "gemm_dense", _gemm_transposed_weight)],
    "fp8_act_scale_first_block": [(G, "decode_activations", _fp8_scale_transposed),
                                  (oracle, "decode_activations", _fp8_scale_transposed)],
    "moe_perm_unstable": [(MOE, "moe_route", _route_unstable), (oracle, "moe_route", _route_unstable)],
    "moe_combine_unweighted": [(MOE, "moe_gemm", _moe_unweighted), (oracle, "moe_gemm", _moe_unweighted)],
    "moe_masked_count_off_by_one": [(MOE, "moe_grouped_ranges", _ranges_masked_off_by_one)],
    "silu_sign_flipped": [(MOE, "silu", _silu_flipped)],
    "ffn_gate_up_swapped": [(MOE, "moe_ffn", _ffn_gate_up_swapped), (oracle, "moe_ffn", _ffn_gate_up_swapped)],
    "nvfp4_scale_per_32": [(G, "dequantize", _nvfp4_variant(32, True)),
                           (oracle, "dequantize", _nvfp4_variant(32, True))],
    "nvfp4_tensor_scale_dropped": [(G, "dequantize", _nvfp4_variant(16, False)),
                                   (oracle, "dequantize", _nvfp4_variant(16, False))],
    "mxint4_codes_unsigned": [(G, "dequantize", _mxint4_unsigned), (oracle, "dequantize", _mxint4_unsigned)],
    "mx_shared_exponent_emax_7": [(W, "mx_shared_exponent", _shared_exp_emax_7)],
    "e4m3_encode_truncates": [(W, "e4m3_encode", _e4m3_variant(np.trunc, True))],
    "e4m3_encode_no_saturation": [(W, "e4m3_encode", _e4m3_variant(np.round, False))],
    "bf16_round_truncates": [(MOE, "round_bf16", _bf16_truncate)],
    "bf16_round_ties_away": [(MOE, "round_bf16", _bf16_ties_away)],
    "ffn_intermediates_unrounded": [(MOE, "moe_ffn", _ffn_unrounded), (oracle, "moe_ffn", _ffn_unrounded)],
}


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_mutation_is_caught(name, monkeypatch):
    for mod, attr, fn in MUTATIONS[name]:
        monkeypatch.setattr(mod, attr, fn)
    caught = []
    for pin in P.ALL_PINS:
        try:
            pin()
        except (AssertionError, ValueError, IndexError):
            caught.append(pin.__name__)
    assert caught, f"no pin detects the planted mistake {name!r}"
