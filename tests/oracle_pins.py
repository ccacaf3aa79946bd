"""Pins of the CPU oracle against values fixed outside it.

Each ``pin_*`` function raises AssertionError when the oracle disagrees with
something it cannot have produced itself: a library cast (torch's bf16, fp16
and e4m3 types), a published format table (OCP MX / OFP8, in
``tests/golden``), a hand-worked case, exact integer or rational arithmetic,
or an invariant of the definition.  ``test_oracle_pins.py`` runs them;
``test_oracle_mutations.py`` plants plausible mistakes in the oracle and
checks that some pin catches each one.
"""
from __future__ import annotations

import json
import os
from fractions import Fraction

import numpy as np
import torch

import oracle
import synth
from oracle import formats as F

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _load_table(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            rows.append(line.split())
    return rows


def _same(a, b):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    both_nan = np.isnan(a) & np.isnan(b)
    eq = (a == b) & (np.signbit(a) == np.signbit(b))
    return bool(np.all(both_nan | eq))


# ---------------------------------------------------------------------------
# element formats
# ---------------------------------------------------------------------------
def pin_bf16_exhaustive():
    u = np.arange(65536, dtype=np.uint16)
    lib = torch.from_numpy(u.view(np.int16)).view(torch.bfloat16).double().numpy()
    assert _same(F.bf16_to_f64(u), lib), "bf16 decode differs from torch.bfloat16"


def pin_fp16_exhaustive():
    u = np.arange(65536, dtype=np.uint16)
    assert _same(F.fp16_to_f64(u), u.view(np.float16).astype(np.float64)), "fp16 decode differs from numpy"


def pin_e4m3_exhaustive():
    b = np.arange(256, dtype=np.uint8)
    lib = torch.from_numpy(b).view(torch.float8_e4m3fn).double().numpy()
    assert _same(F.e4m3_to_f64(b), lib), "e4m3 decode differs from torch.float8_e4m3fn"


def pin_e4m3_spec_table():
    for hexbyte, val in _load_table("e4m3_ocp_fp8.txt"):
        got = F.e4m3_to_f64(np.array([int(hexbyte, 16)]))[0]
        assert _same(got, float(val)), f"e4m3 0x{hexbyte}: {got} != {val}"


def pin_e2m1_spec_table():
    for code, val in _load_table("e2m1_ocp_mx_v1.txt"):
        got = F.e2m1_to_f64(np.array([int(code)]))[0]
        assert _same(got, float(val)), f"e2m1 code {code}: {got} != {val}"
    # every e2m1 value lies on the e4m3 grid (torch cast round-trips exactly)
    vals = F.e2m1_to_f64(np.arange(16))
    back = torch.tensor(vals, dtype=torch.float32).to(torch.float8_e4m3fn).double().numpy()
    assert _same(back, vals)


def pin_ue8m0_spec_table():
    for e, lg in _load_table("ue8m0_ocp_mx_v1.txt"):
        got = F.ue8m0_to_f64(np.array([int(e)]))[0]
        want = float("nan") if lg == "nan" else 2.0 ** int(lg)
        assert _same(got, want), f"ue8m0 {e}: {got} != {want}"


# ---------------------------------------------------------------------------
# integer packing
# ---------------------------------------------------------------------------
def pin_int4_nibbles():
    # bytes 0x21, 0xF8 hold codes 1, 2, 8, 15 (low nibble first)
    u = F.unpack_nibbles(np.array([[0x21, 0xF8]], np.uint8), 4)
    assert u.tolist() == [[1, 2, 8, 15]]
    assert F.twos_complement(u, 4).tolist() == [[1, 2, -8, -1]]
    # odd count: the last high nibble is padding
    assert F.unpack_nibbles(np.array([[0x43, 0x05]], np.uint8), 3).tolist() == [[3, 4, 5]]


def pin_int6_stream_exhaustive():
    # every 6-bit code at each of the four phases of a 3-byte group, built as a
    # Python big integer (code k << 6k) and serialised little-endian
    for phase in range(4):
        for code in range(64):
            codes = [(7 * i + 3) % 64 for i in range(8)]
            codes[phase] = code
            codes[4 + phase] = 63 - code
            big = sum(c << (6 * i) for i, c in enumerate(codes))
            packed = np.frombuffer(big.to_bytes(6, "little"), dtype=np.uint8)[None, :]
            got = F.unpack_int6(packed, 8)[0].tolist()
            assert got == codes, (phase, code, got, codes)
    assert F.twos_complement(np.array([31, 32, 63, 0]), 6).tolist() == [31, -32, -1, 0]


# ---------------------------------------------------------------------------
# hand-worked GEMM cases
# ---------------------------------------------------------------------------
def _hand_cases():
    with open(os.path.join(GOLDEN, "hand_gemm_cases.json")) as f:
        return json.load(f)["cases"]


def _case_inputs(c):
    m, n, k = c["m"], c["n"], c["k"]
    if c["atype"] == "fp8":
        xd = np.array(c["x_bytes"], np.uint8)
        xs = np.array(c["x_scales"], np.float32)
    else:
        xb = np.zeros((m, k), np.uint16)
        xb[:, :len(c["x_bits"][0])] = np.array(c["x_bits"], np.uint16)
        xd, xs = xb, None
    codes = np.array(c["codes"], np.uint8)[None]
    if c["wtype"] == "fp8":
        scales = np.array(c["scales"], np.float32)[None]
    elif c["wtype"] in ("mxfp4", "nvfp4", "mxint4"):
        scales = np.array(c["scales"], np.uint8)[None]
    else:
        scales = np.array(c["scales_bits"], np.uint16)[None]
    zeros = np.array(c["zeros"], np.uint8)[None] if "zeros" in c else None
    return xd, xs, codes, scales, zeros


def pin_hand_gemm_cases():
    for c in _hand_cases():
        xd, xs, codes, scales, zeros = _case_inputs(c)
        ts = np.array(c["tensor_scale"], np.float32) if "tensor_scale" in c else None
        w = oracle.dequantize(c["wtype"], c["n"], c["k"], codes, scales, zeros, c["group_k"],
                              c["signed"], c["stype"], 1, ts)
        a = oracle.decode_activations(c["atype"], xd, xs)
        nz = len(c["x_values"][0])
        assert np.array_equal(a[:, :nz], np.array(c["x_values"], np.float64)), c["name"]
        y = oracle.gemm_dense(a, w)
        assert np.array_equal(y, np.array(c["y"], np.float64)), (c["name"], y.tolist(), c["y"])


def pin_hand_moe_case():
    with open(os.path.join(GOLDEN, "hand_moe_case.json")) as f:
        c = json.load(f)
    ids = np.array(c["topk_ids"], np.int32)
    counts, offsets, perm = oracle.moe_route(ids, 3)
    assert counts.tolist() == c["counts"] and offsets.tolist() == c["offsets"] and perm.tolist() == c["perm"]
    # expert weights as int4 symmetric codes, scale 1, one group per row
    wv = np.array(c["w_values"], np.int64)
    codes = synth.pack_nibbles(wv & 0xF)
    one = np.full((3, 2, 1), 0x3F80, np.uint16)
    w = oracle.dequantize("int4", 2, 2, codes, one, None, 0, True, "bf16", 3)
    assert np.array_equal(w, wv.astype(np.float64))
    y = oracle.moe_gemm(np.array(c["x_values"], np.float64), ids, np.array(c["topk_w"], np.float32), w)
    assert np.array_equal(y, np.array(c["y"], np.float64)), y.tolist()


# ---------------------------------------------------------------------------
# invariants and exact arithmetic
# ---------------------------------------------------------------------------
def pin_integer_invariant():
    """All-ones scales with zero points at the code midpoint give the exact integer matmul."""
    rng = np.random.default_rng(11)
    for wtype, bits, mid in (("int4", 4, 8), ("int6", 6, 32)):
        m, n, k, g = 3, 5, 256, 128
        u = rng.integers(0, 2 ** bits, size=(1, n, k))
        xi = rng.integers(-4, 5, size=(m, k))
        pack = synth.pack_nibbles if bits == 4 else synth.pack_int6
        zeros = pack(np.full((1, n, 4 if bits == 6 else k // g), mid))
        ones = np.full((1, n, k // g), 0x3F80, np.uint16)
        w = oracle.dequantize(wtype, n, k, pack(u), ones, zeros, g, False, "bf16", 1)
        y = oracle.gemm_dense(F.bf16_to_f64(synth.to_bf16_bits(xi.astype(np.float64))), w)
        exact = [[sum(int(xi[i, kk]) * (int(u[0, j, kk]) - mid) for kk in range(k)) for j in range(n)]
                 for i in range(m)]
        assert np.array_equal(y, np.array(exact, np.float64)), wtype


def _scalar_code(wtype, row_bytes, kk):
    """Independent per-element unpacking (bit arithmetic on one Python int)."""
    if wtype in ("int4", "mxfp4", "nvfp4", "mxint4"):
        return (int(row_bytes[kk // 2]) >> (4 * (kk % 2))) & 0xF
    stream = int.from_bytes(bytes(int(b) for b in row_bytes), "little")
    return (stream >> (6 * kk)) & 0x3F


def _frac_bf16(u):
    t = torch.from_numpy(np.array([int(u)], np.uint16).view(np.int16)).view(torch.bfloat16)
    return Fraction(float(t.double().item()))


def pin_rational_bruteforce():
    """Tiny random problems: oracle vs exact rational arithmetic in Python loops."""
    e2m1_tab = {int(c): Fraction(v) for c, v in _load_table("e2m1_ocp_mx_v1.txt")}
    e4 = lambda b: Fraction(float(torch.tensor([int(b)], dtype=torch.uint8)
                                  .view(torch.float8_e4m3fn).double().item()))
    for seed, wtype, zeros, group in ((1, "int4", False, 32), (2, "int4", True, 32), (3, "int6", True, 64),
                                      (4, "int6", False, 0), (5, "mxfp4", False, 32), (6, "nvfp4", False, 16),
                                      (7, "mxint4", False, 32)):
        m, n, k = 2, 3, 64
        qw = synth.random_codes_weight(seed, wtype, n, k, group_k=group, has_zeros=zeros)
        x = synth.make_activations(np.random.default_rng(seed), m, k, "bf16")
        y = oracle.gemm_dense(oracle.decode_activations("bf16", x.data),
                              oracle.dequantize(qw.wtype, n, k, qw.codes, qw.scales, qw.zeros, qw.group_k,
                                                qw.signed, qw.stype, 1, qw.tensor_scale))
        bits = 6 if wtype == "int6" else 4
        for i in range(m):
            for j in range(n):
                acc = Fraction(0)
                for kk in range(k):
                    c = _scalar_code(wtype, qw.codes[0, j], kk)
                    if wtype == "mxfp4":
                        wv = e2m1_tab[c] * Fraction(2) ** (int(qw.scales[0, j, kk // 32]) - 127)
                    elif wtype == "nvfp4":
                        wv = e2m1_tab[c] * e4(qw.scales[0, j, kk // 16]) * Fraction(float(qw.tensor_scale[0]))
                    elif wtype == "mxint4":
                        wv = (c - 16 if c >= 8 else c) * Fraction(2) ** (int(qw.scales[0, j, kk // 32]) - 127)
                    else:
                        gi = 0 if group == 0 else kk // group
                        s = _frac_bf16(qw.scales[0, j, gi])
                        if zeros:
                            z = _scalar_code(wtype, qw.zeros[0, j], gi)
                            wv = (c - z) * s
                        else:
                            q = c - (1 << bits) if c >= (1 << (bits - 1)) else c
                            wv = q * s
                    acc += _frac_bf16(x.data[i, kk]) * wv
                assert abs(float(acc) - y[i, j]) <= 1e-12 * (abs(float(acc)) + 1e-30), (wtype, i, j)


def pin_fp8_block_definition():
    """Block-scaled sum  sum_kb s_x s_w (e4m3 . e4m3)  with exact rationals, K spanning 3 blocks."""
    qw = synth.random_codes_weight(7, "fp8", 130, 300)
    acts = synth.make_activations(np.random.default_rng(7), 2, 300, "fp8")
    y = oracle.gemm.reference(qw, acts)
    e4 = lambda b: Fraction(float(torch.tensor([int(b)], dtype=torch.uint8)
                                  .view(torch.float8_e4m3fn).double().item()))
    for i in range(2):
        for j in (0, 129):
            tot = Fraction(0)
            for kb in range(3):
                part = sum(e4(acts.data[i, kk]) * e4(qw.codes[0, j, kk])
                           for kk in range(kb * 128, min(300, kb * 128 + 128)))
                tot += Fraction(float(acts.scales[i, kb])) * Fraction(float(qw.scales[0, j // 128, kb])) * part
            assert abs(float(tot) - y[i, j]) <= 1e-12 * abs(float(tot)) + 1e-300, (i, j)


def pin_quant_roundtrip():
    """Quantise(dequantise(q)) == q for hand-picked codes whose group range fixes the scale."""
    # int4 symmetric: each group's largest magnitude is 7, so absmax/7 recovers s
    q = np.array([[[7, -3, 0, 1, -7, 2, 5, -1]]], np.int64)
    s_bits = synth.to_bf16_bits(np.array([[[0.03125]]]))
    w = oracle.dequantize("int4", 1, 8, synth.pack_nibbles(q & 0xF), s_bits, None, 0, True, "bf16", 1)
    again = synth.quantize_int_groupwise(w, 4, 0, True, "bf16")
    assert np.array_equal(again.codes, synth.pack_nibbles(q & 0xF)) and np.array_equal(again.scales, s_bits)
    # int4 asymmetric: codes span 0..15, so (max-min)/15 recovers s and -min/s recovers z
    u = np.array([[[0, 15, 3, 9, 4, 4, 12, 1]]], np.int64)
    z = np.array([[[6]]], np.int64)
    s_bits = synth.to_bf16_bits(np.array([[[0.0078125]]]))
    w = oracle.dequantize("int4", 1, 8, synth.pack_nibbles(u), s_bits, synth.pack_nibbles(z), 0, False, "bf16", 1)
    again = synth.quantize_int_groupwise(w, 4, 0, False, "bf16")
    assert np.array_equal(again.codes, synth.pack_nibbles(u)) and np.array_equal(again.zeros, synth.pack_nibbles(z))
    # mxfp4: a block whose largest magnitude is 6 recovers its exponent
    codes = np.array([[list(range(16)) * 2]], np.int64)
    e = np.array([[[121]]], np.uint8)
    w = oracle.dequantize("mxfp4", 1, 32, synth.pack_nibbles(codes), e, None, 32, True, "ue8m0", 1)
    again = synth.quantize_mxfp4(w)
    assert np.array_equal(again.scales, e)
    assert np.array_equal(oracle.dequantize("mxfp4", 1, 32, again.codes, again.scales, None, 32, True, "ue8m0", 1), w)
    # nvfp4: every block holds a magnitude 6 and the largest block scale is
    # 448, so the tensor scale and every block scale are recovered
    codes = np.array([[list(range(16)) * 2]], np.int64)
    sb = np.array([[[0x7E, 0x38]]], np.uint8)          # 448, 1.0
    g = np.array([2.0 ** -10], np.float32)
    w = oracle.dequantize("nvfp4", 1, 32, synth.pack_nibbles(codes), sb, None, 16, True, "e4m3", 1, g)
    again = synth.quantize_nvfp4(w)
    assert np.array_equal(again.tensor_scale, g) and np.array_equal(again.scales, sb)
    assert np.array_equal(oracle.dequantize("nvfp4", 1, 32, again.codes, again.scales, None, 16, True, "e4m3", 1,
                                            again.tensor_scale), w)
    # mxint4: the block's largest magnitude is 7 (in [4, 8)), so E is recovered
    q = np.array([[[7, -3, 0, 1, -7, 2, 5, -1] * 4]], np.int64)
    e = np.array([[[121]]], np.uint8)
    w = oracle.dequantize("mxint4", 1, 32, synth.pack_nibbles(q & 0xF), e, None, 32, True, "ue8m0", 1)
    again = synth.quantize_mxint4(w)
    assert np.array_equal(again.scales, e) and np.array_equal(again.codes, synth.pack_nibbles(q & 0xF))


def pin_moe_route_properties():
    rng = np.random.default_rng(5)
    for t, e in ((1, 4), (37, 16), (300, 128)):
        ids = rng.integers(0, e, size=(t, 8)).astype(np.int32)
        ids[: t // 3] = 0                              # a hot expert
        counts, offsets, perm = oracle.moe_route(ids, e)
        flat = ids.reshape(-1)
        assert np.array_equal(counts, np.bincount(flat, minlength=e))
        assert np.array_equal(offsets, np.concatenate([[0], np.cumsum(np.bincount(flat, minlength=e))]))
        assert np.array_equal(perm, np.argsort(flat, kind="stable"))


def pin_moe_reductions():
    """topk = 1 with weight 1 reduces to a dense GEMM per expert; Y is linear in topk_w."""
    rng = np.random.default_rng(9)
    qw = synth.random_codes_weight(9, "mxfp4", 16, 64, num_experts=4)
    wd = oracle.dequantize("mxfp4", 16, 64, qw.codes, qw.scales, None, 32, True, "ue8m0", 4)
    a = rng.standard_normal((5, 64))
    ids = np.array([[0], [3], [3], [1], [0]], np.int32)
    y = oracle.moe_gemm(a, ids, np.ones((5, 1), np.float32), wd)
    for t in range(5):
        assert np.allclose(y[t], a[t] @ wd[ids[t, 0]].T, rtol=0, atol=1e-12)
    ids2 = rng.integers(0, 4, size=(5, 3)).astype(np.int32)
    w1 = (rng.integers(0, 64, size=(5, 3)) / 64.0).astype(np.float32)   # sums stay exact in fp32
    w2 = (rng.integers(0, 64, size=(5, 3)) / 64.0).astype(np.float32)
    ya = oracle.moe_gemm(a, ids2, w1, wd) + oracle.moe_gemm(a, ids2, w2, wd)
    yb = oracle.moe_gemm(a, ids2, w1.astype(np.float64) + w2.astype(np.float64), wd)
    assert np.allclose(ya, yb, rtol=1e-12, atol=1e-12)


def pin_moe_grouped_forms():
    """Grouped forms on tiny integer inputs against brute-force triple loops,
    the masked form against the contiguous form on the same rows, and rows
    outside every expert's range left out."""
    rng = np.random.default_rng(13)
    e_n, n, k, rows = 3, 4, 5, 4
    w = rng.integers(-3, 4, size=(e_n, n, k)).astype(np.float64)
    # contiguous: experts 0, 1, 2 own rows [0, 2), [2, 2), [2, 5) of 6 (row 5 unused)
    offs = np.array([0, 2, 2, 5], np.int32)
    xc = rng.integers(-4, 5, size=(6, k)).astype(np.float64)
    yc = oracle.moe_grouped_gemm(xc, "contiguous", offs, 6, w)
    assert sorted(yc) == [0, 1, 2, 3, 4]
    owner = {0: 0, 1: 0, 2: 2, 3: 2, 4: 2}
    for i, e in owner.items():
        brute = [sum(xc[i, kk] * w[e, j, kk] for kk in range(k)) for j in range(n)]
        assert np.array_equal(yc[i], np.array(brute)), (i, e)
    # masked: counts 2, 0, 3 in blocks of 4 rows hold the same rows as above
    counts = np.array([2, 0, 3], np.int32)
    xm = np.zeros((e_n * rows, k))
    xm[0:2] = xc[0:2]
    xm[8:11] = xc[2:5]
    ym = oracle.moe_grouped_gemm(xm, "masked", counts, rows, w)
    assert sorted(ym) == [0, 1, 8, 9, 10]
    for im, ic in ((0, 0), (1, 1), (8, 2), (9, 3), (10, 4)):
        assert np.array_equal(ym[im], yc[ic]), (im, ic)


def pin_silu_values():
    """silu at points where the sigmoid is a known rational: 0, ln 3 (3/4), -ln 3 (1/4)."""
    l3 = np.log(3.0)
    got = oracle.moe.silu(np.array([0.0, l3, -l3, 60.0]))
    want = np.array([0.0, 0.75 * l3, -0.25 * l3, 60.0])
    assert np.allclose(got, want, rtol=1e-15, atol=0), (got, want)


def pin_moe_ffn_reductions():
    """A gate of exactly ln 3 makes the block 0.75 ln 3 times the up projection
    through the down weights; with W2 = I it is 0.75 ln 3 times the MoE GEMM of
    the up rows (itself pinned), so the gate/up order and the down orientation
    are both checked; weights enter linearly."""
    rng = np.random.default_rng(17)
    e_n, inter, k, t, topk = 3, 4, 6, 5, 2
    a = rng.integers(-3, 4, size=(t, k)).astype(np.float64)
    a[:, 0] = 1.0                                      # a constant input column
    w_up = rng.integers(-2, 3, size=(e_n, inter, k)).astype(np.float64)
    w_gate = np.zeros((e_n, inter, k))
    w_gate[:, :, 0] = np.log(3.0)                      # gate = ln 3 for every row
    w13 = np.concatenate([w_gate, w_up], axis=1)
    ids = rng.integers(0, e_n, size=(t, topk)).astype(np.int32)
    tw = (rng.integers(1, 16, size=(t, topk)) / 16.0).astype(np.float32)
    eye = np.broadcast_to(np.eye(inter), (e_n, inter, inter))
    y = oracle.moe_ffn(a, ids, tw, w13, eye, intermediate=None)
    ref = 0.75 * np.log(3.0) * oracle.moe_gemm(a, ids, tw, w_up)
    assert np.allclose(y, ref, rtol=1e-13, atol=1e-13)
    w2 = rng.integers(-2, 3, size=(e_n, 7, inter)).astype(np.float64)   # non-square down weight
    y2 = oracle.moe_ffn(a, ids, tw, w13, w2, intermediate=None)
    for ti in range(t):
        want = sum(float(tw[ti, j]) * (0.75 * np.log(3.0) * (w_up[ids[ti, j]] @ a[ti])) @ w2[ids[ti, j]].T
                   for j in range(topk))
        assert np.allclose(y2[ti], want, rtol=1e-13, atol=1e-13), ti
    y3 = oracle.moe_ffn(a, ids, 2 * tw, w13, w2, intermediate=None)
    assert np.allclose(y3, 2 * y2, rtol=1e-14, atol=1e-14)


def pin_bf16_rounding():
    """The oracle's float64 -> bf16 rounding against torch's float32 -> bf16 cast
    on float32-exact values (halfway cases included), and the intermediate
    rounding of the feed-forward block is exactly that rounding."""
    rng = np.random.default_rng(21)
    v = rng.standard_normal(20000).astype(np.float32).astype(np.float64) * 2.0 ** rng.integers(-20, 20, 20000)
    # exact halfway points between neighbouring bf16 values: a bf16 pattern
    # (exponents 100..149, every mantissa) followed by 0x8000 in the low half
    hi = (np.arange(100, 150, dtype=np.uint32)[:, None] << 7 | np.arange(128, dtype=np.uint32)[None, :]).ravel()
    bits = hi << 16 | 0x8000
    v = np.concatenate([v, bits.view(np.float32).astype(np.float64), -bits.view(np.float32).astype(np.float64)])
    want = torch.from_numpy(v.astype(np.float32)).to(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(oracle.moe.round_bf16(v), want)
    rng = np.random.default_rng(22)
    a = rng.standard_normal((3, 8))
    w13 = rng.standard_normal((2, 4, 8))
    w2 = rng.standard_normal((2, 5, 2))
    ids = np.array([[0], [1], [1]], np.int32)
    tw = np.ones((3, 1), np.float32)
    y = oracle.moe_ffn(a, ids, tw, w13, w2)
    for t in range(3):
        h = oracle.moe.round_bf16(w13[ids[t, 0]] @ a[t])
        act = oracle.moe.round_bf16(oracle.moe.silu(h[:2]) * h[2:])
        assert np.allclose(y[t], w2[ids[t, 0]] @ act, rtol=1e-14, atol=1e-14)


# ---------------------------------------------------------------------------
# W4A8-MXFP4: MXFP8 activation quantisation and the block-scaled product
# ---------------------------------------------------------------------------
def _torch_e4m3_sat(v):
    """torch's round-to-nearest-even cast, after clamping to +-448 (torch does
    not saturate)."""
    v = np.clip(np.asarray(v, np.float64), -448.0, 448.0).astype(np.float32)
    return torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def pin_e4m3_encoder():
    """The oracle's e4m3 encoder against torch's cast: every finite value, every
    midpoint between neighbours (ties to even), random values; saturation,
    signed zero and the subnormal boundary by hand."""
    enc = oracle.w4a8.e4m3_encode
    vals = np.unique(np.abs(torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).double().numpy()))
    vals = vals[np.isfinite(vals)]                            # 0 .. 448, 127 magnitudes
    mids = (vals[1:] + vals[:-1]) / 2
    rng = np.random.default_rng(31)
    rnd = rng.uniform(-448, 448, 5000) * 2.0 ** rng.integers(-14, 1, 5000)
    for v in (vals, -vals[1:], mids, -mids, rnd):
        assert np.array_equal(enc(v), _torch_e4m3_sat(v))
    # 448 is S.1111.110; anything larger saturates to it (0x7E / 0xFE)
    assert enc(np.array([448.0, 448.5, 464.0, 480.0, 1e9, -500.0])).tolist() == [0x7E] * 5 + [0xFE]
    # -0 keeps its sign; 2^-10 is the tie between 0 and 2^-9 (even: 0); just above rounds up
    assert enc(np.array([-0.0, 2.0 ** -10, 2.0 ** -10 * 1.0001, 2.0 ** -9])).tolist() == [0x80, 0x00, 0x01, 0x01]


def pin_mx_shared_exponent():
    """floor(log2 amax) - 8 + 127 on hand-picked block maxima, clamped to [0, 254]."""
    amax = np.array([448.0, 480.0, 511.9, 512.0, 1.0, 0.75, 3.0, 0.0, 2.0 ** -140, 2.0 ** 130, 2.0 ** 200])
    want = [127, 127, 127, 128, 119, 118, 120, 0, 0, 249, 254]
    assert oracle.w4a8.mx_shared_exponent(amax, 8).tolist() == want


def pin_mxfp8_hand_block():
    """One block of 32 worked by hand.  amax = 3 gives E = 1 - 8 + 127 = 120
    (scale 2^-7), so each element is x * 128 rounded on the e4m3 grid:
      1.0        -> 128 = 1.0 * 2^7       -> exp 14, mant 0 -> 0x70
      -3.0       -> -384 = -1.5 * 2^8     -> 0x80 | 15 << 3 | 4 = 0xFC
      13/128     -> 13 = 1.625 * 2^3      -> 10 << 3 | 5 = 0x55
      12.5/128   -> 12.5, tie between 12 and 13 on the unit grid -> 12 (even)
                    = 1.5 * 2^3           -> 0x54
      2^-16      -> 2^-9, the smallest subnormal -> 0x01
      2^-17      -> 2^-10, tie between 0 and 2^-9 -> 0 -> 0x00
      the other 26 elements 0            -> 0x00"""
    x = np.zeros((1, 32))
    x[0, :6] = [1.0, -3.0, 13 / 128, 12.5 / 128, 2.0 ** -16, 2.0 ** -17]
    q, e = oracle.w4a8.mxfp8_quantize(x)
    assert e.tolist() == [[120]]
    assert q[0, :6].tolist() == [0x70, 0xFC, 0x55, 0x54, 0x01, 0x00] and not q[0, 6:].any()
    assert np.array_equal(oracle.w4a8.mxfp8_decode(q, e)[0, :4], [1.0, -3.0, 13 / 128, 12 / 128])


def _floor_log2(fr):
    """floor(log2 fr) of a positive Fraction, by exact comparison."""
    e = 0
    while Fraction(2) ** e > fr:
        e -= 1
    while Fraction(2) ** (e + 1) <= fr:
        e += 1
    return e


def pin_w4a8_rational_bruteforce():
    """Tiny W4A8-MXFP4 products against exact rationals: the block exponent
    from exact comparisons, the element rounding from torch's e4m3 cast, the
    weights from the OCP e2m1 table."""
    e2m1_tab = {int(c): Fraction(v) for c, v in _load_table("e2m1_ocp_mx_v1.txt")}
    e4 = lambda b: Fraction(float(torch.tensor([int(b)], dtype=torch.uint8)
                                  .view(torch.float8_e4m3fn).double().item()))
    for seed in (41, 42):
        m, n, k = 2, 3, 96
        qw = synth.random_codes_weight(seed, "mxfp4", n, k)
        rng = np.random.default_rng(seed)
        xv = rng.standard_normal((m, k)) * 2.0 ** rng.integers(-6, 6, (m, 1))
        xv[0, 32:64] = 0.0                                   # an all-zero block
        x = oracle.decode_activations("bf16", synth.to_bf16_bits(xv))
        w = oracle.dequantize("mxfp4", n, k, qw.codes, qw.scales, None, 32, True, "ue8m0", 1)[0]
        y = oracle.w4a8.w4a8_mxfp4_gemm(x, w)
        for i in range(m):
            xs = []
            for b in range(k // 32):
                blk = [Fraction(float(v)) for v in x[i, 32 * b:32 * b + 32]]
                amax = max(abs(v) for v in blk)
                ex = 0 if amax == 0 else min(254, max(0, _floor_log2(amax) - 8 + 127))
                sc = Fraction(2) ** (ex - 127)
                xs += [e4(_torch_e4m3_sat(np.array([float(v / sc)]))[0]) * sc for v in blk]
            for j in range(n):
                acc = sum(xs[kk] * e2m1_tab[_scalar_code("mxfp4", qw.codes[0, j], kk)]
                          * Fraction(2) ** (int(qw.scales[0, j, kk // 32]) - 127) for kk in range(k))
                assert abs(float(acc) - y[i, j]) <= 1e-12 * abs(float(acc)) + 1e-300, (seed, i, j)


ALL_PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_")]
