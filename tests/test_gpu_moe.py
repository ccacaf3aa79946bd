"""MoE grouped GEMM: routing bit-exact, outputs vs the CPU oracle (GPU)."""
import numpy as np
import pytest

import oracle
import synth
from tolerance import check, check_ffn

pytestmark = pytest.mark.gpu


def _ref(qw, acts, routing, tokens=None):
    ids, tw, a = routing.topk_ids, routing.topk_w, oracle.decode_activations(acts.atype, acts.data)
    if tokens is not None:
        ids, tw, a = ids[tokens], tw[tokens], a[tokens]

    def expert(e):
        z = None if qw.zeros is None else qw.zeros[e:e + 1]
        ts = None if qw.tensor_scale is None else qw.tensor_scale[e:e + 1]
        return oracle.dequantize(qw.wtype, qw.n, qw.k, qw.codes[e:e + 1], qw.scales[e:e + 1], z, qw.group_k,
                                 qw.signed, qw.stype, 1, ts)[0]
    return oracle.moe_gemm(a, ids, tw, expert)


def _run(qw, acts, routing, **kw):
    from gpu_helpers import DevWeight, run_moe
    return run_moe(DevWeight(qw), acts, routing, **kw)


SMALL = [
    # seed, tokens, experts, n, k, topk
    (0, 37, 16, 256, 512, 4),
    (1, 1, 8, 128, 256, 2),
    (2, 200, 16, 384, 384, 8),
    (3, 64, 4, 200, 160, 3),      # ragged N and K
    (4, 2100, 8, 128, 128, 4),    # 8400 pairs: routing on several blocks
]


@pytest.mark.parametrize("idx", range(len(SMALL)), ids=lambda i: "-".join(map(str, SMALL[i])))
def test_small_parity_and_routing(idx):
    seed, t, e, n, k, topk = SMALL[idx]
    qw, acts, r = synth.moe_mxfp4(seed, t, num_experts=e, n=n, k=k, topk=topk)
    y, st, offs, perm = _run(qw, acts, r, want_route=True)
    assert st == 0
    counts, offs_ref, perm_ref = oracle.moe_route(r.topk_ids, e)
    assert np.array_equal(offs, offs_ref)
    assert np.array_equal(perm, perm_ref)
    check(y, _ref(qw, acts, r), f"moe {SMALL[idx]}")


def test_one_expert_takes_all_and_empty_experts():
    qw, acts, r = synth.moe_mxfp4(5, 300, num_experts=8, n=256, k=256, topk=2)
    r.topk_ids[:, 0] = 3                     # expert 3 gets every token: many m-tiles
    r.topk_ids[:, 1] = np.where(np.arange(300) % 2 == 0, 3, 6)
    y, st = _run(qw, acts, r)
    assert st == 0
    check(y, _ref(qw, acts, r), "hot expert")


def test_int4_experts():
    rng = np.random.default_rng(6)
    w = rng.standard_normal((6, 256, 512)) * 0.02
    qw = synth.quantize_int_groupwise(w, 4, 128, False, "bf16")
    acts = synth.make_activations(rng, 40, 512, "bf16")
    r = synth.make_routing(rng, 40, 6, 2)
    y, st = _run(qw, acts, r)
    assert st == 0
    check(y, _ref(qw, acts, r), "int4 experts")


@pytest.mark.parametrize("wtype", ["nvfp4", "mxint4"])
def test_nvfp4_mxint4_experts(wtype):
    rng = np.random.default_rng(16)
    w = rng.standard_normal((6, 256, 512)) * 0.02 * np.exp2(rng.integers(-2, 3, size=(6, 1, 1)))
    qw = synth.quantize_nvfp4(w) if wtype == "nvfp4" else synth.quantize_mxint4(w)
    acts = synth.make_activations(rng, 40, 512, "bf16")
    r = synth.make_routing(rng, 40, 6, 2)
    y, st = _run(qw, acts, r)
    assert st == 0
    check(y, _ref(qw, acts, r), f"{wtype} experts")


def test_invalid_expert_id_sets_status():
    import quantized_gemm_tma_gb300 as hq
    qw, acts, r = synth.moe_mxfp4(7, 8, num_experts=4, n=128, k=128, topk=2)
    r.topk_ids[2, 1] = 9
    y, st = _run(qw, acts, r)
    assert st == hq.HQ_ERR_INVALID_VALUE
    ok = np.nonzero(np.arange(8) != 2)[0]
    check(y[ok], _ref(qw, acts, r, ok), "valid tokens")


FULL = [16, 256, 4096]


@pytest.mark.slow
@pytest.mark.parametrize("tokens", FULL)
def test_full_size_sampled(tokens):
    qw, acts, r = synth.moe_mxfp4(0, tokens)
    y, st, offs, perm = _run(qw, acts, r, want_route=True)
    assert st == 0
    counts, offs_ref, perm_ref = oracle.moe_route(r.topk_ids, 128)
    assert np.array_equal(offs, offs_ref)
    assert np.array_equal(perm, perm_ref)
    rng = np.random.default_rng(tokens)
    rows = np.unique(np.concatenate([[0, tokens - 1], rng.integers(0, tokens, size=min(tokens, 12))]))
    check(y[rows], _ref(qw, acts, r, rows), f"moe T={tokens}")


# ------------------------------------------------------------------ grouped forms
def _grouped(qw, form, rows, expert_rows, x_bits, expected=0, ldy=None):
    """hq_moe_grouped_gemm on device copies; returns (Y as float64 with NaN where
    nothing was written, device status)."""
    import torch
    import quantized_gemm_tma_gb300 as hq
    from gpu_helpers import DevWeight, stream, to_dev, workspace
    dw = DevWeight(qw)
    x_rows, k = x_bits.shape
    ldx = -(-k // 8) * 8
    xh = np.zeros((x_rows, ldx), np.uint16)
    xh[:, :k] = x_bits
    ldy = ldy or -(-qw.n // 8) * 8
    y = torch.full((x_rows, ldy), float("nan"), dtype=torch.bfloat16, device="cuda")
    fcode = hq.HQ_MOE_GROUPED_MASKED if form == "masked" else hq.HQ_MOE_GROUPED_CONTIGUOUS
    ws = workspace(hq.hq_moe_grouped_workspace_size(dw.desc, fcode, rows))
    er = to_dev(np.asarray(expert_rows, np.int32))
    hq.hq_moe_grouped_gemm(dw.desc, dw.wt, fcode, rows, er, expected, "bf16", to_dev(xh), ldx, y, ldy, ws,
                           ws.numel(), 0, stream())
    st = hq.hq_status_read(ws, clear=True, stream=stream())
    return y[:, :qw.n].double().cpu().numpy(), st


def _grouped_ref(qw, form, rows, expert_rows, x_bits):
    def expert(e):
        z = None if qw.zeros is None else qw.zeros[e:e + 1]
        return oracle.dequantize(qw.wtype, qw.n, qw.k, qw.codes[e:e + 1], qw.scales[e:e + 1], z, qw.group_k,
                                 qw.signed, qw.stype, 1)[0]
    return oracle.moe_grouped_gemm(oracle.decode_activations("bf16", x_bits), form, expert_rows, rows, expert)


GROUPED = [
    # form, seed, weight, experts, n, k, rows (total, or per expert when masked)
    ("masked", 20, "mxfp4", 8, 256, 512, 40),
    ("masked", 21, "int4", 4, 384, 256, 300),       # several 64-token tiles per expert
    ("contiguous", 22, "mxfp4", 8, 200, 384, 150),  # ragged N
    ("contiguous", 23, "int4", 6, 256, 512, 700),
]


@pytest.mark.parametrize("idx", range(len(GROUPED)), ids=lambda i: "-".join(map(str, GROUPED[i][:3])))
def test_grouped_forms(idx):
    form, seed, wt, e, n, k, rows = GROUPED[idx]
    rng = np.random.default_rng(seed)
    if wt == "mxfp4":
        qw = synth.random_codes_weight(seed, "mxfp4", n, k, num_experts=e, group_k=32)
    else:
        qw = synth.quantize_int_groupwise(rng.standard_normal((e, n, k)) * 0.02, 4, 128, False, "bf16")
    if form == "masked":
        counts = rng.integers(0, rows + 1, size=e)
        counts[0], counts[-1] = rows, 0               # a full block and an empty expert
        expert_rows, x_rows = counts, e * rows
    else:
        cuts = np.sort(rng.integers(0, rows - 5, size=e - 1))
        expert_rows = np.concatenate([[0], cuts, [rows - 5]])   # the last 5 rows belong to no expert
        x_rows = rows
    x_bits = synth.make_activations(rng, x_rows, k, "bf16").data
    y, st = _grouped(qw, form, rows, expert_rows, x_bits)
    assert st == 0
    ref = _grouped_ref(qw, form, rows, expert_rows, x_bits)
    valid = np.array(sorted(ref), dtype=np.int64)
    check(y[valid], np.stack([ref[i] for i in valid]), f"grouped {GROUPED[idx]}")
    untouched = np.setdiff1d(np.arange(x_rows), valid)
    assert np.isnan(y[untouched]).all(), "rows outside every expert's range were written"


def test_grouped_invalid_counts_set_status():
    import quantized_gemm_tma_gb300 as hq
    rng = np.random.default_rng(30)
    qw = synth.random_codes_weight(30, "mxfp4", 128, 256, num_experts=4, group_k=32)
    counts = np.array([16, 40, 3, 16])                 # expert 1 claims more rows than its block holds
    x_bits = synth.make_activations(rng, 4 * 32, 256, "bf16").data
    y, st = _grouped(qw, "masked", 32, counts, x_bits)
    assert st == hq.HQ_ERR_INVALID_VALUE
    ok = np.array(counts)
    ok[1] = 0
    ref = _grouped_ref(qw, "masked", 32, ok, x_bits)
    valid = np.array(sorted(ref), dtype=np.int64)
    check(y[valid], np.stack([ref[i] for i in valid]), "valid experts")
    assert np.isnan(y[32:64]).all()


# ------------------------------------------------------------------ feed-forward block
def _expert_fn(qw):
    """Expert weights [N, K] in float64, dequantised exactly (no operand rounding)."""
    def expert(e):
        z = None if qw.zeros is None else qw.zeros[e:e + 1]
        ts = None if qw.tensor_scale is None else qw.tensor_scale[e:e + 1]
        return oracle.dequantize(qw.wtype, qw.n, qw.k, qw.codes[e:e + 1], qw.scales[e:e + 1], z, qw.group_k,
                                 qw.signed, qw.stype, 1, ts)[0]
    return expert


def _cached(fn):
    cache = {}

    def get(e):
        if e not in cache:
            cache[e] = fn(e)
        return cache[e]
    return get


def _run_ffn(d13, d2, acts, r, n):
    import torch
    import quantized_gemm_tma_gb300 as hq
    from gpu_helpers import stream, to_dev, workspace
    t, k = acts.m, acts.k
    topk = r.topk_ids.shape[1]
    ldy = -(-n // 8) * 8
    y = torch.full((t, ldy), float("nan"), dtype=torch.bfloat16, device="cuda")
    ws = workspace(hq.hq_moe_ffn_workspace_size(d13.desc, d2.desc, t, topk))
    hq.hq_moe_ffn(d13.desc, d13.wt, d2.desc, d2.wt, t, topk, to_dev(np.ascontiguousarray(r.topk_ids, np.int32)),
                  to_dev(np.ascontiguousarray(r.topk_w, np.float32)), "bf16", to_dev(acts.data), k, y, ldy, ws,
                  ws.numel(), 0, stream())
    st = hq.hq_status_read(ws, clear=True, stream=stream())
    return y[:, :n].double().cpu().numpy(), st


FFN = [
    # seed, weight, tokens, experts, intermediate I, hidden K, output n, topk, fused
    (40, "mxfp4", 37, 8, 128, 256, 256, 4, True),    # 32-token tiles
    (41, "int4", 64, 6, 192, 384, 200, 2, False),    # I not a multiple of 128: H stored, elementwise kernel
    (42, "int4", 4, 8, 256, 512, 256, 2, True),      # 16-token tiles, asymmetric INT4 g128
    (43, "mxfp4", 300, 4, 256, 256, 128, 4, True),   # 128-token tiles
    (44, "int6ch", 40, 4, 128, 256, 256, 2, True),   # row scales of the gate and the up rows
    (45, "nvfp4", 64, 4, 128, 256, 256, 2, True),    # per-expert tensor scales
]


def _ffn_weight(kind, rng, e, n, k, seed):
    if kind == "mxfp4":
        return synth.moe_mxfp4(seed, 1, num_experts=e, n=n, k=k, topk=1)[0]
    w = rng.standard_normal((e, n, k)) * 0.02
    if kind == "int4":
        return synth.quantize_int_groupwise(w, 4, 128 if k % 128 == 0 else 64, False, "bf16")
    if kind == "int6ch":
        return synth.quantize_int_groupwise(w, 6, 0, True, "bf16")
    return synth.quantize_nvfp4(w)


@pytest.mark.parametrize("idx", range(len(FFN)), ids=lambda i: "-".join(map(str, FFN[i][:2])))
def test_moe_ffn_parity(idx):
    """The feed-forward block against the exact oracle (exact expert weights,
    exact intermediates) at the block tolerance of two chained GEMMs; with I a
    multiple of 128 silu(gate) * up comes from the gate+up epilogue (five
    launches), else from an elementwise kernel between the GEMMs (six)."""
    import quantized_gemm_tma_gb300 as hq
    from gpu_helpers import DevWeight
    seed, wt, t, e, inter, k, n, topk, fused = FFN[idx]
    rng = np.random.default_rng(seed)
    w13 = _ffn_weight(wt, rng, e, 2 * inter, k, seed)
    w2 = _ffn_weight(wt, rng, e, n, inter, seed + 100)
    acts = synth.make_activations(rng, t, k, "bf16")
    r = synth.make_routing(rng, t, e, topk)
    got, st = _run_ffn(DevWeight(w13), DevWeight(w2), acts, r, n)
    assert st == 0
    assert hq.hq_last_plan()["launches"] == (5 if fused else 6), hq.hq_last_plan()
    ref = oracle.moe_ffn(oracle.decode_activations("bf16", acts.data), r.topk_ids, r.topk_w, _expert_fn(w13),
                         _expert_fn(w2), intermediate=None)
    check_ffn(got, ref, f"moe ffn {FFN[idx]}")


# ------------------------------------------------------------------ full size: every tile width, the FFN
@pytest.fixture(scope="module")
def moe_full():
    """E = 128, N = 1536, K = 2048 MXFP4 gate+up experts, T = 4096 tokens of
    activations and skewed top-8 routing (the T = 256 case takes the first
    256 tokens), the transformed weight, and a caching expert dequantiser."""
    from gpu_helpers import DevWeight
    qw, acts, r = synth.moe_mxfp4(0, 4096)
    return qw, acts, r, DevWeight(qw), _cached(_expert_fn(qw))


def _first(acts, r, t):
    return (synth.Activations(acts.atype, t, acts.k, acts.data[:t]),
            synth.MoeRouting(r.topk_ids[:t], r.topk_w[:t], r.extra))


_WIDTH_REFS = {}


@pytest.mark.slow
@pytest.mark.parametrize("bn", [16, 32, 48, 64, 128])
def test_every_tile_width_full_size_repeated(moe_full, bn):
    """Full-size MoE at every expert tile width the planner can choose (the
    two-K-block stream dequantisers for 16..64 tokens, per-lane row gathers
    for 32..128), T = 256 (every token checked) and T = 4096 (64 sampled
    tokens).  Four calls each: every call bit-identical to the first (a
    race shows up as a difference), the first against the oracle."""
    import quantized_gemm_tma_gb300 as hq
    from gpu_helpers import run_moe, tuning
    qw, acts, r, dw, expert = moe_full
    for t in (256, 4096):
        a, rt = _first(acts, r, t)
        rows = np.arange(t) if t <= 256 else np.unique(np.concatenate(
            [[0, t - 1], np.random.default_rng(t).integers(0, t, size=62)]))
        if t not in _WIDTH_REFS:
            _WIDTH_REFS[t] = oracle.moe_gemm(oracle.decode_activations("bf16", a.data)[rows], rt.topk_ids[rows],
                                             rt.topk_w[rows], expert)
        outs = []
        with tuning(HQ_FORCE_BN=bn):
            for _ in range(4):
                y, st = run_moe(dw, a, rt)
                assert st == 0, st
                p = hq.hq_last_plan()
                assert p["bn"] == bn, p
                outs.append(y)
        if p["tile_class"] <= 1:
            assert p["stages"] % 2 == 0, p
        check(outs[0][rows], _WIDTH_REFS[t], f"T={t} bn={bn}")
        for i, y in enumerate(outs[1:], 1):
            assert np.array_equal(y, outs[0]), f"T={t} bn={bn}: call {i} differs from call 0"


@pytest.mark.slow
@pytest.mark.parametrize("tokens", [256, 4096])
def test_moe_ffn_full_size_sampled(moe_full, tokens):
    """The feed-forward block at the benchmark shape: the gate+up experts
    above (I = 768), MXFP4 down experts [128][2048][768], 16 sampled tokens
    against the exact oracle."""
    from gpu_helpers import DevWeight
    qw, acts, r, dw, expert = moe_full
    w2, _, _ = synth.moe_mxfp4(1, 1, num_experts=128, n=2048, k=768)
    a, rt = _first(acts, r, tokens)
    got, st = _run_ffn(dw, DevWeight(w2), a, rt, 2048)
    assert st == 0
    rows = np.unique(np.concatenate([[0, tokens - 1], np.random.default_rng(tokens + 1).integers(0, tokens, 14)]))
    ref = oracle.moe_ffn(oracle.decode_activations("bf16", a.data)[rows], rt.topk_ids[rows], rt.topk_w[rows], expert,
                         _expert_fn(w2), intermediate=None)
    check_ffn(got[rows], ref, f"moe ffn full size T={tokens}")


@pytest.mark.slow
@pytest.mark.parametrize("wtype", ["nvfp4", "mxint4"])
def test_nvfp4_mxint4_experts_full_size(moe_full, wtype):
    """The gate+up shape (E = 128, N = 1536, K = 2048) with NVFP4 or MXINT4
    experts, T = 4096 tokens of the routing above, 32 sampled tokens against
    the oracle."""
    from gpu_helpers import DevWeight, run_moe
    _, acts, r, _, _ = moe_full
    qw = synth.moe_experts(3, wtype)
    y, st = run_moe(DevWeight(qw), acts, r)
    assert st == 0
    rows = np.unique(np.concatenate([[0, 4095], np.random.default_rng(5).integers(0, 4096, size=30)]))
    check(y[rows], _ref(qw, acts, r, rows), f"{wtype} experts full size")
