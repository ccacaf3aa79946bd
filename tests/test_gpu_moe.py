"""MoE grouped GEMM: routing bit-exact, outputs vs the CPU oracle (GPU)."""
import numpy as np
import pytest

import oracle
import synth
from tolerance import check

pytestmark = pytest.mark.gpu


def _ref(qw, acts, routing, tokens=None):
    ids, tw, a = routing.topk_ids, routing.topk_w, oracle.decode_activations(acts.atype, acts.data)
    if tokens is not None:
        ids, tw, a = ids[tokens], tw[tokens], a[tokens]

    def expert(e):
        z = None if qw.zeros is None else qw.zeros[e:e + 1]
        return oracle.dequantize(qw.wtype, qw.n, qw.k, qw.codes[e:e + 1], qw.scales[e:e + 1], z, qw.group_k,
                                 qw.signed, qw.stype, 1)[0]
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
    """Dequantised expert weights as the MMA operand: a groupwise INT weight
    with zero points enters as (q - z) * s rounded once to bf16 (the operand
    rounding both GEMMs of the block apply); MXFP4 values are exact in bf16."""
    def expert(e):
        z = None if qw.zeros is None else qw.zeros[e:e + 1]
        w = oracle.dequantize(qw.wtype, qw.n, qw.k, qw.codes[e:e + 1], qw.scales[e:e + 1], z, qw.group_k,
                              qw.signed, qw.stype, 1)[0]
        return oracle.moe.round_bf16(w) if qw.zeros is not None else w
    return expert


FFN = [
    # seed, weight, tokens, experts, intermediate I, hidden K, output n, topk
    (40, "mxfp4", 37, 8, 128, 256, 256, 4),
    (41, "int4", 64, 6, 192, 384, 200, 2),     # ragged output n, three gate/up tiles
]


@pytest.mark.parametrize("idx", range(len(FFN)), ids=lambda i: "-".join(map(str, FFN[i][:2])))
def test_moe_ffn_parity(idx):
    import torch
    import quantized_gemm_tma_gb300 as hq
    from gpu_helpers import DevWeight, stream, to_dev, workspace
    seed, wt, t, e, inter, k, n, topk = FFN[idx]
    rng = np.random.default_rng(seed)
    if wt == "mxfp4":
        w13, acts, r = synth.moe_mxfp4(seed, t, num_experts=e, n=2 * inter, k=k, topk=topk)
        w2, _, _ = synth.moe_mxfp4(seed + 100, 1, num_experts=e, n=n, k=inter, topk=1)
    else:
        w13 = synth.quantize_int_groupwise(rng.standard_normal((e, 2 * inter, k)) * 0.02, 4, 128, False, "bf16")
        w2 = synth.quantize_int_groupwise(rng.standard_normal((e, n, inter)) * 0.02, 4, 64, False, "bf16")
        acts = synth.make_activations(rng, t, k, "bf16")
        r = synth.make_routing(rng, t, e, topk)
    d13, d2 = DevWeight(w13), DevWeight(w2)
    ldy = -(-n // 8) * 8
    y = torch.full((t, ldy), float("nan"), dtype=torch.bfloat16, device="cuda")
    ws = workspace(hq.hq_moe_ffn_workspace_size(d13.desc, d2.desc, t, topk))
    hq.hq_moe_ffn(d13.desc, d13.wt, d2.desc, d2.wt, t, topk, to_dev(np.ascontiguousarray(r.topk_ids, np.int32)),
                  to_dev(np.ascontiguousarray(r.topk_w, np.float32)), "bf16", to_dev(acts.data), k, y, ldy, ws,
                  ws.numel(), 0, stream())
    assert hq.hq_status_read(ws, clear=True, stream=stream()) == 0
    got = y[:, :n].double().cpu().numpy()
    ref = oracle.moe_ffn(oracle.decode_activations("bf16", acts.data), r.topk_ids, r.topk_w, _expert_fn(w13),
                         _expert_fn(w2))
    check(got, ref, f"moe ffn {FFN[idx]}")
