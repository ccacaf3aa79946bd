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
