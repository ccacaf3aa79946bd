"""W4A8-MXFP4 MoE (GPU): hq_moe_gemm with atype "mxfp8" quantises each
routed bf16 row to MXFP8 while it gathers the rows in expert order, then runs
the grouped GEMM on the block-scaled MMA.  The oracle quantises the same bf16
activations (OCP MX conversion, per token and 32 K, so before or after the
gather alike), routes, multiplies and combines in float64."""
import numpy as np
import pytest

import oracle
import synth
from tolerance import check

pytestmark = pytest.mark.gpu


def _ref(qw, acts, routing, tokens=None):
    a = oracle.decode_activations(acts.atype, acts.data)
    xq, ex = oracle.w4a8.mxfp8_quantize(a)
    a = oracle.w4a8.mxfp8_decode(xq, ex)
    ids, tw = routing.topk_ids, routing.topk_w
    if tokens is not None:
        ids, tw, a = ids[tokens], tw[tokens], a[tokens]

    def expert(e):
        return oracle.dequantize(qw.wtype, qw.n, qw.k, qw.codes[e:e + 1], qw.scales[e:e + 1], None, qw.group_k,
                                 qw.signed, qw.stype, 1)[0]
    return oracle.moe_gemm(a, ids, tw, expert)


def _run(qw, acts, routing, **kw):
    from gpu_helpers import DevWeight, run_moe
    return run_moe(DevWeight(qw), acts, routing, atype="mxfp8", **kw)


SMALL = [
    # seed, tokens, experts, n, k, topk
    (0, 37, 16, 256, 512, 4),
    (1, 1, 8, 128, 256, 2),
    (2, 200, 16, 384, 384, 8),
    (3, 64, 4, 200, 640, 3),      # ragged N
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
    check(y, _ref(qw, acts, r), f"w4a8 moe {SMALL[idx]}")


@pytest.mark.parametrize("bn", [16, 32, 64, 128, 256])
def test_every_tile_width(bn):
    """Tiles of 16 / 32 / 64 / 128 / 256 routed rows (forced), a hot expert
    with many m-tiles and empty experts."""
    from gpu_helpers import tuning
    qw, acts, r = synth.moe_mxfp4(9, 300, num_experts=8, n=256, k=512, topk=2)
    r.topk_ids[:, 0] = 3
    with tuning(HQ_FORCE_BN=bn):
        y, st = _run(qw, acts, r)
    assert st == 0
    check(y, _ref(qw, acts, r), f"w4a8 moe bn={bn}")


def test_invalid_expert_id_sets_status():
    import quantized_gemm_tma_gb300 as hq
    qw, acts, r = synth.moe_mxfp4(7, 8, num_experts=4, n=128, k=128, topk=2)
    r.topk_ids[2, 1] = 9
    y, st = _run(qw, acts, r)
    assert st == hq.HQ_ERR_INVALID_VALUE
    ok = np.nonzero(np.arange(8) != 2)[0]
    check(y[ok], _ref(qw, acts, r, ok), "w4a8 moe valid tokens")


@pytest.mark.slow
@pytest.mark.parametrize("tokens", [16, 256, 4096])
def test_full_size_sampled(tokens):
    """E = 128 MXFP4 experts of N = 1536, K = 2048, top-8 routing: sampled
    tokens against the oracle."""
    qw, acts, r = synth.moe_mxfp4(0, tokens)
    y, st = _run(qw, acts, r)
    assert st == 0
    rng = np.random.default_rng(tokens)
    rows = np.unique(np.concatenate([[0, tokens - 1], rng.integers(0, tokens, size=min(tokens, 12))]))
    check(y[rows], _ref(qw, acts, r, rows), f"w4a8 moe T={tokens}")
