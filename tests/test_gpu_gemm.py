"""Dense quantized GEMM: CUDA path vs the CPU oracle, element by element (GPU).

Small cases span several 128x128 tiles with ragged M, N and K tails and run
with and without split-K; the full-size cases are the benchmark shapes, in the
launch configuration the benchmark times, checked on sampled rows.
"""
import numpy as np
import pytest

import oracle
import synth
from tolerance import check

pytestmark = pytest.mark.gpu


def _ref(qw, acts, rows=None):
    w = oracle.dequantize(qw.wtype, qw.n, qw.k, qw.codes, qw.scales, qw.zeros, qw.group_k, qw.signed, qw.stype,
                          qw.num_experts, qw.tensor_scale)
    a = oracle.decode_activations(acts.atype, acts.data, acts.scales)
    if rows is not None:
        a = a[rows]
    return oracle.gemm_dense(a, w)


def _gpu(qw, acts, **kw):
    from gpu_helpers import DevWeight, run_gemm
    return run_gemm(DevWeight(qw), acts, **kw)


# ------------------------------------------------------------------ small, element-wise
SMALL = [
    # name, generator, m, n, k
    ("w4a16_sym_g128", synth.dense_w4a16_sym, 16, 384, 1024),
    ("w4a16_sym_g128_m1", synth.dense_w4a16_sym, 1, 256, 512),
    ("w4a16_sym_g128_ragged", synth.dense_w4a16_sym, 37, 448, 640),
    ("w4a16_asym_g128", synth.dense_w4a16_asym, 16, 512, 1024),
    ("w4a16_asym_g128_m100", synth.dense_w4a16_asym, 100, 384, 768),
    ("w4a16_asym_g128_m300", synth.dense_w4a16_asym, 300, 256, 512),
    ("int6_channel_fp16", synth.dense_int6_channel, 128, 384, 1024),
    ("int6_channel_fp16_ragged", synth.dense_int6_channel, 45, 200, 520),
    ("fp8_block", synth.dense_fp8_block, 64, 512, 1024),
    ("fp8_block_ragged", synth.dense_fp8_block, 130, 300, 700),
]


@pytest.mark.parametrize("idx", range(len(SMALL)), ids=lambda i: SMALL[i][0])
@pytest.mark.parametrize("flags", [0, 1], ids=["splitk", "batch_invariant"])
def test_small_parity(idx, flags):
    name, gen, m, n, k = SMALL[idx]
    qw, acts = gen(idx, m, n, k)
    check(_gpu(qw, acts, flags=flags), _ref(qw, acts), name)


GROUPS = [
    # wtype, group_k, zeros, stype/atype, m, n, k
    ("int4", 32, True, "bf16", 20, 256, 384),
    ("int4", 64, False, "fp16", 33, 256, 448),
    ("int4", 256, True, "bf16", 17, 128, 1024),
    ("int4", 0, True, "bf16", 9, 200, 300),
    ("int4", 0, False, "fp16", 64, 256, 512),
    ("int6", 128, True, "bf16", 50, 256, 512),
    ("int6", 32, False, "fp16", 16, 128, 256),
    ("int6", 0, True, "bf16", 24, 160, 256),
]


@pytest.mark.parametrize("idx", range(len(GROUPS)), ids=lambda i: "-".join(map(str, GROUPS[i])))
def test_group_variants(idx):
    wtype, g, zeros, st, m, n, k = GROUPS[idx]
    rng = np.random.default_rng(50 + idx)
    w = rng.standard_normal((1, n, k)) * 0.02
    qw = synth.quantize_int_groupwise(w, 4 if wtype == "int4" else 6, g, not zeros, st)
    acts = synth.make_activations(rng, m, k, st)
    check(_gpu(qw, acts), _ref(qw, acts), f"{wtype} g{g} zeros={zeros} {st}")


def test_mxfp4_dense():
    qw, acts, _ = synth.moe_mxfp4(1, 24, num_experts=1, n=384, k=512)
    check(_gpu(qw, acts), _ref(qw, acts), "mxfp4 dense")


def test_mxfp4_extreme_exponents():
    """Scales at both ends of UE8M0 (subnormal bf16 results, E > 128 two-step path)."""
    qw = synth.random_codes_weight(8, "mxfp4", 128, 256)
    qw.scales[:] = np.where(np.arange(8)[None, None, :] % 2 == 0, 0, 140).astype(np.uint8)[:, :, :8]
    acts = synth.make_activations(np.random.default_rng(8), 16, 256, "bf16")
    y = _gpu(qw, acts)
    r = _ref(qw, acts)
    check(y, r, "mxfp4 extreme exponents")


N3 = [
    # wtype, m, n, k: every tile-width class, ragged M, N and K (K = 4 tiles + one group)
    ("nvfp4", 16, 384, 1024),
    ("nvfp4", 37, 200, 528),
    ("nvfp4", 100, 256, 512),
    ("nvfp4", 300, 256, 256),
    ("mxint4", 16, 384, 1024),
    ("mxint4", 45, 200, 544),
    ("mxint4", 200, 256, 512),
]


@pytest.mark.parametrize("idx", range(len(N3)), ids=lambda i: "-".join(map(str, N3[i])))
def test_nvfp4_mxint4_dense(idx):
    wtype, m, n, k = N3[idx]
    rng = np.random.default_rng(60 + idx)
    w = rng.standard_normal((1, n, k)) * 0.02
    qw = synth.quantize_nvfp4(w) if wtype == "nvfp4" else synth.quantize_mxint4(w)
    acts = synth.make_activations(rng, m, k, "bf16")
    check(_gpu(qw, acts), _ref(qw, acts), f"{wtype} {m}x{n}x{k}")


def test_mxint4_extreme_exponents():
    """UE8M0 exponents at the low end (q * 2^-122) and above 247 (the two-step
    power), against small activations so the sums stay finite."""
    qw = synth.random_codes_weight(9, "mxint4", 128, 256)
    qw.scales[:] = np.where(np.arange(8)[None, None, :] % 2 == 0, 5, 248).astype(np.uint8)[:, :, :8]
    acts = synth.make_activations(np.random.default_rng(9), 16, 256, "bf16", std=2.0 ** -20)
    check(_gpu(qw, acts), _ref(qw, acts), "mxint4 extreme exponents")


def test_strided_x_and_y():
    qw, acts = synth.dense_w4a16_asym(7, 24, 256, 512)
    check(_gpu(qw, acts, ldx=520, ldy=264), _ref(qw, acts), "strided")


def test_y_pitch_not_16_byte_multiple():
    """A Y row pitch that tensor stores cannot take (516 bytes) falls back to plain stores."""
    qw, acts = synth.dense_w4a16_asym(9, 24, 256, 512)
    check(_gpu(qw, acts, ldy=258), _ref(qw, acts), "ldy 258")
    qw, acts = synth.dense_w4a16_asym(10, 16, 8192, 640)  # cluster split with plain stores
    check(_gpu(qw, acts, ldy=8194), _ref(qw, acts), "ldy 8194, cluster")


def test_m_zero_is_noop():
    import torch
    import quantized_gemm_tma_gb300 as hq
    from gpu_helpers import DevWeight, workspace
    qw, acts = synth.dense_w4a16_sym(0, 1, 128, 128)
    dw = DevWeight(qw)
    ws = workspace(256)
    hq.hq_gemm(dw.desc, dw.wt, 0, "bf16", 0, 128, None, 0, 128, ws, 256, 0, None)
    torch.cuda.synchronize()


def test_split_k_deterministic():
    """Two runs with split-K give identical bits (fixed-order reduction)."""
    qw, acts = synth.dense_w4a16_asym(3, 16, 512, 4096)
    a = _gpu(qw, acts)
    b = _gpu(qw, acts)
    assert np.array_equal(a, b)


CLUSTER = [
    # name, generator, m, n, k: 57..76 output tiles of 128 rows, so each tile
    # runs on a 2-CTA cluster that splits K in halves (odd K-block counts give
    # rank 1 the extra block)
    ("w4a16_cls0_m16", synth.dense_w4a16_asym, 16, 8192, 640),
    ("w4a16_cls1_m40", synth.dense_w4a16_asym, 40, 8192, 512),
    ("w4a16_cls4_m100_ragged", synth.dense_w4a16_asym, 100, 8000, 384),
    ("int6_cls4_fp16", synth.dense_int6_channel, 128, 7680, 256),
    ("w4a16_cls3_m200", synth.dense_w4a16_sym, 200, 8192, 256),
]


@pytest.mark.parametrize("idx", range(len(CLUSTER)), ids=lambda i: CLUSTER[i][0])
def test_cluster_split(idx):
    import quantized_gemm_tma_gb300 as hq
    name, gen, m, n, k = CLUSTER[idx]
    qw, acts = gen(40 + idx, m, n, k)
    y = _gpu(qw, acts)
    assert hq.hq_last_plan()["splits"] == 2, hq.hq_last_plan()
    check(y, _ref(qw, acts), name)


@pytest.mark.parametrize("n,cls", [(12800, 4), (20480, 2)], ids=["one_tile_per_cta", "many_tiles_per_cta"])
def test_128_token_classes(n, cls):
    """Tiles of 65..128 tokens, whole tiles: the stream class with one
    accumulator (4) when every CTA runs one tile (100 tiles), the one-K-block
    class with two accumulators (2) when CTAs run several (160 tiles on 152
    SMs; the 2-CTA cluster split of class 4 is in test_cluster_split)."""
    import quantized_gemm_tma_gb300 as hq
    qw, acts = synth.dense_w4a16_asym(46, 100, n, 512)
    y = _gpu(qw, acts)
    assert hq.hq_last_plan()["tile_class"] == cls, hq.hq_last_plan()
    check(y, _ref(qw, acts), f"128-token class {cls}")


def test_128_token_streams_under_stream_k():
    """Tiles of 128 tokens with one K-block per stage (four dequantiser
    streams, each on every fourth stage) under stream-K, whose CTAs take K
    ranges of any length and several units each."""
    import quantized_gemm_tma_gb300 as hq
    from gpu_helpers import tuning
    qw, acts = synth.dense_w4a16_asym(47, 100, 20480, 1536)
    with tuning(HQ_FORCE_SPLITK=1):
        y = _gpu(qw, acts)
        p = hq.hq_last_plan()
    assert (p["tile_class"], p["splits"]) == (2, 0), p
    check(y, _ref(qw, acts), "128-token streams, stream-K")


def test_workspace_reused_across_shapes():
    """One workspace serves split-K problems of different shapes in turn: the
    fp32 partials of one shape never land on the counters of the next."""
    import quantized_gemm_tma_gb300 as hq
    from gpu_helpers import DevWeight, run_gemm, workspace
    probs = [synth.dense_int6_channel(13, 8, 640, 2048), synth.dense_w4a16_asym(14, 300, 768, 1536),
             synth.dense_w4a16_asym(11, 16, 1024, 4096), synth.dense_int6_channel(13, 8, 640, 2048)]
    dws = [DevWeight(qw) for qw, _ in probs]
    need = max(hq.hq_gemm_workspace_size(dw.desc, a.m, a.atype) for dw, (_, a) in zip(dws, probs))
    ws = workspace(need)
    for i, (dw, (qw, acts)) in enumerate(zip(dws, probs)):
        check(run_gemm(dw, acts, ws=ws), _ref(qw, acts), f"shared workspace, problem {i}")


# ------------------------------------------------------------------ full size, sampled rows
FULL = [
    ("c1_w4a16_sym_16x1024x1024", synth.dense_w4a16_sym, 16, 1024, 1024),
    ("c1_w4a16_sym_1x1024x1024", synth.dense_w4a16_sym, 1, 1024, 1024),
    ("c2_w4a16_asym_m1", synth.dense_w4a16_asym, 1, 8192, 8192),
    ("c2_w4a16_asym_m16", synth.dense_w4a16_asym, 16, 8192, 8192),
    ("c2_w4a16_asym_m128", synth.dense_w4a16_asym, 128, 8192, 8192),
    ("c2_w4a16_asym_m1024", synth.dense_w4a16_asym, 1024, 8192, 8192),
    ("c2_w4a16_asym_m4096", synth.dense_w4a16_asym, 4096, 8192, 8192),
    ("c3_int6_channel_128x8192x8192", synth.dense_int6_channel, 128, 8192, 8192),
    ("c4_fp8_block_m64", synth.dense_fp8_block, 64, 4096, 7168),
    ("c4_fp8_block_m512", synth.dense_fp8_block, 512, 4096, 7168),
    ("c4_fp8_block_m4096", synth.dense_fp8_block, 4096, 4096, 7168),
]


@pytest.mark.slow
@pytest.mark.parametrize("idx", range(len(FULL)), ids=lambda i: FULL[i][0])
def test_full_size_sampled(idx):
    name, gen, m, n, k = FULL[idx]
    qw, acts = gen(0, m, n, k)
    y = _gpu(qw, acts)
    rng = np.random.default_rng(idx)
    rows = np.unique(np.concatenate([[0, m - 1], rng.integers(0, m, size=min(m, 24))]))
    check(y[rows], _ref(qw, acts, rows), name)


# ------------------------------------------------------------------ full size: class 1, batch invariance
@pytest.fixture(scope="module")
def c2_full():
    """The asymmetric INT4 g128 weight at N = K = 8192 (the decode benchmark
    shape) with 1024 activation rows, its transform, and its dequantised
    values (float64) for the oracle."""
    from gpu_helpers import DevWeight
    qw, acts = synth.dense_w4a16_asym(0, 1024, 8192, 8192)
    w = oracle.dequantize(qw.wtype, qw.n, qw.k, qw.codes, qw.scales, qw.zeros, qw.group_k, qw.signed, qw.stype,
                          qw.num_experts)
    return qw, acts, DevWeight(qw), w


def _head(acts, m):
    return synth.Activations(acts.atype, m, acts.k, acts.data[:m], None if acts.scales is None else acts.scales[:m])


@pytest.mark.slow
@pytest.mark.parametrize("m", [32, 48, 64])
def test_class1_full_size_every_split(c2_full, m):
    """Tiles of 32..64 tokens (two K-blocks per stage, weight ring wrapped
    many times) at N = K = 8192 under each work split: the 2-CTA cluster split
    the planner picks, stream-K and whole tiles.  Three calls each, every one
    bit-identical; sampled rows against the oracle."""
    import quantized_gemm_tma_gb300 as hq
    from gpu_helpers import run_gemm, tuning
    qw, acts, dw, w = c2_full
    a = _head(acts, m)
    rows = np.unique(np.concatenate([[0, m - 1], np.random.default_rng(m).integers(0, m, size=12)]))
    ref = oracle.gemm_dense(oracle.decode_activations(a.atype, a.data)[rows], w)
    for switches, split in (({}, 2), ({"HQ_FORCE_SPLITK": 1}, 0), ({"HQ_FORCE_SPLITK": 2}, 1)):
        with tuning(**switches):
            outs = [run_gemm(dw, a) for _ in range(3)]
            plan = hq.hq_last_plan()
        assert (plan["bn"], plan["tile_class"], plan["splits"]) == (m, 1, split), plan
        assert plan["stages"] % 2 == 0, plan
        check(outs[0][rows], ref, f"m={m} split={split}")
        for i, y in enumerate(outs[1:], 1):
            assert np.array_equal(y, outs[0]), f"m={m} split={split}: call {i} differs from call 0"


INVARIANT_M = [1, 16, 17, 64, 128, 256, 1024]


@pytest.mark.slow
def test_batch_invariant_rows_bit_identical(c2_full):
    """HQ_FLAG_BATCH_INVARIANT: rows 0..15 of X are the same at every M, the
    other rows differ in number; rows 0..15 of Y are bit-identical at
    M = 1, 16, 17, 64, 128, 256, 1024 (N = K = 8192, asymmetric INT4 g128),
    and agree with the oracle."""
    import quantized_gemm_tma_gb300 as hq
    from gpu_helpers import run_gemm
    qw, acts, dw, w = c2_full
    head = {}
    for m in INVARIANT_M:
        y = run_gemm(dw, _head(acts, m), flags=hq.HQ_FLAG_BATCH_INVARIANT)
        p = hq.hq_last_plan()
        assert (p["bn"], p["tile_class"], p["splits"]) == (64, 1, 1), (m, p)
        head[m] = y[:16]
    ref = oracle.gemm_dense(oracle.decode_activations(acts.atype, acts.data[:16]), w)
    check(head[1024], ref, "batch-invariant rows 0..15")
    for m in INVARIANT_M:
        r = min(m, 16)
        assert np.array_equal(head[m][:r], head[1024][:r]), f"M={m}: rows differ from M=1024"


@pytest.mark.slow
@pytest.mark.parametrize("kind", ["int6_channel_fp16", "int4_sym_g32", "fp8_block"])
def test_batch_invariant_other_formats(kind):
    """The same row identity for INT6 channelwise (fp16), symmetric INT4 with
    32-wide groups, and FP8 with block scales."""
    import quantized_gemm_tma_gb300 as hq
    from gpu_helpers import DevWeight, run_gemm
    if kind == "int6_channel_fp16":
        qw, acts = synth.dense_int6_channel(60, 1024, 2048, 2048)
        ms = INVARIANT_M
    elif kind == "int4_sym_g32":
        qw, acts = synth.dense_w4a16_sym(61, 1024, 1536, 2048, group_k=32)
        ms = INVARIANT_M
    else:
        qw, acts = synth.dense_fp8_block(62, 1024, 2048, 3072)
        ms = [1, 64, 130, 512, 1024]
    dw = DevWeight(qw)
    head = {m: run_gemm(dw, _head(acts, m), flags=hq.HQ_FLAG_BATCH_INVARIANT)[:16] for m in ms}
    check(head[ms[-1]], _ref(qw, _head(acts, 16)), f"{kind} batch-invariant rows")
    for m in ms:
        r = min(m, 16)
        assert np.array_equal(head[m][:r], head[ms[-1]][:r]), f"{kind} M={m}: rows differ"
