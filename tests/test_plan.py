"""The host-side launch planner (no GPU): tile width, work split and grid for
the benchmark shapes on a 152-SM device with 227 KB of opt-in shared memory,
through hq_plan_query."""
import pytest

SMS, OPTIN = 152, 232448

WHOLE, STREAM_K, CLUSTER = 1, 0, 2


@pytest.fixture(scope="module")
def hq():
    import quantized_gemm_tma_gb300 as m
    from quantized_gemm_tma_gb300 import _build
    _build.build()
    return m


def _int4(hq, n=8192, k=8192):
    return hq.make_desc("int4", "bf16", n, k, group_k=128, signed_codes=False, has_zeros=True)


@pytest.mark.parametrize("m,bn,cls,split,grid", [
    (1, 16, 0, CLUSTER, 128),       # 64 tiles fill 57..76 of the SMs twice over: 2-CTA K split
    (16, 16, 0, CLUSTER, 128),
    (48, 48, 1, CLUSTER, 128),
    (128, 128, 4, CLUSTER, 128),
    (1024, 256, 3, WHOLE, SMS),     # 256 wide tiles: whole tiles beat stream-K
    (4096, 256, 3, WHOLE, SMS),
])
def test_dense_int4_bench_shapes(hq, m, bn, cls, split, grid):
    p = hq.hq_plan_query(_int4(hq), m, "bf16", SMS, OPTIN)
    assert (p["bn"], p["tile_class"], p["splits"], p["grid"]) == (bn, cls, split, grid), p
    assert p["stages"] >= 2 and p["launches"] == 1


def test_dense_few_tiles_take_stream_k(hq):
    # N = 4096: 32 tiles are too few for the cluster split; the K-blocks are
    # dealt out over every SM, at least 8 per CTA
    p = hq.hq_plan_query(_int4(hq, n=4096), 16, "bf16", SMS, OPTIN)
    assert (p["splits"], p["grid"]) == (STREAM_K, SMS), p
    p = hq.hq_plan_query(_int4(hq, n=256, k=1024), 16, "bf16", SMS, OPTIN)   # 2 tiles x 8 K-blocks
    assert (p["splits"], p["grid"]) == (STREAM_K, 2), p


def test_batch_invariant_plans_one_configuration(hq):
    """With the flag every M gets the same kernel configuration: 64-token
    tiles of class 1, whole tiles (no stream-K, no cluster split); FP8 gets
    128-row weight tiles and no split-K."""
    plans = []
    for m in (1, 16, 17, 64, 128, 256, 1024, 4096):
        p = hq.hq_plan_query(_int4(hq), m, "bf16", SMS, OPTIN, hq.HQ_FLAG_BATCH_INVARIANT)
        assert (p["bn"], p["tile_class"], p["splits"]) == (64, 1, WHOLE), (m, p)
        plans.append((p["stages"], p["groups"]))
    assert len(set(plans)) == 1, plans
    f8 = hq.make_desc("fp8", "fp32", 4096, 7168, group_k=128, group_n=128)
    for m in (64, 512, 4096):
        p = hq.hq_plan_query(f8, m, "fp8", SMS, OPTIN, hq.HQ_FLAG_BATCH_INVARIANT)
        assert (p["bn"], p["splits"]) == (128, 1), (m, p)


def test_single_k_block_is_never_split(hq):
    p = hq.hq_plan_query(_int4(hq, n=1024, k=128), 16, "bf16", SMS, OPTIN)
    assert (p["splits"], p["grid"]) == (WHOLE, 8), p


def test_fp8_block_plans(hq):
    d = hq.make_desc("fp8", "fp32", 4096, 7168, group_k=128, group_n=128)
    p = hq.hq_plan_query(d, 64, "fp8", SMS, OPTIN)      # 32 tiles of 128 x 128: split K four ways
    assert (p["bn"], p["splits"], p["grid"]) == (128, 4, 128), p
    p = hq.hq_plan_query(d, 4096, "fp8", SMS, OPTIN)    # 512 tiles of 128 x 256: no split
    assert (p["bn"], p["splits"], p["grid"]) == (256, 1, SMS), p


def test_plan_tracks_sm_count_and_shared_memory(hq):
    # fewer SMs: 64 tiles no longer fit the cluster rule (2 x 64 > 100)
    p = hq.hq_plan_query(_int4(hq), 16, "bf16", 100, OPTIN)
    assert p["splits"] != CLUSTER and p["grid"] <= 100, p
    # less shared memory: fewer weight stages, still at least two
    big = hq.hq_plan_query(_int4(hq), 16, "bf16", SMS, OPTIN)
    small = hq.hq_plan_query(_int4(hq), 16, "bf16", SMS, 160 * 1024)
    assert 2 <= small["stages"] < big["stages"], (small, big)
    # 256-token tiles: three 64 KB activation stages leave room for two weight
    # stages; with less shared memory two activation stages and more weights
    wide = hq.hq_plan_query(_int4(hq), 4096, "bf16", SMS, OPTIN)
    narrow = hq.hq_plan_query(_int4(hq), 4096, "bf16", SMS, 200 * 1024)
    assert wide["tile_class"] == narrow["tile_class"] == 3 and wide["stages"] == 2 < narrow["stages"], (wide, narrow)
    assert (wide["x_stages"], narrow["x_stages"]) == (3, 2), (wide, narrow)


def test_plan_query_validation(hq):
    d = _int4(hq)
    for args, want in [((d, -1, "bf16", SMS, OPTIN), hq.HQ_ERR_INVALID_ARG),
                       ((d, 16, "bf16", 0, OPTIN), hq.HQ_ERR_INVALID_ARG),
                       ((d, 16, "bf16", SMS, 0), hq.HQ_ERR_INVALID_ARG),
                       ((d, 16, "fp16", SMS, OPTIN), hq.HQ_ERR_UNSUPPORTED),   # bf16 scales need bf16
                       ((d, 16, "fp8", SMS, OPTIN), hq.HQ_ERR_UNSUPPORTED),
                       ((hq.make_desc("mxfp4", "ue8m0", 256, 256, num_experts=4, group_k=32), 16, "bf16", SMS,
                         OPTIN), hq.HQ_ERR_INVALID_ARG)]:
        with pytest.raises(hq.HQError) as ei:
            hq.hq_plan_query(*args)
        assert ei.value.status == want, (args[1:], ei.value.status)
    assert hq.hq_plan_query(d, 0, "bf16", SMS, OPTIN)["launches"] == 0


def test_stage_override_switch(hq):
    """HQ_FORCE_XSTAGES / HQ_FORCE_WSTAGES (read once per process) set the
    activation ring and cap the weight ring for sweeps."""
    import os
    import subprocess
    import sys
    code = ("import quantized_gemm_tma_gb300 as hq; "
            "d = hq.make_desc('int4', 'bf16', 8192, 8192, group_k=128, signed_codes=False, has_zeros=True); "
            "print(hq.hq_plan_query(d, 4096, 'bf16', 152, 232448)['stages'])")
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

    def stages(**force):
        env = dict(os.environ, PYTHONPATH=root, **force)
        out = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True, timeout=120)
        assert out.returncode == 0, out.stderr
        return int(out.stdout.strip())

    # two 64 KB activation stages leave room for the whole weight ring, which
    # the second switch caps
    assert stages(HQ_FORCE_XSTAGES="2") == 8
    assert stages(HQ_FORCE_XSTAGES="2", HQ_FORCE_WSTAGES="3") == 3
    assert hq.hq_plan_query(_int4(hq), 4096, "bf16", SMS, OPTIN)["stages"] == 2


@pytest.mark.parametrize("tokens,bn,cls", [(1, 16, 0), (16, 16, 0), (17, 32, 1), (128, 32, 1), (129, 64, 1),
                                           (256, 64, 1), (1024, 64, 1), (1025, 128, 2), (4096, 128, 2)])
def test_moe_tile_width_from_mean_rows(hq, tokens, bn, cls):
    """E = 128, top-8: expert tiles of 16 tokens up to a mean of 1 routed row
    per expert, 32 up to 8, 64 up to 64, else 128."""
    d = hq.make_desc("mxfp4", "ue8m0", 1536, 2048, num_experts=128, group_k=32)
    p = hq.hq_moe_plan_query(d, tokens, 8, SMS, OPTIN)
    assert (p["bn"], p["tile_class"], p["grid"], p["launches"]) == (bn, cls, SMS, 4), p
    assert p["stages"] >= 2
    if p["tile_class"] <= 1:
        assert p["stages"] % 2 == 0, p   # two K-blocks per stage: even weight ring
    if p["tile_class"] == 2:
        assert p["stages"] % 4 == 0, p   # four dequantiser streams, each on every fourth stage


@pytest.mark.parametrize("bn", [16, 32, 48, 64])
def test_two_k_block_classes_plan_an_even_weight_ring(hq, bn):
    """Stages of two K-blocks are split between dequantiser streams by stage
    parity, so every weight-ring slot must keep one parity: the ring depth is
    even for every tile width of classes 0 and 1, dense and MoE, with and
    without zero points, for every format."""
    descs = [_int4(hq), hq.make_desc("int4", "bf16", 8192, 8192, group_k=32, signed_codes=False, has_zeros=True),
             hq.make_desc("int6", "fp16", 8192, 8192, group_k=0), hq.make_desc("mxfp4", "ue8m0", 1536, 2048,
                                                                               group_k=32)]
    for d in descs:
        for optin in (OPTIN, 200 * 1024, 160 * 1024):
            p = hq.hq_plan_query(d, bn, "fp16" if d.wtype == hq.HQ_W_INT6 else "bf16", SMS, optin)
            assert p["bn"] == bn and p["tile_class"] <= 1 and p["stages"] % 2 == 0, (bn, optin, p)


def test_moe_plan_query_validation(hq):
    d = hq.make_desc("mxfp4", "ue8m0", 1536, 2048, num_experts=128, group_k=32)
    with pytest.raises(hq.HQError) as ei:
        hq.hq_moe_plan_query(d, 16, 0, SMS, OPTIN)
    assert ei.value.status == hq.HQ_ERR_INVALID_ARG
    f8 = hq.make_desc("fp8", "fp32", 256, 256, num_experts=4, group_k=128, group_n=128)
    with pytest.raises(hq.HQError) as ei:
        hq.hq_moe_plan_query(f8, 16, 2, SMS, OPTIN)
    assert ei.value.status == hq.HQ_ERR_UNSUPPORTED
    assert hq.hq_moe_plan_query(d, 0, 8, SMS, OPTIN)["launches"] == 0


def test_w4a8_plans(hq):
    """W4A8-MXFP4 plans the same tile widths and work splits as W4A16 (256
    tokens at large M: the scale factors of a tile's tokens take 8 TMEM
    columns beside the A operand); its 128-token tiles keep the class with
    one K-block per stage even with one tile per CTA."""
    d = hq.make_desc("mxfp4", "ue8m0", 8192, 8192, group_k=32)
    for m, bn, cls, split in ((1, 16, 0, CLUSTER), (16, 16, 0, CLUSTER), (48, 48, 1, CLUSTER),
                              (128, 128, 2, CLUSTER), (1024, 256, 3, WHOLE), (4096, 256, 3, WHOLE)):
        p = hq.hq_plan_query(d, m, "mxfp8", SMS, OPTIN)
        assert (p["bn"], p["tile_class"], p["splits"]) == (bn, cls, split), (m, p)
        if cls in (0, 1, 4):
            assert p["stages"] % 2 == 0, p
        if cls == 3:   # four dequantiser streams, each on every fourth stage
            assert p["stages"] % 4 == 0, p
            # the streams wait for their stage's activations and the producer
            # refills on their A-slot release: exactly one stream period of
            # activation stages keeps both parity waits unambiguous
            assert p["x_stages"] == 4, p
    with pytest.raises(hq.HQError) as ei:
        hq.hq_plan_query(hq.make_desc("int4", "bf16", 8192, 8192, group_k=128), 16, "mxfp8", SMS, OPTIN)
    assert ei.value.status == hq.HQ_ERR_UNSUPPORTED
