"""W4A8-MXFP4 (GPU): MXFP4 weights against activations quantised to MXFP8 on
the device (hq_mxfp8_quantize), multiplied by the block-scaled tensor-core
path of hq_gemm (atype "mxfp8"), against the oracle's W4A8 product, which
quantises the same bf16 activations itself (OCP MX conversion) and sums in
float64."""
import numpy as np
import pytest

import oracle
import synth
from tolerance import check

pytestmark = pytest.mark.gpu


def _w4a8(dw, x_bits, k, flags=0):
    """Quantise bf16 rows x_bits [m][k] to MXFP8 on the device, then the
    W4A8 GEMM; returns Y [m][n] as float64."""
    import torch
    import quantized_gemm_tma_gb300 as hq
    from gpu_helpers import stream, to_dev, workspace
    m = x_bits.shape[0]
    n = dw.qw.n
    x = to_dev(np.ascontiguousarray(x_bits))
    q = torch.empty((m, k), dtype=torch.uint8, device="cuda")
    e = torch.empty((m, k // 32), dtype=torch.uint8, device="cuda")
    hq.hq_mxfp8_quantize(m, k, x, k, q, k, e, k // 32, stream())
    ldy = -(-n // 8) * 8
    y = torch.full((m, ldy), float("nan"), dtype=torch.bfloat16, device="cuda")
    ws = workspace(hq.hq_gemm_workspace_size(dw.desc, m, "mxfp8"))
    hq.hq_gemm(dw.desc, dw.wt, m, "mxfp8", q, k, e, y, ldy, ws, ws.numel(), flags, stream())
    st = hq.hq_status_read(ws, clear=True, stream=stream())
    assert st == 0, hq.status_string(st)
    return y[:, :n].double().cpu().numpy()


def _ref(qw, x_bits, rows=None):
    w = oracle.dequantize(qw.wtype, qw.n, qw.k, qw.codes, qw.scales, None, qw.group_k, qw.signed, qw.stype, 1)[0]
    x = oracle.decode_activations("bf16", x_bits if rows is None else x_bits[rows])
    return oracle.w4a8.w4a8_mxfp4_gemm(x, w)


def _weight(seed, n, k):
    rng = np.random.default_rng(seed)
    return synth.quantize_mxfp4(rng.standard_normal((1, n, k)) * 0.02)


SMALL = [
    # m, n, k: tiles of 16 (m <= 16), 32..64 (two K-blocks per stage) and 128 tokens, ragged M and N
    (1, 256, 512),
    (16, 384, 1024),
    (37, 448, 640),
    (64, 256, 512),
    (100, 384, 768),
    (300, 256, 512),
]


@pytest.mark.parametrize("idx", range(len(SMALL)), ids=lambda i: "x".join(map(str, SMALL[i])))
def test_w4a8_small(idx):
    from gpu_helpers import DevWeight
    m, n, k = SMALL[idx]
    qw = _weight(80 + idx, n, k)
    x = synth.make_activations(np.random.default_rng(90 + idx), m, k, "bf16").data
    check(_w4a8(DevWeight(qw), x, k), _ref(qw, x), f"w4a8 {m}x{n}x{k}")


def test_w4a8_extreme_exponents():
    """Activation blocks from 2^-40 to 2^40 and weight exponents at both ends
    of what keeps the products finite: the scale factors reach the MMA
    unchanged."""
    from gpu_helpers import DevWeight
    m, n, k = 24, 256, 512
    qw = synth.random_codes_weight(81, "mxfp4", n, k)
    rng = np.random.default_rng(81)
    qw.scales[:] = rng.integers(100, 150, size=qw.scales.shape).astype(np.uint8)
    x = rng.standard_normal((m, k)) * np.exp2(rng.integers(-40, 40, size=(m, k // 32))).repeat(32, axis=1)
    xb = synth.to_bf16_bits(x)
    y = _w4a8(DevWeight(qw), xb, k)
    r = _ref(qw, xb)
    # rows differ in magnitude by up to 2^80: check each row on its own scale
    for i in range(m):
        check(y[i:i + 1], r[i:i + 1], f"w4a8 extreme exponents row {i}")


@pytest.mark.parametrize("m", [16, 24, 100])
def test_w4a8_large_weight_exponents(m):
    """Weight block scales from 2^122 to 2^127 (UE8M0 249..254), mixed within
    rows with ordinary ones, against activations near 2^-100: those sub-blocks
    take the exact conversion table instead of the shifted conversion whose
    2^6 goes into the weight exponent.  m = 16 and 24 run the two-K-block
    streams, m = 100 one K-block per stage."""
    from gpu_helpers import DevWeight
    n, k = 256, 1024
    qw = synth.random_codes_weight(84 + m, "mxfp4", n, k)
    rng = np.random.default_rng(84 + m)
    sc = rng.integers(115, 135, size=qw.scales.shape)
    big = rng.random(qw.scales.shape) < 0.3
    sc[big] = rng.integers(249, 255, size=int(big.sum()))
    qw.scales[:] = sc.astype(np.uint8)
    x = rng.standard_normal((m, k)) * np.exp2(rng.integers(-110, -100, size=(m, k // 32))).repeat(32, axis=1)
    xb = synth.to_bf16_bits(x)
    y = _w4a8(DevWeight(qw), xb, k)
    r = _ref(qw, xb)
    assert np.isfinite(r).all()
    for i in range(m):
        check(y[i:i + 1], r[i:i + 1], f"w4a8 large weight exponents row {i}")


@pytest.mark.parametrize("bn", [16, 32, 48, 64, 128, 192, 256])
def test_w4a8_every_tile_width(bn):
    """Tiles of every width the planner can choose (forced), ragged M and N:
    the scale factors of up to 256 tokens beside the A operand."""
    from gpu_helpers import DevWeight, tuning
    m, n, k = 300, 384, 1024
    qw = _weight(85, n, k)
    x = synth.make_activations(np.random.default_rng(85), m, k, "bf16").data
    with tuning(HQ_FORCE_BN=bn):
        y = _w4a8(DevWeight(qw), x, k)
    check(y, _ref(qw, x), f"w4a8 bn={bn}")


@pytest.mark.parametrize("splitk", ["cluster", "stream_k", "whole"])
def test_w4a8_work_splits(splitk):
    """N = 8192 gives 64 weight tiles: the 2-CTA cluster split (the planner's
    choice at M = 16), stream-K and whole tiles."""
    import quantized_gemm_tma_gb300 as hq
    from gpu_helpers import DevWeight, tuning
    m, n, k = 16, 8192, 1024
    qw = _weight(82, n, k)
    x = synth.make_activations(np.random.default_rng(82), m, k, "bf16").data
    switches = {"cluster": {}, "stream_k": {"HQ_FORCE_SPLITK": 1}, "whole": {"HQ_FORCE_SPLITK": 2}}[splitk]
    with tuning(**switches):
        y = _w4a8(DevWeight(qw), x, k)
        p = hq.hq_last_plan()
    assert p["splits"] == {"cluster": 2, "stream_k": 0, "whole": 1}[splitk], p
    check(y, _ref(qw, x), f"w4a8 {splitk}")


@pytest.mark.parametrize("splitk", ["cluster", "stream_k", "whole"])
def test_w4a8_256_token_tiles_every_split(splitk):
    """Tiles of 256 tokens (four dequantiser streams, each on every fourth
    stage, with four activation stages) under each work split: stream-K hands
    CTAs K ranges of any length, the cluster split half of K each."""
    import quantized_gemm_tma_gb300 as hq
    from gpu_helpers import DevWeight, tuning
    m, n, k = 256, 8192, 1024
    qw = _weight(84, n, k)
    x = synth.make_activations(np.random.default_rng(84), m, k, "bf16").data
    switches = {"cluster": {}, "stream_k": {"HQ_FORCE_SPLITK": 1}, "whole": {"HQ_FORCE_SPLITK": 2}}[splitk]
    with tuning(**switches):
        y = _w4a8(DevWeight(qw), x, k)
        p = hq.hq_last_plan()
    assert (p["bn"], p["tile_class"], p["x_stages"]) == (256, 3, 4), p
    assert p["splits"] == {"cluster": 2, "stream_k": 0, "whole": 1}[splitk], p
    check(y, _ref(qw, x), f"w4a8 256-token {splitk}")


def test_w4a8_batch_invariant():
    """With HQ_FLAG_BATCH_INVARIANT rows 0..15 are bit-identical at every M."""
    import quantized_gemm_tma_gb300 as hq
    from gpu_helpers import DevWeight
    n, k = 1024, 2048
    qw = _weight(83, n, k)
    dw = DevWeight(qw)
    x = synth.make_activations(np.random.default_rng(83), 512, k, "bf16").data
    head = {m: _w4a8(dw, x[:m], k, hq.HQ_FLAG_BATCH_INVARIANT)[:16] for m in (1, 16, 17, 64, 200, 512)}
    check(head[512], _ref(qw, x[:16]), "w4a8 batch-invariant rows")
    for m, h in head.items():
        r = min(m, 16)
        assert np.array_equal(h[:r], head[512][:r]), f"M={m}: rows differ"


@pytest.mark.slow
@pytest.mark.parametrize("m", [1, 16, 128, 1024])
def test_w4a8_full_size_sampled(m):
    """N = K = 8192 MXFP4 weights (W~N(0,0.02)), X~N(0,1): the dense decode
    and prefill shapes, sampled rows against the oracle."""
    from gpu_helpers import DevWeight
    n = k = 8192
    qw = _weight(0, n, k)
    x = synth.make_activations(np.random.default_rng(1), m, k, "bf16").data
    y = _w4a8(DevWeight(qw), x, k)
    rows = np.unique(np.concatenate([[0, m - 1], np.random.default_rng(m).integers(0, m, size=min(m, 16))]))
    check(y[rows], _ref(qw, x, rows), f"w4a8 full size m={m}")
