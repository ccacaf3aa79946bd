"""The C-ABI library loads, exports every symbol include/hq.h declares, and
rejects bad arguments on the host before touching a GPU (no GPU needed)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _header_functions():
    src = open(os.path.join(ROOT, "include", "hq.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(hq_[a-z0-9_]+)\s*\(", src)))


@pytest.fixture(scope="module")
def hq():
    import quantized_gemm_tma_gb300 as m
    from quantized_gemm_tma_gb300 import _build
    _build.build()
    return m


def test_exports_every_declared_symbol(hq):
    declared = _header_functions()
    assert declared, "no functions parsed from hq.h"
    assert sorted(hq.EXPORTS) == declared
    lib = ctypes.CDLL(hq.LIB_PATH)
    for name in declared:
        assert hasattr(lib, name), name


def test_version_and_strings(hq):
    assert hq.hq_version() >= 100
    for s in range(9):
        assert hq.status_string(s) and hq.status_string(s) != "unknown status"


def _desc(hq, **kw):
    base = dict(wtype="int4", stype="bf16", n=256, k=512, group_k=128)
    base.update(kw)
    return hq.make_desc(**base)


@pytest.mark.parametrize("kw,status", [
    (dict(n=0), 1), (dict(k=-5), 1), (dict(group_k=48), 1), (dict(group_k=96), 1), (dict(k=500), 1),
    (dict(wtype="int6", k=130, group_k=0), 1), (dict(stype="fp32"), 1), (dict(wtype="mxfp4", stype="bf16"), 1),
    (dict(wtype="mxfp4", stype="ue8m0", group_k=64), 1), (dict(wtype="fp8", stype="fp32", group_k=128, group_n=1), 1),
    (dict(wtype=7), 1), (dict(num_experts=0), 1),
    (dict(wtype="nvfp4", stype="ue8m0", group_k=16), 1), (dict(wtype="nvfp4", stype="e4m3", group_k=32), 1),
    (dict(wtype="nvfp4", stype="e4m3", group_k=16, k=520), 1),
    (dict(wtype="nvfp4", stype="e4m3", group_k=16, has_zeros=True), 1),
    (dict(wtype="mxint4", stype="e4m3", group_k=32), 1), (dict(wtype="mxint4", stype="ue8m0", group_k=16), 1),
])
def test_transform_size_validation(hq, kw, status):
    with pytest.raises(hq.HQError) as ei:
        hq.hq_transform_size(_desc(hq, **kw))
    assert ei.value.status == status


def test_transform_size_layouts(hq):
    # one 128x128 INT4 tile with bf16 g128 scales = 8192 + 256 bytes (+256 header)
    assert hq.hq_transform_size(_desc(hq, n=128, k=128)) == 256 + 8192 + 256
    s = hq.hq_transform_size(_desc(hq, n=8192, k=8192, has_zeros=True, signed_codes=False))
    assert s == 256 + 64 * 64 * (8192 + 256 + 128)
    # nvfp4: codes + e4m3 scales [128][8] per tile, then the float32 tensor scales (one 256-byte block)
    assert hq.hq_transform_size(hq.make_desc("nvfp4", "e4m3", 128, 128, group_k=16)) == 256 + 8192 + 1024 + 256
    assert hq.hq_transform_size(hq.make_desc("nvfp4", "e4m3", 256, 256, num_experts=3, group_k=16)) == \
        256 + 3 * 4 * (8192 + 1024) + 256
    # mxint4: codes + UE8M0 scales [128][4] per tile, like mxfp4
    assert hq.hq_transform_size(hq.make_desc("mxint4", "ue8m0", 128, 128, group_k=32)) == 256 + 8192 + 512
    # fp8: 16 KiB images + block scales
    d = hq.make_desc("fp8", "fp32", 4096, 7168, group_k=128, group_n=128)
    assert hq.hq_transform_size(d) >= 256 + 32 * 56 * 16384 + 4 * 32 * 56


def test_gemm_host_validation(hq):
    d = _desc(hq)
    ws = 1 << 20
    fake = 0x10000  # never dereferenced: every case below fails validation first
    cases = [
        (dict(m=-1), hq.HQ_ERR_INVALID_ARG),
        (dict(atype=9), hq.HQ_ERR_INVALID_ARG),
        (dict(x=None), hq.HQ_ERR_INVALID_ARG),
        (dict(ldx=100), hq.HQ_ERR_INVALID_ARG),
        (dict(atype="fp16"), hq.HQ_ERR_UNSUPPORTED),        # bf16 group scales need bf16 activations
        (dict(atype="fp8"), hq.HQ_ERR_UNSUPPORTED),
        (dict(x=fake + 8), hq.HQ_ERR_ALIGNMENT),
        (dict(ldx=516), hq.HQ_ERR_ALIGNMENT),
        (dict(ws_bytes=16), hq.HQ_ERR_WORKSPACE_TOO_SMALL),
    ]
    for over, want in cases:
        args = dict(desc=d, w_t=fake, m=16, atype="bf16", x=fake, ldx=512, x_scales=None, y=fake, ldy=256,
                    workspace=fake, ws_bytes=ws, flags=0, stream=None)
        args.update(over)
        with pytest.raises(hq.HQError) as ei:
            hq.hq_gemm(args["desc"], args["w_t"], args["m"], args["atype"], args["x"], args["ldx"],
                       args["x_scales"], args["y"], args["ldy"], args["workspace"], args["ws_bytes"],
                       args["flags"], args["stream"])
        assert ei.value.status == want, (over, ei.value.status)


def test_gemm_m_zero_returns_ok_without_gpu(hq):
    hq.hq_gemm(_desc(hq), 0, 0, "bf16", 0, 512, None, 0, 256, 0, 0, 0, None)


def test_moe_host_validation(hq):
    d = hq.make_desc("mxfp4", "ue8m0", 1536, 2048, num_experts=128, group_k=32)
    fake = 0x10000
    with pytest.raises(hq.HQError) as ei:
        hq.hq_moe_gemm(d, fake, 16, 0, fake, fake, "bf16", fake, 2048, fake, 1536, None, None, fake, 1 << 30)
    assert ei.value.status == hq.HQ_ERR_INVALID_ARG
    with pytest.raises(hq.HQError) as ei:
        hq.hq_moe_gemm(d, fake, 16, 8, fake, fake, "fp16", fake, 2048, fake, 1536, None, None, fake, 1 << 30)
    assert ei.value.status == hq.HQ_ERR_UNSUPPORTED
    need = hq.hq_moe_workspace_size(d, 4096, 8, "bf16")
    assert need >= 4096 * 8 * 1536 * 4
    # W4A8 (activations quantised to MXFP8 on the gather): MXFP4 experts only,
    # K a multiple of 128; the quantised rows fit the bf16 rows' space
    assert hq.hq_moe_workspace_size(d, 4096, 8, "mxfp8") == need
    di4 = hq.make_desc("int4", "bf16", 1536, 2048, num_experts=128, group_k=128)
    with pytest.raises(hq.HQError) as ei:
        hq.hq_moe_gemm(di4, fake, 16, 8, fake, fake, "mxfp8", fake, 2048, fake, 1536, None, None, fake, 1 << 30)
    assert ei.value.status == hq.HQ_ERR_UNSUPPORTED
    dk = hq.make_desc("mxfp4", "ue8m0", 1536, 2080, num_experts=128, group_k=32)
    with pytest.raises(hq.HQError) as ei:
        hq.hq_moe_gemm(dk, fake, 16, 8, fake, fake, "mxfp8", fake, 2080, fake, 1536, None, None, fake, 1 << 30)
    assert ei.value.status == hq.HQ_ERR_UNSUPPORTED


def test_moe_grouped_host_validation(hq):
    d = hq.make_desc("mxfp4", "ue8m0", 1536, 2048, num_experts=128, group_k=32)
    fake = 0x10000
    with pytest.raises(hq.HQError) as ei:  # unknown form
        hq.hq_moe_grouped_gemm(d, fake, 7, 64, fake, 0, "bf16", fake, 2048, fake, 1536, fake, 1 << 30)
    assert ei.value.status == hq.HQ_ERR_INVALID_ARG
    with pytest.raises(hq.HQError) as ei:  # fp16 activations: the grouped kernels are bf16-only
        hq.hq_moe_grouped_gemm(d, fake, hq.HQ_MOE_GROUPED_MASKED, 64, fake, 0, "fp16", fake, 2048, fake, 1536,
                               fake, 1 << 30)
    assert ei.value.status == hq.HQ_ERR_UNSUPPORTED
    with pytest.raises(hq.HQError) as ei:  # unaligned row pitch
        hq.hq_moe_grouped_gemm(d, fake, hq.HQ_MOE_GROUPED_CONTIGUOUS, 64, fake, 0, "bf16", fake, 2052, fake, 1536,
                               fake, 1 << 30)
    assert ei.value.status == hq.HQ_ERR_ALIGNMENT
    small = hq.hq_moe_grouped_workspace_size(d, hq.HQ_MOE_GROUPED_MASKED, 64)
    with pytest.raises(hq.HQError) as ei:
        hq.hq_moe_grouped_gemm(d, fake, hq.HQ_MOE_GROUPED_MASKED, 64, fake, 0, "bf16", fake, 2048, fake, 1536,
                               fake, small - 1)
    assert ei.value.status == hq.HQ_ERR_WORKSPACE_TOO_SMALL
    # the row map covers E * rows (masked) or rows (contiguous) entries
    assert small >= 128 * 64 * 4
    assert hq.hq_moe_grouped_workspace_size(d, hq.HQ_MOE_GROUPED_CONTIGUOUS, 64) < small
    hq.hq_moe_grouped_gemm(d, 0, hq.HQ_MOE_GROUPED_MASKED, 0, 0, 0, "bf16", 0, 2048, 0, 1536, 0, 0)  # no rows


def test_workspace_sizes_bounded(hq):
    d = _desc(hq, n=8192, k=8192, has_zeros=True, signed_codes=False)
    small = hq.hq_gemm_workspace_size(d, 16, "bf16")
    big = hq.hq_gemm_workspace_size(d, 4096, "bf16")
    assert small >= 256
    # large M needs no split-K scratch; small M needs at most 64 splits of fp32 partials
    assert big < 64 << 20
    assert small <= 256 + 64 * 16 * 8192 * 4 + (1 << 20)


def test_size_limits_rejected_on_host(hq):
    """Shapes whose tile counts or offsets would leave 32-bit range are
    refused before any launch (and before any device query)."""
    fake = 0x10000
    for kw in (dict(n=(1 << 28) + 128), dict(k=(1 << 28) + 128)):
        with pytest.raises(hq.HQError) as ei:
            hq.hq_transform_size(_desc(hq, **kw))
        assert ei.value.status == hq.HQ_ERR_UNSUPPORTED
    hq.hq_transform_size(_desc(hq, n=1 << 20, k=1 << 20))  # large but within the limits
    # dense: M above 2^30, or (M/16 + 1) * n_tiles at 2^31
    d = _desc(hq, n=1 << 20)  # 8192 n-tiles
    for m in ((1 << 30) + 1, (1 << 22) * 16):
        with pytest.raises(hq.HQError) as ei:
            hq.hq_gemm_workspace_size(d, m, "bf16")
        assert ei.value.status == hq.HQ_ERR_UNSUPPORTED
        with pytest.raises(hq.HQError) as ei:
            hq.hq_gemm(d, fake, m, "bf16", fake, 512, None, fake, 1 << 20, fake, 1 << 20, 0, None)
        assert ei.value.status == hq.HQ_ERR_UNSUPPORTED
    # MoE: 2^24 pairs over 8192 n-tiles overflow the device tile counter
    dm = hq.make_desc("mxfp4", "ue8m0", 1 << 20, 2048, num_experts=8, group_k=32)
    with pytest.raises(hq.HQError) as ei:
        hq.hq_moe_gemm(dm, fake, 1 << 21, 8, fake, fake, "bf16", fake, 2048, fake, 1 << 20, None, None, fake,
                       1 << 62)
    assert ei.value.status == hq.HQ_ERR_UNSUPPORTED
    with pytest.raises(hq.HQError) as ei:
        hq.hq_moe_grouped_gemm(dm, fake, hq.HQ_MOE_GROUPED_MASKED, 1 << 21, fake, 0, "bf16", fake, 2048, fake,
                               1 << 20, fake, 1 << 62)
    assert ei.value.status == hq.HQ_ERR_UNSUPPORTED


def test_selftest_timeout_host_validation(hq):
    for ws, want in [(None, hq.HQ_ERR_INVALID_ARG), (0x10008, hq.HQ_ERR_ALIGNMENT)]:
        with pytest.raises(hq.HQError) as ei:
            hq.hq_selftest_wait_timeout(ws)
        assert ei.value.status == want


def test_noalloc_rejects_problems_beyond_the_scratch(hq):
    """hq_gemm_noalloc refuses, on the host and before any device query or
    launch, a problem whose workspace would exceed its fixed scratch."""
    d = hq.make_desc("int4", "bf16", 16384, 16384, group_k=128, has_zeros=True, signed_codes=False)
    assert hq.hq_gemm_workspace_size(d, 64, "bf16") > hq.HQ_NOALLOC_SCRATCH_BYTES
    fake = 0x10000  # never dereferenced: the size check comes first
    for flags in (0, hq.HQ_FLAG_NOALLOC_RESET):
        with pytest.raises(hq.HQError) as ei:
            hq.hq_gemm_noalloc(d, fake, 64, "bf16", fake, 16384, None, fake, 16384, flags, None, None)
        assert ei.value.status == hq.HQ_ERR_WORKSPACE_TOO_SMALL


def test_mxfp8_quantize_host_validation(hq):
    fake = 0x10000
    for args, want in [((4, 48, fake, 48, fake, 48, fake, 2), hq.HQ_ERR_INVALID_ARG),        # k % 32
                       ((4, 64, fake, 60, fake, 64, fake, 2), hq.HQ_ERR_INVALID_ARG),        # ldx < k
                       ((4, 64, fake + 8, 64, fake, 64, fake, 2), hq.HQ_ERR_ALIGNMENT),      # x not 16-byte aligned
                       ((4, 64, fake, 68, fake, 64, fake, 2), hq.HQ_ERR_ALIGNMENT),          # ldx % 8
                       ((4, 64, fake, 64, fake + 4, 64, fake, 2), hq.HQ_ERR_ALIGNMENT)]:     # q not 8-byte aligned
        with pytest.raises(hq.HQError) as ei:
            hq.hq_mxfp8_quantize(*args)
        assert ei.value.status == want, (args, ei.value.status)
    hq.hq_mxfp8_quantize(0, 64, 0, 64, 0, 64, 0, 2)     # no rows: no-op without a device


def test_w4a8_host_validation(hq):
    """MXFP8 activations (W4A8-MXFP4) are taken only against MXFP4 weights,
    with K a multiple of 128 and 4-byte aligned exponent rows; checked on the
    host before any device query."""
    fake = 0x10000
    mx = hq.make_desc("mxfp4", "ue8m0", 256, 512, group_k=32)
    i4 = hq.make_desc("int4", "bf16", 256, 512, group_k=128)
    cases = [(i4, 512, fake, hq.HQ_ERR_UNSUPPORTED),                   # INT4 weights
             (hq.make_desc("mxfp4", "ue8m0", 256, 544, group_k=32), 544, fake, hq.HQ_ERR_INVALID_ARG),  # K % 128
             (mx, 512, None, hq.HQ_ERR_INVALID_ARG),                   # no exponents
             (mx, 512, fake + 2, hq.HQ_ERR_ALIGNMENT)]                 # exponents not 4-byte aligned
    for d, k, xs, want in cases:
        with pytest.raises(hq.HQError) as ei:
            hq.hq_gemm(d, fake, 16, "mxfp8", fake, k, xs, fake, 256, fake, 1 << 20, 0, None)
        assert ei.value.status == want, (k, xs, ei.value.status)
