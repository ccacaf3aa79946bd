"""hq_transform -> hq_untransform is the identity, bit for bit (GPU)."""
import numpy as np
import pytest

import synth

pytestmark = pytest.mark.gpu

CASES = [
    # wtype, n, k, group_k, signed, zeros, stype
    ("int4", 256, 1024, 128, True, False, "bf16"),
    ("int4", 200, 640, 128, False, True, "bf16"),     # ragged N
    ("int4", 130, 96, 32, True, False, "fp16"),       # K < one tile, group 32
    ("int4", 129, 192, 64, False, True, "bf16"),      # ragged K with group 64
    ("int4", 64, 512, 256, False, True, "bf16"),      # group spans two tiles
    ("int4", 77, 101, 0, True, False, "bf16"),        # channelwise, odd K
    ("int4", 77, 260, 0, False, True, "fp16"),        # channelwise with zeros
    ("int6", 256, 512, 0, True, False, "fp16"),       # the INT6 channelwise format
    ("int6", 130, 384, 128, False, True, "bf16"),
    ("int6", 64, 160, 32, True, False, "bf16"),
    ("int6", 33, 1024, 512, False, True, "fp16"),     # 2 groups -> padded 6-bit zero stream
    ("mxfp4", 256, 512, 32, True, False, "ue8m0"),
    ("mxfp4", 150, 96, 32, True, False, "ue8m0"),
    ("fp8", 256, 384, 128, True, False, "fp32"),
    ("fp8", 130, 200, 128, True, False, "fp32"),
    ("nvfp4", 256, 512, 16, True, False, "e4m3"),
    ("nvfp4", 150, 96, 16, True, False, "e4m3"),      # ragged N, K < one tile
    ("mxint4", 256, 512, 32, True, False, "ue8m0"),
    ("mxint4", 150, 96, 32, True, False, "ue8m0"),
]


@pytest.mark.parametrize("idx", range(len(CASES)), ids=lambda i: "-".join(map(str, CASES[i])))
def test_roundtrip_bit_exact(idx):
    from gpu_helpers import DevWeight
    wtype, n, k, g, signed, zeros, stype = CASES[idx]
    qw = synth.random_codes_weight(100 + idx, wtype, n, k, group_k=g, signed=signed, has_zeros=zeros,
                                   stype=stype if stype in ("bf16", "fp16") else None)
    dw = DevWeight(qw)
    codes, scales, z = dw.untransform()
    assert np.array_equal(codes.cpu().numpy(), qw.codes)
    assert np.array_equal(scales.cpu().numpy().view(qw.scales.dtype), qw.scales)
    if zeros:
        assert np.array_equal(z.cpu().numpy(), qw.zeros)
    if qw.tensor_scale is not None:                  # NVFP4 tensor scales come back through `zeros`
        assert np.array_equal(z.cpu().numpy(), qw.tensor_scale)


def test_roundtrip_moe_experts():
    from gpu_helpers import DevWeight
    qw = synth.random_codes_weight(3, "mxfp4", 256, 256, num_experts=5)
    dw = DevWeight(qw)
    codes, scales, _ = dw.untransform()
    assert np.array_equal(codes.cpu().numpy(), qw.codes)
    assert np.array_equal(scales.cpu().numpy(), qw.scales)


def test_roundtrip_nvfp4_experts():
    from gpu_helpers import DevWeight
    qw = synth.random_codes_weight(5, "nvfp4", 200, 160, num_experts=3)
    dw = DevWeight(qw)
    codes, scales, ts = dw.untransform()
    assert np.array_equal(codes.cpu().numpy(), qw.codes)
    assert np.array_equal(scales.cpu().numpy(), qw.scales)
    assert np.array_equal(ts.cpu().numpy(), qw.tensor_scale)


def test_transform_rejects_nan_nvfp4_scale():
    import quantized_gemm_tma_gb300 as hq
    from gpu_helpers import DevWeight
    qw = synth.random_codes_weight(6, "nvfp4", 128, 128)
    qw.scales[0, 9, 3] = 0xFF                        # e4m3 NaN
    with pytest.raises(hq.HQError) as ei:
        DevWeight(qw)
    assert ei.value.status == hq.HQ_ERR_INVALID_VALUE


def test_transform_rejects_nan_scale():
    import quantized_gemm_tma_gb300 as hq
    from gpu_helpers import DevWeight
    qw = synth.random_codes_weight(4, "mxfp4", 128, 128)
    qw.scales[0, 5, 1] = 255
    with pytest.raises(hq.HQError) as ei:
        DevWeight(qw)
    assert ei.value.status == hq.HQ_ERR_INVALID_VALUE


def test_transform_rejects_nan_e4m3():
    import quantized_gemm_tma_gb300 as hq
    from gpu_helpers import DevWeight
    qw = synth.random_codes_weight(4, "fp8", 128, 128)
    qw.codes[0, 3, 7] = 0x7F
    with pytest.raises(hq.HQError) as ei:
        DevWeight(qw)
    assert ei.value.status == hq.HQ_ERR_INVALID_VALUE
