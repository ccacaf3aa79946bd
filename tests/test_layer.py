"""QuantLinear: configuration and size checks on the host (CPU), and the
forward pass against the CPU oracle (GPU)."""
import numpy as np
import pytest
import torch

import oracle
import synth
from tolerance import check


@pytest.fixture(scope="module")
def hq():
    import quantized_gemm_tma_gb300 as m
    from quantized_gemm_tma_gb300 import _build
    _build.build()
    return m


def test_layer_checks_configuration_and_sizes(hq):
    from quantized_gemm_tma_gb300.layer import QuantLinear
    with pytest.raises(hq.HQError):
        QuantLinear(256, 500, "int4", "bf16", group_k=128)          # K not a multiple of the group
    lin = QuantLinear(256, 512, "int4", "bf16", group_k=128, signed_codes=False, has_zeros=True)
    assert lin.standard_bytes() == {"codes": 256 * 256, "scales": 2 * 256 * 4, "zeros": 256 * 2}
    codes = torch.zeros(256 * 256, dtype=torch.uint8)
    scales = torch.zeros(256 * 4, dtype=torch.int16)
    zeros = torch.zeros(256 * 2, dtype=torch.uint8)
    lin.load(codes, scales, zeros)
    with pytest.raises(ValueError):
        lin.load(codes[:-1], scales, zeros)                          # one byte short
    with pytest.raises(ValueError):
        lin.load(codes, scales, None)                                # zero points missing
    with pytest.raises(RuntimeError):
        lin(torch.zeros(4, 512, dtype=torch.bfloat16))               # not transformed
    sym = QuantLinear(128, 256, "mxfp4", "ue8m0", group_k=32)
    with pytest.raises(ValueError):
        sym.load(torch.zeros(128 * 128, dtype=torch.uint8), torch.zeros(128 * 8, dtype=torch.uint8),
                 torch.zeros(4, dtype=torch.uint8))                  # MXFP4 takes no zero points


@pytest.mark.gpu
def test_layer_forward_matches_oracle(hq):
    from quantized_gemm_tma_gb300.layer import QuantLinear

    def dev(a):
        a = np.ascontiguousarray(a)
        return torch.from_numpy(a.view(np.int16) if a.dtype == np.uint16 else a).cuda()

    # INT4 with zero points, ragged N, a non-contiguous activation view
    qw, acts = synth.dense_w4a16_asym(21, 40, 200, 512)
    lin = QuantLinear(200, 512, "int4", "bf16", group_k=128, signed_codes=False, has_zeros=True)
    lin.load(dev(qw.codes), dev(qw.scales), dev(qw.zeros)).transform()
    xfull = torch.zeros((40, 1024), dtype=torch.bfloat16, device="cuda")
    xfull[:, ::2] = dev(acts.data).view(torch.bfloat16)
    y = lin(xfull[:, ::2])
    assert y.shape == (40, 200)
    check(y.double().cpu().numpy(), oracle.gemm.reference(qw, acts), "layer int4 asym")
    # INT6 channelwise, fp16
    qw, acts = synth.dense_int6_channel(22, 24, 256, 512)
    lin = QuantLinear(256, 512, "int6", "fp16", group_k=0)
    lin.load(dev(qw.codes), dev(qw.scales)).transform()
    check(lin(dev(acts.data).view(torch.float16)).double().cpu().numpy(), oracle.gemm.reference(qw, acts),
          "layer int6 fp16")
    # FP8 blocks with per-token activation scales
    qw, acts = synth.dense_fp8_block(23, 64, 256, 384)
    lin = QuantLinear(256, 384, "fp8", "fp32", group_k=128, group_n=128)
    lin.load(dev(qw.codes), dev(qw.scales)).transform()
    check(lin(dev(acts.data), dev(acts.scales)).double().cpu().numpy(), oracle.gemm.reference(qw, acts),
          "layer fp8")


@pytest.mark.parametrize("wtype,stype,group_k,zeros,n,k", [
    ("int4", "bf16", 128, False, 200, 512), ("int4", "fp16", 32, True, 130, 96), ("int4", "bf16", 0, True, 77, 260),
    ("int6", "fp16", 0, False, 256, 512), ("int6", "bf16", 64, True, 130, 384), ("mxfp4", "ue8m0", 32, False, 150, 96),
    ("fp8", "fp32", 128, False, 130, 200),
])
def test_layer_sizes_match_the_standard_format(hq, wtype, stype, group_k, zeros, n, k):
    """The sizes QuantLinear checks are those of the standard-format arrays the generators write."""
    from quantized_gemm_tma_gb300.layer import QuantLinear
    qw = synth.random_codes_weight(5, wtype, n, k, group_k=group_k, has_zeros=zeros,
                                   stype=stype if stype in ("bf16", "fp16") else None)
    lin = QuantLinear(n, k, wtype, stype, group_k=group_k, group_n=128 if wtype == "fp8" else 1,
                      signed_codes=qw.signed, has_zeros=zeros)
    want = lin.standard_bytes()
    assert want["codes"] == qw.codes.nbytes and want["scales"] == qw.scales.nbytes
    assert want["zeros"] == (qw.zeros.nbytes if zeros else 0)
