"""MXFP8 activation quantisation (the activation side of W4A8-MXFP4): codes
and block exponents bit-exact against the CPU oracle (GPU)."""
import numpy as np
import pytest

import oracle
import synth
from oracle import formats as F

pytestmark = pytest.mark.gpu


def _inputs(seed, m, k):
    """Normal values with a spread of block magnitudes, plus the edge cases:
    an all-zero block, signed zeros, values far below their block's maximum,
    exact rounding ties and maxima that saturate."""
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((m, k)) * np.exp2(rng.integers(-40, 40, size=(m, k // 32))).repeat(32, axis=1)
    x[0, :32] = 0.0
    if k >= 64:
        x[0, 32:64] = -0.0
    if m > 1 and k >= 64:
        x[1, :32] = 2.0 ** -120                                   # tiny against ...
        x[1, 5] = 3.0e30                                           # ... a huge block maximum
        x[1, 32:64] = [256.0, 17.0, 19.0, -17.0, 480.0, 464.0, 9.5, 0.00390625] * 4   # ties, saturation
    return synth.to_bf16_bits(x)


@pytest.mark.parametrize("m,k", [(1, 32), (16, 2048), (37, 7168), (300, 96)])
def test_mxfp8_quantize_bit_exact(m, k):
    import torch
    import quantized_gemm_tma_gb300 as hq
    from gpu_helpers import stream, to_dev
    xb = _inputs(m * 7 + k, m, k)
    ref_q, ref_e = oracle.w4a8.mxfp8_quantize(F.bf16_to_f64(xb))
    ldx, ldq, lde = k + 8, k + 16, k // 32 + 3                    # strided rows on every side
    xh = np.zeros((m, ldx), np.uint16)
    xh[:, :k] = xb
    q = torch.full((m, ldq), 0xAA, dtype=torch.uint8, device="cuda")
    e = torch.full((m, lde), 0xAA, dtype=torch.uint8, device="cuda")
    hq.hq_mxfp8_quantize(m, k, to_dev(xh), ldx, q, ldq, e, lde, stream())
    torch.cuda.synchronize()
    qh, eh = q.cpu().numpy(), e.cpu().numpy()
    assert np.array_equal(eh[:, :k // 32], ref_e)
    bad = np.argwhere(qh[:, :k] != ref_q)
    assert bad.size == 0, (bad[:8].tolist(), qh[tuple(bad[0])], ref_q[tuple(bad[0])])
    assert (qh[:, k:] == 0xAA).all() and (eh[:, k // 32:] == 0xAA).all()     # nothing written past a row
