"""The GEMM output tolerance used by every parity test.

A kernel output Y (upcast to float64) agrees with the oracle R when
    ||Y - R||_F / ||R||_F <= 5e-3                        (relative Frobenius)
and, element by element,
    |Y - R| <= 2^-7 * |R| + 1e-2 * rms(R).
The first bound absorbs fp32 accumulation order; the second absorbs the
rounding of the output to bf16/fp16 (relative 2^-8 or 2^-11) and of
intermediate dequantised weights to bf16 (asymmetric int4 rounds (q-z)*s to
bf16 before the tensor-core product), with an absolute floor for outputs that
cancel to near zero.

The MoE feed-forward block chains two GEMMs through an intermediate that the
library holds in bf16 (the 16-bit operand of the down GEMM):
    y = sum_j w_j * W2 . bf16(silu(g) * u),  [g, u] = W13 . x.
Each GEMM meets the tolerance above against exact arithmetic.  The gate-up
errors reach the down GEMM's operand scaled by the sensitivity of
silu(g) * u (order one: |d silu/dg| <= 1.1), so the relative errors of the two
stages add.  The bf16 rounding of the intermediate adds one more half-ulp
(2^-9) per operand element.  The block is therefore compared with the exact
oracle (exact weights, exact intermediates) at twice both constants:
    ||Y - R||_F / ||R||_F <= 1e-2,  |Y - R| <= 2^-6 * |R| + 2e-2 * rms(R).
"""
import numpy as np

FROB_TOL = 5e-3
ELEM_REL = 2.0 ** -7
ELEM_ABS_RMS = 1e-2

FFN_FROB_TOL = 2 * FROB_TOL
FFN_ELEM_REL = 2 * ELEM_REL
FFN_ELEM_ABS_RMS = 2 * ELEM_ABS_RMS


def check_ffn(y, r, what=""):
    """The tolerance of the two-GEMM MoE feed-forward block (see above)."""
    return check(y, r, what, FFN_FROB_TOL, FFN_ELEM_REL, FFN_ELEM_ABS_RMS)


def check(y, r, what="", frob_tol=FROB_TOL, elem_rel=ELEM_REL, elem_abs_rms=ELEM_ABS_RMS):
    y = np.asarray(y, dtype=np.float64)
    r = np.asarray(r, dtype=np.float64)
    assert y.shape == r.shape, (what, y.shape, r.shape)
    assert np.all(np.isfinite(y)), f"{what}: non-finite output"
    nr = np.linalg.norm(r)
    rel = np.linalg.norm(y - r) / max(nr, 1e-300)
    rms = nr / np.sqrt(max(r.size, 1))
    bound = elem_rel * np.abs(r) + elem_abs_rms * rms
    bad = np.abs(y - r) > bound
    assert rel <= frob_tol, f"{what}: relative Frobenius error {rel:.3e} > {frob_tol}"
    if bad.any():
        i = np.argwhere(bad)[0]
        raise AssertionError(f"{what}: {int(bad.sum())} elements out of bound, first at {tuple(i)}: "
                             f"y={y[tuple(i)]!r} ref={r[tuple(i)]!r} bound={bound[tuple(i)]!r}")
    return rel
