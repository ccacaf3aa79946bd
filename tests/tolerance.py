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
"""
import numpy as np

FROB_TOL = 5e-3
ELEM_REL = 2.0 ** -7
ELEM_ABS_RMS = 1e-2


def check(y, r, what=""):
    y = np.asarray(y, dtype=np.float64)
    r = np.asarray(r, dtype=np.float64)
    assert y.shape == r.shape, (what, y.shape, r.shape)
    assert np.all(np.isfinite(y)), f"{what}: non-finite output"
    nr = np.linalg.norm(r)
    rel = np.linalg.norm(y - r) / max(nr, 1e-300)
    rms = nr / np.sqrt(max(r.size, 1))
    bound = ELEM_REL * np.abs(r) + ELEM_ABS_RMS * rms
    bad = np.abs(y - r) > bound
    assert rel <= FROB_TOL, f"{what}: relative Frobenius error {rel:.3e} > {FROB_TOL}"
    if bad.any():
        i = np.argwhere(bad)[0]
        raise AssertionError(f"{what}: {int(bad.sum())} elements out of bound, first at {tuple(i)}: "
                             f"y={y[tuple(i)]!r} ref={r[tuple(i)]!r} bound={bound[tuple(i)]!r}")
    return rel
