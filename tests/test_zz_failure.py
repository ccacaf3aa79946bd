"""Failure detection without a fault (GPU): a bounded device wait that nothing
completes runs out, the status word reports HQ_ERR_DEVICE_TIMEOUT, and the
context keeps working."""
import time

import pytest

import oracle
import synth
from tolerance import check

pytestmark = pytest.mark.gpu


def test_bounded_wait_reports_timeout_and_context_survives():
    import quantized_gemm_tma_gb300 as hq
    from gpu_helpers import DevWeight, run_gemm, stream, workspace
    ws = workspace(256)
    t0 = time.perf_counter()
    hq.hq_selftest_wait_timeout(ws, stream())
    st = hq.hq_status_read(ws, clear=True, stream=stream())
    waited = time.perf_counter() - t0
    assert st == hq.HQ_ERR_DEVICE_TIMEOUT
    assert 0.2 < waited < 60.0, waited                 # the wait's limit is about 2 s
    assert hq.hq_status_read(ws, clear=False, stream=stream()) == hq.HQ_OK   # cleared
    # the same context still computes correctly
    qw, acts = synth.dense_w4a16_asym(3, 16, 256, 512)
    check(run_gemm(DevWeight(qw), acts), oracle.gemm.reference(qw, acts), "after a device timeout")
