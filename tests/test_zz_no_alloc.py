"""hq_gemm_noalloc (library-owned scratch, no workspace argument) against
hq_gemm with a caller workspace, on two calls in a row (GPU).

The same kernels run on the same inputs in the same plan, so the no-alloc
output must equal hq_gemm's bit for bit; both are also checked against the
CPU oracle.  Collected last: the scratch is process-wide, so this file also
checks that earlier tests leave nothing in it that breaks the next call.
(The host-side size limit is checked without a GPU in test_abi.py.)
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from tolerance import check

pytestmark = pytest.mark.gpu

CASES = [
    # name, weight + activation maker, M, N, K
    ("w4a16-asym-splitk", lambda: synth.dense_w4a16_asym(11, 16, 1024, 4096)),
    ("w4a16-sym-g64-ragged", lambda: synth.dense_w4a16_sym(12, 37, 520, 960, group_k=64)),
    ("int6-channel", lambda: synth.dense_int6_channel(13, 8, 640, 2048)),
    ("w4a16-asym-m300", lambda: synth.dense_w4a16_asym(14, 300, 768, 1536)),
    ("fp8-block", lambda: synth.dense_fp8_block(15, 24, 512, 2048)),
]


def _inputs(qw, acts):
    from gpu_helpers import DevWeight, to_dev
    dw = DevWeight(qw)
    m, k, n = acts.m, acts.k, qw.n
    esz = 1 if acts.atype == "fp8" else 2
    ldx = -(-k * esz // 16) * 16 // esz
    ldy = -(-n // 8) * 8
    xh = np.zeros((m, ldx), np.uint8 if acts.atype == "fp8" else np.uint16)
    xh[:, :k] = acts.data
    x = to_dev(xh)
    xs = to_dev(np.ascontiguousarray(acts.scales, np.float32)) if acts.scales is not None else None
    out_dtype = torch.float16 if acts.atype == "fp16" else torch.bfloat16
    return dw, x, ldx, xs, ldy, out_dtype


@pytest.mark.parametrize("idx", range(len(CASES)), ids=[c[0] for c in CASES])
def test_noalloc_matches_hq_gemm_twice(idx):
    import quantized_gemm_tma_gb300 as hq
    from gpu_helpers import stream, workspace
    qw, acts = CASES[idx][1]()
    dw, x, ldx, xs, ldy, out_dtype = _inputs(qw, acts)
    m, n = acts.m, qw.n

    ws = workspace(hq.hq_gemm_workspace_size(dw.desc, m, acts.atype))
    y_ref = torch.full((m, ldy), float("nan"), dtype=out_dtype, device="cuda")
    hq.hq_gemm(dw.desc, dw.wt, m, acts.atype, x, ldx, xs, y_ref, ldy, ws, ws.numel(), 0, stream())
    assert hq.hq_status_read(ws, clear=True, stream=stream()) == 0
    ref = y_ref[:, :n].double().cpu().numpy()
    w = oracle.dequantize(qw.wtype, qw.n, qw.k, qw.codes, qw.scales, qw.zeros, qw.group_k, qw.signed, qw.stype,
                          qw.num_experts)
    check(ref, oracle.gemm_dense(oracle.decode_activations(acts.atype, acts.data, acts.scales), w),
          f"{CASES[idx][0]} hq_gemm vs oracle")

    status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    for call in range(2):
        y = torch.full((m, ldy), float("nan"), dtype=out_dtype, device="cuda")
        hq.hq_gemm_noalloc(dw.desc, dw.wt, m, acts.atype, x, ldx, xs, y, ldy, 0, status, stream())
        torch.cuda.synchronize()
        assert int(status.item()) == 0, f"call {call}: device status {int(status.item())}"
        got = y[:, :n].double().cpu().numpy()
        assert np.array_equal(got, ref), f"{CASES[idx][0]} no-alloc call {call}: differs from hq_gemm"


def test_noalloc_reset_flag():
    """HQ_FLAG_NOALLOC_RESET clears the scratch's status word and counters on
    the stream before the GEMM; the result is unchanged."""
    import quantized_gemm_tma_gb300 as hq
    from gpu_helpers import stream
    qw, acts = CASES[0][1]()
    dw, x, ldx, xs, ldy, out_dtype = _inputs(qw, acts)
    m, n = acts.m, qw.n
    status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    outs = []
    for flags in (hq.HQ_FLAG_NOALLOC_RESET, 0, hq.HQ_FLAG_NOALLOC_RESET):
        y = torch.full((m, ldy), float("nan"), dtype=out_dtype, device="cuda")
        hq.hq_gemm_noalloc(dw.desc, dw.wt, m, acts.atype, x, ldx, xs, y, ldy, flags, status, stream())
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        outs.append(y[:, :n].double().cpu().numpy())
    assert np.array_equal(outs[0], outs[1]) and np.array_equal(outs[0], outs[2])
