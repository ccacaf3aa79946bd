"""Move ``synth`` inputs to the device and call the library through its C ABI.

Only argument marshalling lives here: numpy arrays become torch CUDA tensors
with the same bytes, and results come back as float64 numpy arrays for the
comparison with the oracle.
"""
from __future__ import annotations

import numpy as np
import torch

import quantized_gemm_tma_gb300 as hq


def to_dev(a: np.ndarray) -> torch.Tensor:
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        t = torch.from_numpy(a.view(np.int16))
    elif a.dtype in (np.uint8, np.float32, np.int32, np.int16):
        t = torch.from_numpy(a)
    else:
        raise TypeError(a.dtype)
    return t.cuda()


def from_dev_u(t: torch.Tensor, dtype) -> np.ndarray:
    return t.cpu().numpy().view(dtype)


def stream():
    return torch.cuda.current_stream().cuda_stream


class DevWeight:
    """A standard-format weight on the device plus its hq_transform output."""

    def __init__(self, qw, transform: bool = True):
        self.qw = qw
        self.codes = to_dev(qw.codes)
        self.scales = to_dev(qw.scales)
        self.zeros = to_dev(qw.zeros) if qw.zeros is not None else None
        ts = getattr(qw, "tensor_scale", None)
        self.tensor_scales = to_dev(np.asarray(ts, np.float32)) if ts is not None else None
        self.desc = hq.make_desc(qw.wtype, qw.stype, qw.n, qw.k, qw.num_experts, qw.group_k, qw.group_n,
                                 qw.signed, qw.has_zeros, self.codes, self.scales, self.zeros,
                                 self.tensor_scales)
        self.size = hq.hq_transform_size(self.desc)
        self.wt = torch.empty(self.size + 256, dtype=torch.uint8, device="cuda")
        off = (-self.wt.data_ptr()) % 256
        self.wt = self.wt[off:off + self.size]
        if transform:
            hq.hq_transform(self.desc, self.wt, self.size, stream())

    def untransform(self):
        codes = torch.zeros_like(self.codes)
        scales = torch.zeros_like(self.scales)
        zeros = torch.zeros_like(self.zeros) if self.zeros is not None else None
        if self.tensor_scales is not None:          # NVFP4: tensor scales come back through `zeros`
            zeros = torch.zeros_like(self.tensor_scales)
        hq.hq_untransform(self.desc, self.wt, codes, scales, zeros, stream())
        torch.cuda.synchronize()
        return codes, scales, zeros


def workspace(nbytes: int) -> torch.Tensor:
    ws = torch.zeros(max(nbytes, 256), dtype=torch.uint8, device="cuda")
    return ws


def run_gemm(dw: DevWeight, acts, ldx: int | None = None, ldy: int | None = None, flags: int = 0,
             ws: torch.Tensor | None = None) -> np.ndarray:
    """hq_gemm on device copies of ``acts``; returns Y as float64 [M, N]."""
    m, k = acts.m, acts.k
    n = dw.qw.n
    esz = 1 if acts.atype == "fp8" else 2
    ldx = ldx or -(-k * esz // 16) * 16 // esz      # rows 16-byte aligned (the TMA stride rule)
    ldy = ldy or -(-n // 8) * 8
    if acts.atype == "fp8":
        xh = np.zeros((m, ldx), np.uint8)
    else:
        xh = np.zeros((m, ldx), np.uint16)
    xh[:, :k] = acts.data
    x = to_dev(xh)
    xs = to_dev(np.ascontiguousarray(acts.scales, np.float32)) if acts.scales is not None else None
    out_dtype = torch.float16 if acts.atype == "fp16" else torch.bfloat16
    y = torch.full((max(m, 1), ldy), float("nan"), dtype=out_dtype, device="cuda")
    need = hq.hq_gemm_workspace_size(dw.desc, m, acts.atype)
    if ws is None:
        ws = workspace(need)
    hq.hq_gemm(dw.desc, dw.wt, m, acts.atype, x, ldx, xs, y, ldy, ws, ws.numel(), flags, stream())
    st = hq.hq_status_read(ws, clear=True, stream=stream())
    if st != 0:
        raise hq.HQError(st, "device status")
    return y[:m, :n].double().cpu().numpy()


def run_moe(dw: DevWeight, acts, routing, ws: torch.Tensor | None = None, want_route: bool = False,
            atype: str = "bf16"):
    """hq_moe_gemm on device copies; atype "mxfp8" quantises the bf16 rows to
    MXFP8 as they are gathered (W4A8)."""
    t, k = acts.m, acts.k
    topk = routing.topk_ids.shape[1]
    n = dw.qw.n
    x = to_dev(acts.data)
    ids = to_dev(np.ascontiguousarray(routing.topk_ids, np.int32))
    tw = to_dev(np.ascontiguousarray(routing.topk_w, np.float32))
    y = torch.full((max(t, 1), n), float("nan"), dtype=torch.bfloat16, device="cuda")
    e = dw.qw.num_experts
    offs = torch.full((e + 1,), -1, dtype=torch.int32, device="cuda") if want_route else None
    perm = torch.full((max(t * topk, 1),), -1, dtype=torch.int32, device="cuda") if want_route else None
    need = hq.hq_moe_workspace_size(dw.desc, t, topk, atype)
    if ws is None:
        ws = workspace(need)
    hq.hq_moe_gemm(dw.desc, dw.wt, t, topk, ids, tw, atype, x, k, y, n, offs, perm, ws, ws.numel(), 0, stream())
    st = hq.hq_status_read(ws, clear=True, stream=stream())
    out = y[:t, :n].double().cpu().numpy()
    if want_route:
        return out, st, offs.cpu().numpy(), perm[: t * topk].cpu().numpy()
    return out, st


class tuning:
    """Set HQ_FORCE_* switches for the duration of a ``with`` block (in this
    process: the library re-reads them through hq_tuning_reload)."""

    def __init__(self, **switches):
        self.switches = {k: str(v) for k, v in switches.items()}
        self.saved = {}

    def __enter__(self):
        import os
        for k, v in self.switches.items():
            self.saved[k] = os.environ.get(k)
            os.environ[k] = v
        hq.hq_tuning_reload()
        return self

    def __exit__(self, *exc):
        import os
        for k, v in self.saved.items():
            if v is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = v
        hq.hq_tuning_reload()
        return False
