#!/usr/bin/env python
"""Benchmark of the quantized GEMM hot path on one GB300 (or N replicas).

One step = one pass over the dense W4A16 workload the metric is quoted on:
asymmetric INT4 weights (uint4 zero points, group 128, bf16 scales), bf16
activations, N = K = 8192, for every M of the sweep {1, 16, 128, 1024, 4096}
(one hq_gemm call per M).  The MoE grouped GEMM (MXFP4 experts, E = 128,
N = 1536, K = 2048, top-8 routing, T in {16, 256, 4096}) is timed the same
way and reported under "moe".

Timing: W untimed warm-up steps, then K timed steps.  Each step makes one
call per shape; the K calls of one shape are issued back to back (as
consecutive layers of a model would be), timed with CUDA events on the
launching stream in blocks of 25 calls, so a kernel's launch can overlap the
previous kernel's tail (programmatic dependent launch).  Consecutive calls
rotate over 8 transformed copies of the weight (8 x 36 MiB, well above the
129 MB L2) and 4 copies of each activation, so no call finds its operands in
L2.  A device-side sleep is queued before the timed steps so that the host
enqueues ahead of the GPU and host submission gaps stay outside the events.
`value` is the whole-job aggregate TFLOP/s: all FLOPs of the timed steps on
all ranks over the slowest rank's summed GEMM time.  `e2e` is the same metric
through the public C-ABI call with host buffers: per step, the activations
are copied in from pinned host memory, the GEMMs run and the outputs are
copied back, timed by the host clock from enqueue to completion.

`--impl reference` times the CPU oracle (the parity reference; this subject
has no runnable reference implementation) on a bounded sample of the same
workload on the host cores.
"""
from __future__ import annotations

import argparse
import tempfile
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "Quantized GEMM TFLOP/s & HBM GB/s vs M (W4A16, MoE); % of roofline"
N = K = 8192
M_SWEEP = [1, 16, 128, 1024, 4096]
MOE_T = [16, 256, 4096]
MOE_E, MOE_N, MOE_K, MOE_TOPK = 128, 1536, 2048, 8
WORKLOAD = ("dense W4A16: asymmetric INT4 g128 (uint4 zeros, bf16 scales), bf16 activations, "
            "N=K=8192, M sweep {1,16,128,1024,4096}")
W_COPIES = 8       # rotated transformed weight copies (> L2 in total)
X_COPIES = 4       # rotated activation copies per M
MOE_COPIES = 2     # rotated MoE expert sets (213 MB each)
MOE_H = MOE_K      # feed-forward block: down projection [E][hidden = K][intermediate = N / 2]
HEAD_START_CYCLES = 200_000_000
# The other dense configurations, timed the same way as the sweep (extra keys
# of the JSON line): INT6 channelwise with fp16 activations at M = 128, and
# FP8 e4m3 with 128 x 128 block scales at M in {64, 512, 4096}.
EXTRA = {
    "c3_int6_channel_fp16": {"n": 8192, "k": 8192, "ms": [128], "copies": 4,
                             "workload": "dense INT6 channelwise symmetric (fp16 row scales), fp16 activations, "
                                         "N=K=8192, M=128"},
    "c4_fp8_block": {"n": 4096, "k": 7168, "ms": [64, 512, 4096], "copies": 6,
                     "workload": "dense W8A8 FP8: e4m3 weights with fp32 128x128 block scales, e4m3 activations "
                                 "with per-token per-128-K fp32 scales, N=4096, K=7168, M sweep {64,512,4096}"},
    "w4a8_mxfp4": {"n": 8192, "k": 8192, "ms": [1, 16, 128, 1024, 4096], "copies": 8,
                   "workload": "dense W4A8-MXFP4: MXFP4 weights (e2m1, UE8M0 per 32) against MXFP8 activations "
                               "(e4m3, UE8M0 per 32, quantised from bf16 by hq_mxfp8_quantize before the timed "
                               "calls), block-scaled MMA, N=K=8192, M sweep {1,16,128,1024,4096}"},
}
# FP8 dense peak: the measured bf16 peak times 2, the nominal fp8:bf16 ratio of
# the tensor cores (4.5 : 2.25 PFLOP/s dense)
FP8_PER_BF16 = 2.0
BLOCK = 25         # back-to-back calls of one shape between two events
# DRAM bytes (read + write) per launch of the WnA16 INT4 kernel, from one ncu
# capture (dram__bytes_read.sum + dram__bytes_write.sum, third warm-up pass of
# the dense sweep; the command is kept with the profile summaries), keyed by
# M; valid only while the kernel sources hash to `sha` (else null).
NCU_TRAFFIC = {"sha": "7f5bdcb60b8360de", "files": ["gemm_wna16.cuh", "hq_ptx.cuh", "wna16_int4.cu"],
               "bytes": {16: 35_467_776, 128: 37_304_576, 1024: 53_092_608, 4096: 170_119_424}}
FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def dense_bytes(m: int) -> int:
    """Algorithmic bytes of one W4A16 call: packed weights + scales + zeros + activations."""
    return N * K // 2 + N * (K // 128) * 2 + N * (K // 128) // 2 + m * K * 2


def dense_flops(m: int) -> int:
    return 2 * m * N * K


def extra_bytes(name: str, m: int) -> int:
    """Algorithmic bytes of one call of an extra configuration (output excluded)."""
    cfg = EXTRA[name]
    n, k = cfg["n"], cfg["k"]
    if name.startswith("c3"):   # 6-bit codes, fp16 row scales, fp16 activations
        return n * k * 3 // 4 + n * 2 + m * k * 2
    if name.startswith("w4a8"):  # e2m1 codes + UE8M0 per 32; e4m3 activations + UE8M0 per 32
        return n * k // 2 + n * k // 32 + m * k + m * k // 32
    kb = -(-k // 128)           # e4m3 weights, fp32 block scales, e4m3 activations, fp32 per-token scales
    return n * k + (-(-n // 128)) * kb * 4 + m * k + m * kb * 4


def ncu_traffic(m: int):
    """Captured DRAM bytes per launch at this M, or None if the kernel changed since."""
    import hashlib
    h = hashlib.sha256()
    for f in NCU_TRAFFIC["files"]:
        with open(os.path.join(ROOT, "quantized_gemm_tma_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    if h.hexdigest()[:16] != NCU_TRAFFIC["sha"]:
        return None
    return NCU_TRAFFIC["bytes"].get(m)


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        try:
            d = json.load(open(path))
            out = {}
            for key in ("hbm_gbs", "bf16_tflops", "bf16_tflops_sustained"):
                v = d.get(key)
                if isinstance(v, dict):
                    v = v.get("value")
                if isinstance(v, (int, float)) and v > 0:
                    out[key] = float(v)
            if "hbm_gbs" in out and "bf16_tflops" in out:
                out.setdefault("bf16_tflops_sustained", out["bf16_tflops"])
                out["source"] = "measured"
                return out
        except (OSError, ValueError):
            pass
    out = dict(FALLBACK)
    out["source"] = "fallback"
    return out


# ---------------------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, out_dir: str | None = None):
        self.idx = gpu_index
        self.proc = None
        self.out_dir = out_dir or tempfile.mkdtemp(prefix="hq_clocks_")
        self.path = os.path.join(self.out_dir, f"clocks_rank{gpu_index}.csv")

    def __enter__(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.idx), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=self.fh, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.fh.close()

    def summary(self):
        if self.proc is None or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for nm, val in zip(names, parts[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(nm)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------------------- oracle (CPU)
_ORACLE_W = {}


def cpu_oracle_sample(seed: int = 0, rows_cap: int = 256, n_rows: int = N):
    """Time the CPU oracle on a bounded sample of the same workload.

    One dequantisation of the first `n_rows` output rows of the N=K=8192 weight
    plus float64 matmuls against them for every M of the sweep, capped at
    `rows_cap` rows per M.  The quantised weight is generated once per process,
    outside the timed region.  Returns (TFLOP/s, seconds, description, cores).
    """
    import numpy as np
    import oracle
    import synth
    if seed not in _ORACLE_W:
        _ORACLE_W[seed] = synth.dense_w4a16_asym(seed, 1, N, K)[0]
    qw = _ORACLE_W[seed]
    codes = qw.codes[:, :n_rows]
    scales = qw.scales[:, :n_rows]
    zeros = qw.zeros[:, :n_rows] if qw.zeros is not None else None
    rng = np.random.default_rng(seed + 1)
    acts = [synth.to_bf16_bits(rng.standard_normal((min(m, rows_cap), K))) for m in M_SWEEP]
    t0 = time.perf_counter()
    w = oracle.dequantize(qw.wtype, n_rows, qw.k, codes, scales, zeros, qw.group_k, qw.signed, qw.stype, 1)
    flops = 0
    for a_bits in acts:
        a = oracle.decode_activations("bf16", a_bits)
        oracle.gemm_dense(a, w)
        flops += 2 * a_bits.shape[0] * n_rows * K
    dt = time.perf_counter() - t0
    cores = len(os.sched_getaffinity(0))
    desc = (f"oracle (numpy, float64) on the asym INT4 g128 weight (first {n_rows} of N=8192 rows, K=8192): one "
            f"dequantisation plus matmuls for M in {M_SWEEP} capped at {rows_cap} rows each "
            f"({flops / 1e9:.1f} GFLOP)")
    return flops / dt / 1e12, dt, desc, cores


# ---------------------------------------------------------------------------- GPU arm
def run_gpu(args, rank: int, world: int):
    import numpy as np
    import torch
    import quantized_gemm_tma_gb300 as hq
    import synth
    from quantized_gemm_tma_gb300 import _build

    if not os.path.exists(hq.LIB_PATH):
        _build.build()
    dev = torch.device("cuda", rank % torch.cuda.device_count())
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream()
    sh = stream.cuda_stream

    def to_dev(a):
        a = np.ascontiguousarray(a)
        t = torch.from_numpy(a.view(np.int16) if a.dtype == np.uint16 else a)
        return t.to(dev)

    # ---- dense workload (seeded), transformed once
    qw, _ = synth.dense_w4a16_asym(0, 1, N, K)
    codes, scales, zeros = to_dev(qw.codes), to_dev(qw.scales), to_dev(qw.zeros)
    desc = hq.make_desc("int4", "bf16", N, K, 1, 128, 1, False, True, codes, scales, zeros)
    wt_bytes = hq.hq_transform_size(desc)
    wts = []
    for _ in range(W_COPIES):
        wt = torch.empty(wt_bytes, dtype=torch.uint8, device=dev)
        hq.hq_transform(desc, wt, wt_bytes, sh)
        wts.append(wt)
    del codes, scales, zeros
    rng = np.random.default_rng(1)
    xs, ys, wss, xh, yh = {}, {}, {}, {}, {}
    for m in args.m_sweep:
        xb = synth.to_bf16_bits(rng.standard_normal((m, K)))
        xs[m] = [to_dev(xb) for _ in range(X_COPIES)]
        ys[m] = [torch.empty((m, N), dtype=torch.bfloat16, device=dev) for _ in range(X_COPIES)]
        need = hq.hq_gemm_workspace_size(desc, m, "bf16")
        wss[m] = torch.zeros(need, dtype=torch.uint8, device=dev)
        xh[m] = torch.from_numpy(xb.view(np.int16)).pin_memory()
        yh[m] = torch.empty((m, N), dtype=torch.bfloat16).pin_memory()
    launches = {"n": 0}
    rot = {"w": 0, "x": 0, "moe": 0, "extra": 0}

    # ---- the other dense configurations (weights rotated over copies > L2)
    extra = {}
    if not args.no_extra:
        for name, cfg in EXTRA.items():
            n_, k_ = cfg["n"], cfg["k"]
            if name.startswith("c3"):
                eq, _ = synth.dense_int6_channel(0, 1, n_, k_)
                atype = "fp16"
                edesc = hq.make_desc("int6", "fp16", n_, k_, 1, 0, 1, True, False, to_dev(eq.codes),
                                     to_dev(eq.scales), None)
            elif name.startswith("w4a8"):
                eq = synth.quantize_mxfp4(np.random.default_rng(0).standard_normal((1, n_, k_)) * 0.02)
                atype = "mxfp8"
                edesc = hq.make_desc("mxfp4", "ue8m0", n_, k_, 1, 32, 1, True, False, to_dev(eq.codes),
                                     to_dev(eq.scales), None)
            else:
                eq, _ = synth.dense_fp8_block(0, 1, n_, k_)
                atype = "fp8"
                edesc = hq.make_desc("fp8", "fp32", n_, k_, 1, 128, 128, True, False, to_dev(eq.codes),
                                     to_dev(eq.scales), None)
            nb = hq.hq_transform_size(edesc)
            ewts = []
            for _ in range(cfg["copies"]):
                w = torch.empty(nb, dtype=torch.uint8, device=dev)
                hq.hq_transform(edesc, w, nb, sh)
                ewts.append(w)
            per = {}
            for m in cfg["ms"]:
                erng = np.random.default_rng(100 + m)
                if atype == "mxfp8":
                    # bf16 activations quantised on the device (MXFP8 codes and exponents)
                    xb = to_dev(synth.to_bf16_bits(erng.standard_normal((m, k_))))
                    xd = torch.empty((m, k_), dtype=torch.uint8, device=dev)
                    xsd = torch.empty((m, k_ // 32), dtype=torch.uint8, device=dev)
                    hq.hq_mxfp8_quantize(m, k_, xb, k_, xd, k_, xsd, k_ // 32, sh)
                    torch.cuda.synchronize()
                    # the quantiser's own time per call (CUDA events, 20 calls)
                    q0, q1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                    q0.record(stream)
                    for _ in range(20):
                        hq.hq_mxfp8_quantize(m, k_, xb, k_, xd, k_, xsd, k_ // 32, sh)
                    q1.record(stream)
                    torch.cuda.synchronize()
                    per_quant = q0.elapsed_time(q1) * 1e-3 / 20
                else:
                    a = synth.make_activations(erng, m, k_, atype)
                    xd = to_dev(a.data)
                    xsd = to_dev(np.ascontiguousarray(a.scales, np.float32)) if a.scales is not None else None
                    per_quant = None
                yd = torch.empty((m, n_), dtype=torch.float16 if atype == "fp16" else torch.bfloat16, device=dev)
                wsd = torch.zeros(max(hq.hq_gemm_workspace_size(edesc, m, atype), 256), dtype=torch.uint8,
                                  device=dev)
                per[m] = {"x": xd, "xs": xsd, "y": yd, "ws": wsd, "quant_s": per_quant}
            extra[name] = {"desc": edesc, "wts": ewts, "atype": atype, "per": per, "cfg": cfg}
            del eq

    def extra_call(key):
        name, m = key
        e = extra[name]
        d = e["per"][m]
        wt = e["wts"][rot["extra"] % len(e["wts"])]
        rot["extra"] += 1
        k_ = e["cfg"]["k"]
        hq.hq_gemm(e["desc"], wt, m, e["atype"], d["x"], k_, d["xs"], d["y"], e["cfg"]["n"], d["ws"],
                   d["ws"].numel(), 0, sh)
        launches["n"] += hq.hq_last_plan()["launches"]

    def gemm(m):
        wt = wts[rot["w"] % W_COPIES]
        i = rot["x"] % X_COPIES
        rot["w"] += 1
        rot["x"] += 1
        hq.hq_gemm(desc, wt, m, "bf16", xs[m][i], K, None, ys[m][i], N, wss[m], wss[m].numel(), 0, sh)
        launches["n"] += hq.hq_last_plan()["launches"]

    def gemm_host(m):
        """One call as a user with host buffers makes it: H2D, GEMM, D2H."""
        xs[m][0].copy_(xh[m].view(torch.int16), non_blocking=True)
        rot["x"] = 0
        gemm(m)
        yh[m].copy_(ys[m][0], non_blocking=True)

    # ---- MoE workload
    moe = None
    if not args.no_moe:
        mq, _, _ = synth.moe_mxfp4(0, 1)
        mdesc = hq.make_desc("mxfp4", "ue8m0", MOE_N, MOE_K, MOE_E, 32, 1, True, False,
                             to_dev(mq.codes), to_dev(mq.scales), None)
        mbytes = hq.hq_transform_size(mdesc)
        mwts = []
        for _ in range(MOE_COPIES):
            mwt = torch.empty(mbytes, dtype=torch.uint8, device=dev)
            hq.hq_transform(mdesc, mwt, mbytes, sh)
            mwts.append(mwt)
        moe = {"desc": mdesc, "wt": mwts, "T": {}}
        # feed-forward block: the gate+up experts above, down experts [E][K][N/2]
        dq, _, _ = synth.moe_mxfp4(1, 1, num_experts=MOE_E, n=MOE_H, k=MOE_N // 2)
        ddesc = hq.make_desc("mxfp4", "ue8m0", MOE_H, MOE_N // 2, MOE_E, 32, 1, True, False,
                             to_dev(dq.codes), to_dev(dq.scales), None)
        dbytes = hq.hq_transform_size(ddesc)
        dwts = []
        for _ in range(MOE_COPIES):
            dwt = torch.empty(dbytes, dtype=torch.uint8, device=dev)
            hq.hq_transform(ddesc, dwt, dbytes, sh)
            dwts.append(dwt)
        moe.update({"ddesc": ddesc, "dwt": dwts})
        del dq
        for t in MOE_T:
            r = synth.make_routing(np.random.default_rng(10 + t), t, MOE_E, MOE_TOPK)
            x = synth.to_bf16_bits(np.random.default_rng(20 + t).standard_normal((t, MOE_K)))
            need = hq.hq_moe_workspace_size(mdesc, t, MOE_TOPK, "bf16")
            touched = np.unique(r.topk_ids).size
            moe["T"][t] = {"ids": to_dev(r.topk_ids.astype(np.int32)), "w": to_dev(r.topk_w.astype(np.float32)),
                           "x": to_dev(x), "y": torch.empty((t, MOE_N), dtype=torch.bfloat16, device=dev),
                           "ws": torch.zeros(need, dtype=torch.uint8, device=dev), "touched": int(touched)}
            fneed = hq.hq_moe_ffn_workspace_size(mdesc, ddesc, t, MOE_TOPK)
            moe["T"][t].update({"fws": torch.zeros(fneed, dtype=torch.uint8, device=dev),
                                "fy": torch.empty((t, MOE_H), dtype=torch.bfloat16, device=dev)})
        del mq

    def moe_call(t):
        d = moe["T"][t]
        mwt = moe["wt"][rot["moe"] % MOE_COPIES]
        rot["moe"] += 1
        hq.hq_moe_gemm(moe["desc"], mwt, t, MOE_TOPK, d["ids"], d["w"], "bf16", d["x"], MOE_K, d["y"], MOE_N,
                       None, None, d["ws"], d["ws"].numel(), 0, sh)
        launches["n"] += hq.hq_last_plan()["launches"]

    def moe_a8_call(t):
        # W4A8-MXFP4: the same experts and routing, bf16 rows quantised to
        # MXFP8 in the gather, block-scaled grouped GEMM
        d = moe["T"][t]
        mwt = moe["wt"][rot["moe"] % MOE_COPIES]
        rot["moe"] += 1
        hq.hq_moe_gemm(moe["desc"], mwt, t, MOE_TOPK, d["ids"], d["w"], "mxfp8", d["x"], MOE_K, d["y"], MOE_N,
                       None, None, d["ws"], d["ws"].numel(), 0, sh)
        launches["n"] += hq.hq_last_plan()["launches"]

    def ffn_call(t):
        d = moe["T"][t]
        i = rot["moe"] % MOE_COPIES
        rot["moe"] += 1
        hq.hq_moe_ffn(moe["desc"], moe["wt"][i], moe["ddesc"], moe["dwt"][i], t, MOE_TOPK, d["ids"], d["w"], "bf16",
                      d["x"], MOE_K, d["fy"], MOE_H, d["fws"], d["fws"].numel(), 0, sh)
        launches["n"] += hq.hq_last_plan()["launches"]

    def timed(fn, arg):
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        fn(arg)
        e1.record(stream)
        return e0, e1

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()
        torch.cuda.synchronize()

    # ---- warm-up
    for _ in range(args.warmup):
        for m in args.m_sweep:
            timed(gemm, m)
        if moe:
            for t in MOE_T:
                timed(moe_call, t)
                timed(moe_a8_call, t)
                timed(ffn_call, t)
        for name, e in extra.items():
            for m in e["cfg"]["ms"]:
                timed(extra_call, (name, m))
    torch.cuda.synchronize()
    st = hq.hq_status_read(wss[args.m_sweep[0]], 0, sh)
    if st != 0:
        raise RuntimeError(f"device status after warm-up: {hq.status_string(st)}")

    # ---- timed steps: every step makes one call per shape; the calls of one
    # shape run back to back (as consecutive layers would), BLOCK calls between
    # two events, so one kernel's launch overlaps the previous one's tail.
    launches["n"] = 0
    per_m = {m: [] for m in args.m_sweep}
    per_t = {t: [] for t in MOE_T}
    per_f = {t: [] for t in MOE_T}
    per_a8 = {t: [] for t in MOE_T}
    per_x = {(name, m): [] for name, e in extra.items() for m in e["cfg"]["ms"]}

    def blocks(fn, arg, n):
        out = []
        done = 0
        while done < n:
            k = min(BLOCK, n - done)
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(k):
                fn(arg)
            e1.record(stream)
            out.append((k, e0, e1))
            done += k
        return out

    with ClockSampler(dev.index, args.clocks_dir) as clk:
        barrier()
        wall0 = time.perf_counter()
        torch.cuda._sleep(HEAD_START_CYCLES)
        events = []
        for m in args.m_sweep:
            events += [("d", m, *b) for b in blocks(gemm, m, args.steps)]
        if moe:
            for t in MOE_T:
                events += [("m", t, *b) for b in blocks(moe_call, t, args.steps)]
            for t in MOE_T:
                events += [("a", t, *b) for b in blocks(moe_a8_call, t, args.steps)]
            for t in MOE_T:
                events += [("f", t, *b) for b in blocks(ffn_call, t, args.steps)]
        for key in per_x:
            events += [("x", key, *b) for b in blocks(extra_call, key, args.steps)]
        barrier()
        wall = time.perf_counter() - wall0
    for kind, key, k, e0, e1 in events:
        {"d": per_m, "m": per_t, "f": per_f, "a": per_a8, "x": per_x}[kind][key].append(
            e0.elapsed_time(e1) * 1e-3 / k)
    gpu_launches = launches["n"]

    # ---- end to end through the C ABI with host buffers (pinned): per step the
    # host clock runs from the first H2D enqueue to the last D2H completion.
    # By default the copies run on their own streams (inputs on one, results on
    # another), ordered against the GEMMs by events, so the copies of one shape
    # overlap the GEMMs of the others, largest M first; --e2e-serial keeps every
    # copy and GEMM in order on the GEMM stream.
    e2e_times = []
    if not args.no_e2e:
        if not args.e2e_serial:
            s_in, s_out = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
            order = sorted(args.m_sweep, reverse=True)
        for step in range(args.warmup + args.steps):
            torch.cuda.synchronize()
            t0 = time.perf_counter()
            if not args.e2e_serial:
                landed = {}
                with torch.cuda.stream(s_in):
                    for m in order:
                        xs[m][0].copy_(xh[m].view(torch.int16), non_blocking=True)
                        landed[m] = torch.cuda.Event()
                        landed[m].record(s_in)
                for m in order:
                    stream.wait_event(landed[m])
                    rot["x"] = 0
                    gemm(m)
                    done = torch.cuda.Event()
                    done.record(stream)
                    s_out.wait_event(done)
                    with torch.cuda.stream(s_out):
                        yh[m].copy_(ys[m][0], non_blocking=True)
                s_out.synchronize()
                stream.synchronize()
            else:
                for m in args.m_sweep:
                    gemm_host(m)
                stream.synchronize()
            if step >= args.warmup:
                e2e_times.append(time.perf_counter() - t0)
    st = hq.hq_status_read(wss[args.m_sweep[0]], 0, sh)
    if st != 0:
        raise RuntimeError(f"device status: {hq.status_string(st)}")

    res = {
        "per_m": {m: statistics.mean(v) for m, v in per_m.items()},
        "per_m_min": {m: min(v) for m, v in per_m.items()},
        "step_s": sum(statistics.mean(v) for v in per_m.values()),
        "e2e_step_s": statistics.mean(e2e_times) if e2e_times else None,
        "clocks": clk.summary(),
        "wall_s": wall,
        "gpu_launches": gpu_launches,
        "plans": {},
    }
    for m in args.m_sweep:
        gemm(m)
        res["plans"][m] = hq.hq_last_plan()
    if moe:
        res["moe"] = {t: statistics.mean(v) for t, v in per_t.items()}
        res["moe_ffn"] = {t: statistics.mean(v) for t, v in per_f.items()}
        res["moe_w4a8"] = {t: statistics.mean(v) for t, v in per_a8.items()}
        res["moe_touched"] = {t: moe["T"][t]["touched"] for t in MOE_T}
    res["extra"] = {}
    for (name, m), v in per_x.items():
        extra_call((name, m))
        res["extra"].setdefault(name, {})[m] = {"s": statistics.mean(v), "s_min": min(v),
                                                "plan": hq.hq_last_plan(),
                                                "quant_s": extra[name]["per"][m]["quant_s"]}
    for name, e in extra.items():
        st = hq.hq_status_read(e["per"][e["cfg"]["ms"][0]]["ws"], 0, sh)
        if st != 0:
            raise RuntimeError(f"device status ({name}): {hq.status_string(st)}")
    torch.cuda.synchronize()
    if not args.no_c1_graph:
        res["c1_graph"] = c1_graph_loop(hq, synth, torch, dev)
    return res


C1_COPIES = 256   # 256 x 0.55 MB transformed weights = 146 MB, more than the 129 MB L2


def c1_graph_loop(hq, synth, torch, dev) -> dict:
    """The small dense case (M = 16, N = K = 1024, symmetric INT4 g128, 573,440
    algorithmic bytes per call): one launch is too short to show an HBM rate, so
    C1_COPIES calls, each on its own weight copy, are captured in one CUDA graph
    and the graph is replayed; every call reads a copy that C1_COPIES - 1 calls
    of other weights have passed over since."""
    import numpy as np
    m, n, k = 16, 1024, 1024
    qw, acts = synth.dense_w4a16_sym(0, m, n, k)

    def to_dev(a):
        a = np.ascontiguousarray(a)
        return torch.from_numpy(a.view(np.int16) if a.dtype == np.uint16 else a).to(dev)

    desc = hq.make_desc("int4", "bf16", n, k, 1, 128, 1, True, False, to_dev(qw.codes), to_dev(qw.scales), None)
    size = hq.hq_transform_size(desc)
    s = torch.cuda.Stream(device=dev)
    wts = []
    for _ in range(C1_COPIES):
        wt = torch.empty(size, dtype=torch.uint8, device=dev)
        hq.hq_transform(desc, wt, size, s.cuda_stream)
        wts.append(wt)
    x = to_dev(acts.data)
    y = torch.empty((m, n), dtype=torch.bfloat16, device=dev)
    ws = torch.zeros(hq.hq_gemm_workspace_size(desc, m, "bf16"), dtype=torch.uint8, device=dev)

    def calls():
        for wt in wts:
            hq.hq_gemm(desc, wt, m, "bf16", x, k, None, y, n, ws, ws.numel(), 0, s.cuda_stream)

    with torch.cuda.stream(s):
        calls()                              # warm-up outside the graph (kernel attributes, tensor maps)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        calls()
    reps = 20
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(s):
        g.replay()
        g.replay()
        e0.record(s)
        for _ in range(reps):
            g.replay()
        e1.record(s)
    torch.cuda.synchronize()
    per_call = e0.elapsed_time(e1) * 1e-3 / (reps * C1_COPIES)
    st = hq.hq_status_read(ws, 0, s.cuda_stream)
    if st != 0:
        raise RuntimeError(f"device status: {hq.status_string(st)}")
    byts = n * k // 2 + n * (k // 128) * 2 + m * k * 2
    return {"workload": "M=16, N=K=1024, symmetric INT4 g128, bf16", "us_per_call": round(per_call * 1e6, 3),
            "GB/s": round(byts / per_call / 1e9, 1), "algorithmic_bytes": byts, "weight_copies": C1_COPIES,
            "timing": f"one CUDA graph of {C1_COPIES} calls replayed {reps} times, CUDA events"}


def reduce_max(value: float, world: int) -> float:
    """The maximum of `value` over all ranks (the slowest replica's time)."""
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-moe", action="store_true", help="skip the MoE sweep")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true", help="skip the host-buffer end-to-end pass")
    ap.add_argument("--no-c1-graph", action="store_true",
                    help="skip the M=16, N=K=1024 case timed as a CUDA graph over many weight copies")
    ap.add_argument("--no-extra", action="store_true",
                    help="skip the INT6 channelwise and FP8 block-scaled configurations")
    ap.add_argument("--e2e-serial", action="store_true",
                    help="end-to-end pass with every copy and GEMM in order on one stream (default: the copies "
                         "on their own streams, overlapping the GEMMs of the other shapes, as a pipelined "
                         "caller issues them)")
    ap.add_argument("--m-sweep", type=str, default=",".join(map(str, M_SWEEP)),
                    help="comma-separated M values of the dense sweep")
    ap.add_argument("--moe-t", type=str, default=",".join(map(str, MOE_T)),
                    help="comma-separated token counts of the MoE sweep")
    ap.add_argument("--clocks-dir", type=str, default=None,
                    help="directory for the nvidia-smi clock samples of the timed region (default: a new "
                         "temporary directory)")
    args = ap.parse_args()
    args.m_sweep = [int(v) for v in args.m_sweep.split(",") if v]
    args.warmup = max(args.warmup, 3)
    MOE_T[:] = [int(v) for v in args.moe_t.split(",") if v]

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", str(rank)))

    if args.impl == "reference":
        if rank != 0:
            return
        # the CPU oracle, as it stands, on a bounded sample per step
        times, flops_tot = [], 0.0
        desc, cores = "", len(os.sched_getaffinity(0))
        for i in range(args.warmup + args.steps):
            v, dt, desc, cores = cpu_oracle_sample(seed=0, rows_cap=64, n_rows=1024)
            if i >= args.warmup:
                times.append(dt)
                flops_tot += v * dt * 1e12
        tot = sum(times)
        val = flops_tot / tot / 1e12
        line = {"impl": "reference", "metric": METRIC, "value": val, "unit": "TFLOP/s", "n_gpus": args.gpus,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * tot / len(times),
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
                "data": "synthetic", "config": {"workload": WORKLOAD, "sample": desc},
                "cpu_baseline": {"value": val, "unit": "TFLOP/s", "cores": cores, "kind": "oracle", "sample": desc},
                "e2e": {"value": val, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
        print(json.dumps(line), flush=True)
        return

    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    res = run_gpu(args, local, world)
    step_s = reduce_max(res["step_s"], world)
    e2e_s = reduce_max(res["e2e_step_s"], world) if res["e2e_step_s"] is not None else None
    if rank != 0:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
        return

    pk = peaks()
    sw = args.m_sweep
    flops_step = sum(dense_flops(m) for m in sw)
    value = world * flops_step / step_s / 1e12
    sweep = []
    for m in sw:
        t = res["per_m"][m]
        by, fl = dense_bytes(m), dense_flops(m)
        roof_t = max(by / (pk["hbm_gbs"] * 1e9), fl / (pk["bf16_tflops"] * 1e12))
        sweep.append({"m": m, "us": round(t * 1e6, 2), "us_min": round(res["per_m_min"][m] * 1e6, 2),
                      "tflops": round(fl / t / 1e12, 2), "gbs": round(by / t / 1e9, 1),
                      "roofline_frac": round(roof_t / t, 3),
                      "bound": "hbm" if by / (pk["hbm_gbs"] * 1e9) >= fl / (pk["bf16_tflops"] * 1e12) else "tensor",
                      "algorithmic_bytes": by, "traffic": ncu_traffic(m), "plan": res["plans"][m]})
    big = max(sw)
    t_big = res["per_m"][big]
    ach = dense_flops(big) / t_big / 1e12
    roofline = {"bound": "tensor", "achieved": round(ach, 2), "peak": pk["bf16_tflops"], "unit": "TFLOP/s",
                "frac": round(ach / pk["bf16_tflops"], 4), "traffic": ncu_traffic(big),
                "kernel": f"WnA16 INT4 kernel (M={big} launch)", "peak_source": pk["source"]}
    dec = 16 if 16 in sw else min(sw)
    t_dec = res["per_m"][dec]
    gbs = dense_bytes(dec) / t_dec / 1e9
    roofline_decode = {"bound": "hbm", "achieved": round(gbs, 1), "peak": pk["hbm_gbs"], "unit": "GB/s",
                       "frac": round(gbs / pk["hbm_gbs"], 4), "traffic": ncu_traffic(dec),
                       "kernel": f"WnA16 INT4 kernel (M={dec} launch)", "peak_source": pk["source"]}
    line = {
        "metric": METRIC, "value": round(value, 3), "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(step_s * 1e3, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": WORKLOAD, "m_sweep": sw,
                   "l2": f"inputs larger than L2: calls rotate over {W_COPIES} weight copies "
                         f"({W_COPIES * 36} MiB) and {X_COPIES} activation copies",
                   "parallelism": "replicas" if world > 1 else "single GPU",
                   "timing": "CUDA events on the launching stream around blocks of 25 back-to-back calls of one shape; value = FLOPs / summed mean per-call times"},
        "sweep": sweep,
        "roofline": roofline,
        "roofline_decode": roofline_decode,
        "e2e": None if e2e_s is None else {
            "value": round(world * flops_step / e2e_s / 1e12, 3), "unit": "TFLOP/s",
            "h2d_bytes_per_step": sum(m * K * 2 for m in sw), "d2h_bytes_per_step": sum(m * N * 2 for m in sw),
            "ms_per_step": round(e2e_s * 1e3, 4),
            "copies": "on the GEMM stream, in order" if args.e2e_serial else "own streams, overlapping the GEMMs"},
        "gpu_launches": res["gpu_launches"],
        "clocks": res["clocks"],
    }
    if "c1_graph" in res:
        c1 = res["c1_graph"]
        c1["roofline_frac"] = round(c1["GB/s"] / pk["hbm_gbs"], 3)
        c1["bound"] = "hbm"
        line["c1_graph"] = c1
    for name, per in res.get("extra", {}).items():
        cfg = EXTRA[name]
        fp8 = name.startswith("c4") or name.startswith("w4a8")
        tc_peak = pk["bf16_tflops"] * (FP8_PER_BF16 if fp8 else 1.0)
        esw = []
        for m in cfg["ms"]:
            t = per[m]["s"]
            by, fl = extra_bytes(name, m), 2 * m * cfg["n"] * cfg["k"]
            t_hbm, t_tc = by / (pk["hbm_gbs"] * 1e9), fl / (tc_peak * 1e12)
            esw.append({"m": m, "us": round(t * 1e6, 2), "us_min": round(per[m]["s_min"] * 1e6, 2),
                        "tflops": round(fl / t / 1e12, 2), "gbs": round(by / t / 1e9, 1),
                        "roofline_frac": round(max(t_hbm, t_tc) / t, 3), "bound": "hbm" if t_hbm >= t_tc else "tensor",
                        "algorithmic_bytes": by, "plan": per[m]["plan"]})
            if per[m].get("quant_s") is not None:
                esw[-1]["mxfp8_quantize_us"] = round(per[m]["quant_s"] * 1e6, 2)
        line[name] = {"workload": cfg["workload"], "sweep": esw,
                      "tensor_peak_tflops": round(tc_peak, 1),
                      "tensor_peak_source": (f"measured bf16 x {FP8_PER_BF16} (nominal fp8:bf16 ratio)" if fp8
                                             else "measured bf16"),
                      "l2": f"calls rotate over {cfg['copies']} weight copies (more than L2)"}
    if "moe" in res:
        msw = []
        for t in MOE_T:
            tt = res["moe"][t]
            fl = 2 * t * MOE_TOPK * MOE_N * MOE_K
            by = res["moe_touched"][t] * (MOE_N * MOE_K // 2 + MOE_N * MOE_K // 32) + t * MOE_K * 2
            roof_t = max(by / (pk["hbm_gbs"] * 1e9), fl / (pk["bf16_tflops"] * 1e12))
            msw.append({"tokens": t, "us": round(tt * 1e6, 2), "tflops": round(fl / tt / 1e12, 2),
                        "gbs": round(by / tt / 1e9, 1), "experts_touched": res["moe_touched"][t],
                        "roofline_frac": round(roof_t / tt, 3)})
        fsw = []
        for t in MOE_T:
            tt = res["moe_ffn"][t]
            fl = 2 * t * MOE_TOPK * (MOE_N * MOE_K + MOE_H * (MOE_N // 2))
            wb = MOE_N * MOE_K + MOE_H * (MOE_N // 2)      # weights per expert (elements)
            by = res["moe_touched"][t] * (wb // 2 + wb // 32) + t * MOE_K * 2
            roof_t = max(by / (pk["hbm_gbs"] * 1e9), fl / (pk["bf16_tflops"] * 1e12))
            fsw.append({"tokens": t, "us": round(tt * 1e6, 2), "tflops": round(fl / tt / 1e12, 2),
                        "gbs": round(by / tt / 1e9, 1), "roofline_frac": round(roof_t / tt, 3)})
        asw = []
        for t in MOE_T:
            tt = res["moe_w4a8"][t]
            fl = 2 * t * MOE_TOPK * MOE_N * MOE_K
            by = res["moe_touched"][t] * (MOE_N * MOE_K // 2 + MOE_N * MOE_K // 32) + t * MOE_K * 2
            roof_t = max(by / (pk["hbm_gbs"] * 1e9), fl / (pk["bf16_tflops"] * FP8_PER_BF16 * 1e12))
            asw.append({"tokens": t, "us": round(tt * 1e6, 2), "tflops": round(fl / tt / 1e12, 2),
                        "gbs": round(by / tt / 1e9, 1), "roofline_frac": round(roof_t / tt, 3)})
        line["moe"] = {"workload": "MoE gate+up, MXFP4 (e2m1 + UE8M0/32) experts, E=128, N=1536, K=2048, top-8, "
                                   "bf16 activations; route + grouped GEMM + combine per call",
                       "sweep": msw,
                       "w4a8_workload": "the same MoE with W4A8-MXFP4: routed bf16 rows quantised to MXFP8 in the "
                                        "gather, block-scaled grouped GEMM (roofline against the fp8 peak, measured "
                                        f"bf16 x {FP8_PER_BF16})",
                       "w4a8_sweep": asw,
                       "ffn_workload": "MoE feed-forward block: the gate+up experts above, SiLU(gate)*up, down "
                                       "experts E=128, N=2048, K=768 (MXFP4), routing-weighted combine per call",
                       "ffn_sweep": fsw}
    if not args.no_cpu_baseline and world >= 1:
        v, dt, desc, cores = cpu_oracle_sample(seed=0, rows_cap=max(M_SWEEP))  # the whole sweep
        line["cpu_baseline"] = {"value": v, "unit": "TFLOP/s", "cores": cores, "kind": "oracle", "sample": desc,
                                "seconds": round(dt, 2)}
    print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
