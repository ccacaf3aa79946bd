"""MoE routing and grouped GEMM (oracle; test infrastructure only).

What is computed (aiwiki Humming article, section "Device and workload
selection": the indexed path gathers input rows through routing indices,
grouped-contiguous execution places each expert's rows together; README
"Key Features": MoE GEMM is supported next to the dense GEMM):

routing  For topk_ids [T, topk] over E experts, with flat pair index
         f = t*topk + j:
           counts[e]  = #{f : id(f) = e}
           offsets    = exclusive prefix sum of counts, length E + 1
           perm[offsets[e] + r] = the r-th flat index (in increasing f) with
                        id(f) = e   (a stable counting sort by expert)
GEMM     Z[f, :] = X[t, :] . W_{id(f)}^T          (the gate+up GEMM)
combine  Y[t, :] = sum_j topk_w[t, j] * Z[t*topk + j, :]
         (the routing-weighted sum per token; no activation function)

Feed-forward block (launch article, MoE paragraph: gate-up and down GEMMs
measured together), for pair f = t*topk + j routed to expert e:
         H[f] = X[t] . W13_e^T            (2I outputs: gate rows first, then up)
         A[f] = silu(H[f, :I]) * H[f, I:],  silu(g) = g / (1 + exp(-g))
         Y[t] = sum_j topk_w[t, j] * A[t*topk + j] . W2_e^T
         (H and A held in bf16, the activation type, between the GEMMs)

Grouped forms (same section: rows arrive already grouped per expert, either
back to back or in per-expert storage with a count of valid rows):
         Y[i, :] = X[i, :] . W_e^T for every row i in expert e's range; the
         ranges are [offsets[e], offsets[e+1]) (contiguous) or
         [e*rows, e*rows + counts[e]) (masked); other rows are not defined.
"""
from __future__ import annotations

import numpy as np


def moe_route(topk_ids: np.ndarray, num_experts: int):
    """Counting sort of routed pairs by expert; returns (counts, offsets, perm)."""
    ids = np.asarray(topk_ids, dtype=np.int64).reshape(-1)
    counts = np.zeros(num_experts, dtype=np.int64)
    for f in range(ids.size):                      # histogram
        counts[ids[f]] += 1
    offsets = np.zeros(num_experts + 1, dtype=np.int64)
    for e in range(num_experts):                   # exclusive prefix sum
        offsets[e + 1] = offsets[e] + counts[e]
    fill = offsets[:-1].copy()
    perm = np.zeros(ids.size, dtype=np.int64)
    for f in range(ids.size):                      # stable scatter in flat order
        perm[fill[ids[f]]] = f
        fill[ids[f]] += 1
    return counts, offsets, perm


def moe_gemm(a: np.ndarray, topk_ids: np.ndarray, topk_w: np.ndarray, w) -> np.ndarray:
    """Y [T, N] float64 from activations a [T, K], routing, and expert weights.

    ``w`` is either a float array [E, N, K] or a callable e -> [N, K] (so that
    only the experts that receive tokens are dequantised).
    """
    a = np.asarray(a, dtype=np.float64)
    ids = np.asarray(topk_ids, dtype=np.int64)
    tw = np.asarray(topk_w, dtype=np.float32).astype(np.float64)
    get = w if callable(w) else (lambda e, _w=np.asarray(w, dtype=np.float64): _w[e])
    t_count, topk = ids.shape
    y = None
    for e in np.unique(ids):
        t_idx, j_idx = np.nonzero(ids == e)
        z = a[t_idx] @ np.asarray(get(int(e)), dtype=np.float64).T   # Z rows routed to e
        if y is None:
            y = np.zeros((t_count, z.shape[1]), dtype=np.float64)
        np.add.at(y, t_idx, tw[t_idx, j_idx][:, None] * z)
    return y


def moe_reference(qw, acts, routing) -> np.ndarray:
    """Convenience wrapper over ``synth`` containers."""
    from .gemm import dequantize, decode_activations

    ts = getattr(qw, "tensor_scale", None)

    def expert(e):
        z = None if qw.zeros is None else qw.zeros[e:e + 1]
        return dequantize(qw.wtype, qw.n, qw.k, qw.codes[e:e + 1], qw.scales[e:e + 1], z,
                          qw.group_k, qw.signed, qw.stype, 1, None if ts is None else ts[e:e + 1])[0]
    return moe_gemm(decode_activations(acts.atype, acts.data, acts.scales),
                    routing.topk_ids, routing.topk_w, expert)


def moe_grouped_ranges(form: str, expert_rows, num_experts: int, rows: int):
    """Row range [start, stop) of every expert for a grouped form."""
    v = np.asarray(expert_rows, dtype=np.int64)
    if form == "contiguous":
        return [(int(v[e]), int(v[e + 1])) for e in range(num_experts)]
    if form == "masked":
        return [(e * rows, e * rows + int(v[e])) for e in range(num_experts)]
    raise ValueError(form)


def moe_grouped_gemm(a: np.ndarray, form: str, expert_rows, rows: int, w) -> dict:
    """{row index: Y row (float64)} for every valid row of a grouped form.

    ``a`` holds the activation rows of the whole X buffer (``rows`` rows for
    contiguous, E*rows for masked); ``w`` as in ``moe_gemm``.
    """
    a = np.asarray(a, dtype=np.float64)
    get = w if callable(w) else (lambda e, _w=np.asarray(w, dtype=np.float64): _w[e])
    n_exp = len(expert_rows) - 1 if form == "contiguous" else len(expert_rows)
    out = {}
    for e, (lo, hi) in enumerate(moe_grouped_ranges(form, expert_rows, n_exp, rows)):
        if hi <= lo:
            continue
        z = a[lo:hi] @ np.asarray(get(e), dtype=np.float64).T
        for i in range(lo, hi):
            out[i] = z[i - lo]
    return out


def silu(g):
    """g * sigmoid(g) in float64."""
    g = np.asarray(g, dtype=np.float64)
    return g / (1.0 + np.exp(-g))


def round_bf16(x):
    """Round float64 values to the nearest bf16 value (ties to even), directly
    from float64 (8 significant bits; the normal range)."""
    x = np.asarray(x, dtype=np.float64)
    m, e = np.frexp(x)                       # x = m * 2^e, 0.5 <= |m| < 1
    return np.ldexp(np.round(m * 256.0) / 256.0, e)   # np.round: half to even


def moe_ffn(a: np.ndarray, topk_ids: np.ndarray, topk_w: np.ndarray, w13, w2,
            intermediate: str | None = "bf16") -> np.ndarray:
    """Y [T, n] float64 of the MoE feed-forward block.

    ``w13`` gives [2I, K] per expert (gate rows, then up rows) and ``w2``
    [n, I], each as a float array [E, ...] or a callable e -> array.
    ``intermediate="bf16"`` stores H and A in the activation type between the
    GEMMs (rounded to bf16, the reading the library follows); ``None`` keeps
    them exact.
    """
    rnd = round_bf16 if intermediate == "bf16" else (lambda v: v)
    a = np.asarray(a, dtype=np.float64)
    ids = np.asarray(topk_ids, dtype=np.int64)
    tw = np.asarray(topk_w, dtype=np.float32).astype(np.float64)
    get13 = w13 if callable(w13) else (lambda e, _w=np.asarray(w13, dtype=np.float64): _w[e])
    get2 = w2 if callable(w2) else (lambda e, _w=np.asarray(w2, dtype=np.float64): _w[e])
    t_count, topk = ids.shape
    y = None
    for e in np.unique(ids):
        t_idx, j_idx = np.nonzero(ids == e)
        w_gu = np.asarray(get13(int(e)), dtype=np.float64)
        inter = w_gu.shape[0] // 2
        h = rnd(a[t_idx] @ w_gu.T)                              # [pairs of e, 2I]
        act = rnd(silu(h[:, :inter]) * h[:, inter:])
        z = act @ np.asarray(get2(int(e)), dtype=np.float64).T  # [pairs of e, n]
        if y is None:
            y = np.zeros((t_count, z.shape[1]), dtype=np.float64)
        np.add.at(y, t_idx, tw[t_idx, j_idx][:, None] * z)
    return y
