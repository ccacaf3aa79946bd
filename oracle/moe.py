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

    def expert(e):
        z = None if qw.zeros is None else qw.zeros[e:e + 1]
        return dequantize(qw.wtype, qw.n, qw.k, qw.codes[e:e + 1], qw.scales[e:e + 1], z,
                          qw.group_k, qw.signed, qw.stype, 1)[0]
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
