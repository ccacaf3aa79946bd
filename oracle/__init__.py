"""CPU oracle for the quantized GEMM hot path — TEST INFRASTRUCTURE ONLY.

This package is a plain, slow, obviously correct restatement of what the
quantized GEMM computes:

    Y[M, N] = a(X)[M, K] . dequant(Wq, scales, zeros)[N, K]^T

for the weight formats named in the Humming pages (README "Support Matrix";
launch article on the standard format; aiwiki article, section "Quantization
representation"), dense and MoE-grouped.  It decodes the standard storage
format bit by bit, dequantises to real values and multiplies in float64.

It shares no code with the CUDA library (``quantized_gemm_tma_gb300``) and
neither imports the other.  Only ``tests/``, ``__graft_entry__.smoke()`` and
the ``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import
it; the product path never calls it.

Modules:
    formats  decoders of the storage formats (int4, int6, e2m1, UE8M0, e4m3,
             bf16, fp16), each from its bit-field definition
    gemm     dequantisation (int4, int6, mxfp4, fp8 blocks, nvfp4, mxint4)
             and the dense GEMM
    moe      routing (count, prefix sum, stable permutation) and the MoE
             grouped GEMM with the routing-weighted combine; the grouped
             (contiguous / masked) input forms; the feed-forward block
             (gate+up, SiLU-gated product, down, combine)
    w4a8     MXFP8 quantisation of the activations (OCP MX conversion,
             e4m3 elements) and the W4A8-MXFP4 product

Parity status: every function here is pinned by ``tests/test_oracle_*.py``
against values fixed outside the oracle (library casts, published format
tables, hand-worked cases, exact integer and rational arithmetic, invariants);
none is "parity unpinned".
"""
from . import formats, gemm, moe, w4a8  # noqa: F401
from .gemm import dequantize, gemm_dense, decode_activations  # noqa: F401
from .moe import moe_route, moe_gemm, moe_grouped_gemm, moe_ffn  # noqa: F401
