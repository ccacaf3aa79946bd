/*
 * hq.h — C ABI of the GB300 (sm_103a) quantized GEMM library.
 *
 * The library computes the quantized GEMM of the Humming pages,
 *
 *     Y[M, N] = a(X)[M, K] . dequant(Wq, scales, zeros)[N, K]^T,
 *
 * for low-bit weights against 16-bit or FP8 activations, in a dense form and
 * in an MoE grouped form over routed tokens.  Sources for each operation are
 * cited at its declaration as "<page title>, <section>":
 *   [README]   "Humming" (project README): Key Features, Support Matrix,
 *              Usage Example.
 *   [LAUNCH]   "Humming: Fast, Flexible Kernels for Quantized Inference"
 *              (launch article): the paragraphs on the standard format,
 *              preprocessing, pipelines and tuning controls.
 *   [WIKI]     "Humming" (aiwiki article): sections "Quantization
 *              representation", "Kernel configuration and compilation",
 *              "Device and workload selection", "Precision and deployment
 *              considerations".
 *
 * Conventions for every call:
 *   - All device pointers are owned by the caller.  The library allocates no
 *     device or host memory and keeps no mutable global state except a
 *     read-mostly cache of per-device properties and the fixed device scratch
 *     that hq_gemm_noalloc uses (a module-load array, not an allocation).
 *   - Calls are stream-ordered and asynchronous unless stated otherwise.
 *     Errors the host can detect are returned before anything is launched.
 *   - Errors found on the device (a bounded wait that ran out, an expert id
 *     out of range) are written into a status word at the start of the
 *     caller's workspace; hq_status_read() synchronises and reads it.
 *   - Pointers passed to the GEMM calls must be 16-byte aligned, and row
 *     strides must be multiples of 16 bytes (the TMA rule); otherwise the
 *     call returns HQ_ERR_ALIGNMENT.
 *   - The compute calls need an sm_103 device (B300/GB300); on any other
 *     device they return HQ_ERR_ARCH.  A transformed weight is tied to that
 *     architecture ([WIKI] "Quantization representation": a transformed
 *     layer must match its configured SM version).
 *   - No C++ exception crosses this interface.
 */
#ifndef HQ_H_
#define HQ_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* CUDA stream handle (a cudaStream_t); NULL is the legacy default stream. */
typedef void* hq_stream_t;

typedef enum {
  HQ_OK = 0,
  HQ_ERR_INVALID_ARG = 1,         /* null pointer, bad enum, bad shape, bad group */
  HQ_ERR_UNSUPPORTED = 2,         /* valid combination this build does not implement */
  HQ_ERR_ALIGNMENT = 3,           /* pointer or stride breaks the 16-byte rule */
  HQ_ERR_WORKSPACE_TOO_SMALL = 4, /* dst/workspace smaller than the *_size query */
  HQ_ERR_CUDA = 5,                /* a CUDA runtime call failed */
  HQ_ERR_DEVICE_TIMEOUT = 6,      /* a bounded device-side wait ran out */
  HQ_ERR_ARCH = 7,                /* current device is not sm_103 */
  HQ_ERR_INVALID_VALUE = 8        /* bad data found on the device (NaN scale, expert id out of range) */
} hq_status;

/* Weight element types ([README] Support Matrix; [WIKI] "Quantization representation"). */
typedef enum {
  HQ_W_INT4 = 0,      /* 4-bit integer codes, symmetric (two's complement) or with zero points */
  HQ_W_INT6 = 1,      /* 6-bit integer codes, symmetric or with zero points */
  HQ_W_MXFP4 = 2,     /* OCP MX e2m1 elements with one UE8M0 scale per 32 along K */
  HQ_W_FP8_E4M3 = 3,  /* OCP e4m3 elements with float32 128x128 block scales */
  HQ_W_NVFP4 = 4,     /* e2m1 elements, one e4m3 scale per 16 along K, one float32 scale per expert */
  HQ_W_MXINT4 = 5     /* 4-bit two's complement codes with one UE8M0 scale per 32 along K */
} hq_wtype;

/* Activation types ([README] Support Matrix rows FP16, BF16, FP8 e4m3). */
typedef enum {
  HQ_A_BF16 = 0,
  HQ_A_FP16 = 1,
  HQ_A_FP8_E4M3 = 2,  /* with float32 per-token, per-128-K-group scales */
  HQ_A_MXFP8_E4M3 = 3 /* MXFP8: e4m3 codes with one UE8M0 exponent per 32 along K (from hq_mxfp8_quantize);
                         against MXFP4 weights this is the W4A8-MXFP4 product */
} hq_atype;

/* Scale types ([README] Key Features: BF16, FP16, UE8M0; float32 for FP8 block scales). */
typedef enum {
  HQ_S_BF16 = 0,
  HQ_S_FP16 = 1,
  HQ_S_FP32 = 2,
  HQ_S_UE8M0 = 3,
  HQ_S_E4M3 = 4       /* OCP e4m3 "fn" bytes (NVFP4 block scales) */
} hq_stype;

/*
 * hq_weight_desc — one quantized weight in the standard storage format
 * ([LAUNCH] standard format: weight format, scaling granularity, scale data
 * type and zero points as separate parameters; [WIKI] "Quantization
 * representation": channel, group and block scales, optional zero points, an
 * expert dimension for MoE).
 *
 * Layout of the standard format, all row-major with a leading expert axis E
 * (num_experts = 1 for dense weights), G = K / group_k groups per row
 * (G = 1 when group_k = 0, "channelwise"):
 *   INT4   codes  uint8 [E][N][ceil(K/2)]   element k in byte k/2, low nibble
 *                                            for even k; two's complement when
 *                                            signed_codes, else unsigned 0..15
 *   INT6   codes  uint8 [E][N][3K/4]         little-endian bit stream per row,
 *                                            code k in bits [6k, 6k+6)
 *   MXFP4  codes  uint8 [E][N][K/2]          nibbles as INT4; e2m1 = S.EE.M
 *   FP8    codes  uint8 [E][N][K]            e4m3 "fn" bytes
 *   NVFP4  codes  as MXFP4
 *   MXINT4 codes  as INT4 (two's complement)
 *   scales INT4/INT6: bf16 or fp16 [E][N][G]; MXFP4 and MXINT4: UE8M0 bytes
 *          [E][N][K/32]; NVFP4: e4m3 bytes [E][N][K/16];
 *          FP8: float32 [E][ceil(N/128)][ceil(K/128)]
 *   tensor_scales  NVFP4 only: float32 [E], one secondary scale per expert
 *   zeros  INT4/INT6 with has_zeros only: unsigned codes packed exactly like
 *          that format's codes, [E][N][packed(G)] (INT4: ceil(G/2) bytes,
 *          INT6: 3*ceil(G/4) bytes)
 * Dequantisation: symmetric int  w = q * s;  zero point  w = (q - z) * s;
 * MXFP4  w = e2m1(q) * 2^(E - 127);  FP8  w = e4m3(q) * s_w[n/128][k/128];
 * NVFP4  w = e2m1(q) * e4m3(s[n][k/16]) * g[e];  MXINT4  w = q * 2^(E - 127).
 *
 * Constraints: INT4/INT6 group_k in {0, 32, 64, 128} or a multiple of 128,
 * dividing K; INT6 needs K % 4 == 0; MXFP4 group_k = 32 (K % 32 == 0) and
 * stype UE8M0; FP8 group_k = group_n = 128 and stype FP32; INT stype BF16 or
 * FP16; NVFP4 group_k = 16 (K % 16 == 0) and stype E4M3; MXINT4 group_k =
 * 32 (K % 32 == 0) and stype UE8M0 (signed_codes ignored: always two's
 * complement).  N and K at most 2^28 (HQ_ERR_UNSUPPORTED above, so that tile counts
 * and in-tile offsets fit 32-bit integers).
 * The codes/scales/zeros/tensor_scales pointers are read by hq_transform only; the
 * GEMM calls use the shape fields and ignore the pointers.
 */
typedef struct {
  int32_t wtype;        /* hq_wtype */
  int32_t stype;        /* hq_stype */
  int32_t n;            /* output features N (rows of W) */
  int32_t k;            /* reduction length K */
  int32_t num_experts;  /* E >= 1 */
  int32_t group_k;      /* scale group along K; 0 = one scale per row */
  int32_t group_n;      /* 1, or 128 for FP8 block scales */
  int32_t signed_codes; /* INT without zeros: 1 = two's complement codes */
  int32_t has_zeros;    /* INT only: 1 = zero points present */
  int32_t reserved;
  const void* codes;    /* device pointer, standard format */
  const void* scales;   /* device pointer, standard format */
  const void* zeros;    /* device pointer or NULL */
  const void* tensor_scales; /* NVFP4: device pointer, float32 [E]; else ignored */
} hq_weight_desc;

/* flags for hq_gemm / hq_moe_gemm */
/*
 * HQ_FLAG_BATCH_INVARIANT: a row of Y is bit-identical whatever M is and
 * whatever the other rows of X hold ([WIKI] "Precision and deployment
 * considerations": no Stream-K, and the same MMA configuration at every batch
 * size).  hq_gemm then runs one kernel configuration for every M: WnA16 with
 * 64-token tiles, group scales folded into the 16-bit operand, the K-blocks
 * accumulated by two issuers (even and odd K-blocks, summed in that order),
 * no split-K, stream-K or cluster split; FP8 with 128-row weight tiles and no
 * split-K.  Decode-sized M is slower this way than with the default plans.
 */
#define HQ_FLAG_BATCH_INVARIANT 0x1u

/* Library version (major*10000 + minor*100 + patch). */
int32_t hq_version(void);

/* Static string for a status code; never NULL. */
const char* hq_status_string(int32_t status);

/*
 * hq_transform_size — bytes of the device buffer that hq_transform writes
 * for this weight.  Host only; reads no pointer of the descriptor.
 * Returns HQ_ERR_INVALID_ARG / HQ_ERR_UNSUPPORTED for an invalid descriptor.
 */
hq_status hq_transform_size(const hq_weight_desc* desc, size_t* bytes);

/*
 * hq_transform — repack a standard-format weight into the sm_103 tile layout
 * ([LAUNCH] paragraph on preprocessing: parameters are checked, dimensions
 * padded and the tensors rearranged for the kernel that will read them;
 * [WIKI] "Quantization representation": the layer's transform step turns the
 * weights and their side tensors into the execution layout).
 *
 * desc   standard-format device pointers (codes, scales, zeros)
 * dst    device buffer of at least hq_transform_size() bytes, 256-byte
 *        aligned; owned by the caller; opaque layout (tiles of 128 rows x
 *        128 K, rows and K padded to 128 with zero-valued codes)
 * Synchronous: it waits for the repack kernel on `stream` and returns
 * HQ_ERR_INVALID_VALUE if the weight holds a NaN scale (UE8M0 0xFF) or a
 * NaN e4m3 code; the buffer contents are then unspecified.
 */
hq_status hq_transform(const hq_weight_desc* desc, void* dst, size_t dst_bytes, hq_stream_t stream);

/*
 * hq_untransform — the exact inverse of hq_transform: writes the standard
 * format back into caller buffers codes/scales/zeros (sizes as in the
 * descriptor layout; zeros ignored without has_zeros; for NVFP4 the float32
 * tensor scales [E] are written to `zeros`).  Bit-exact for every
 * input hq_transform accepts.  Asynchronous.
 */
hq_status hq_untransform(const hq_weight_desc* desc, const void* src, void* codes, void* scales,
                         void* zeros, hq_stream_t stream);

/*
 * hq_gemm_workspace_size — bytes of workspace hq_gemm needs for this weight,
 * M and activation type (status word, split-K counters and fp32 partials).
 */
hq_status hq_gemm_workspace_size(const hq_weight_desc* desc, int32_t m, int32_t atype, size_t* bytes);

/*
 * hq_workspace_init — zero a workspace (asynchronous memset on `stream`).
 * A workspace must be initialised once before its first use; every call that
 * completes leaves its counters at zero again, so re-initialising is only
 * needed after HQ_ERR_DEVICE_TIMEOUT.
 */
hq_status hq_workspace_init(void* workspace, size_t bytes, hq_stream_t stream);

/*
 * hq_gemm — dense quantized GEMM  Y = a(X) . dequant(W)^T  ([LAUNCH] WnA16
 * and W8A8 paragraphs; [README] Usage Example layer(inputs)).
 *
 * wdesc     shape of the weight (pointers ignored); num_experts must be 1
 * w_t       hq_transform output for wdesc
 * m         rows of X and Y (0 is a no-op); at most 2^30, with
 *           (m/16 + 1) * ceil(n/128) below 2^31 (HQ_ERR_UNSUPPORTED beyond)
 * atype     hq_atype; INT with group scales needs stype == atype; MXFP4
 *           takes BF16 or MXFP8 (W4A8-MXFP4, [LAUNCH] paragraph "Efficient
 *           W4A8-MXFP4 inference on existing GPUs"; k % 128 == 0); NVFP4 and
 *           MXINT4 need BF16; FP8 weights need FP8 activations
 * x, ldx    X [m][k] row-major, row stride ldx elements (ldx >= k; the row
 *           pitch a multiple of 16 bytes; x 16-byte aligned)
 * x_scales  FP8 activations: float32 [m][ceil(k/128)] row-major (16-byte
 *           aligned).  MXFP8 activations: the UE8M0 bytes [m][k/32]
 *           row-major, as hq_mxfp8_quantize writes them with lde = k/32
 *           (4-byte aligned).  Otherwise ignored.
 *           W4A8-MXFP4 computes Y = sum_k e4m3(x)·2^(Ex-127)·e2m1(w)·2^(Ew-127)
 *           with the block-scaled MMA (one exponent of each operand per 32 K)
 * y, ldy    Y [m][n] row-major, bf16 for BF16/FP8 activations, fp16 for FP16;
 *           y 16-byte aligned, ldy even; with ldy a multiple of 8 the rows are
 *           written by tensor stores, otherwise by plain stores
 * workspace >= hq_gemm_workspace_size() bytes, initialised once
 * flags     HQ_FLAG_* bits
 * Accumulation is fp32 in tensor memory; the output is rounded once.  Errors
 * found on the host (arguments, alignment HQ_ERR_ALIGNMENT, workspace size)
 * return before any launch; device timeouts go to the workspace status word.
 */
hq_status hq_gemm(const hq_weight_desc* wdesc, const void* w_t, int32_t m, int32_t atype,
                  const void* x, int64_t ldx, const void* x_scales, void* y, int64_t ldy,
                  void* workspace, size_t ws_bytes, uint32_t flags, hq_stream_t stream);

/* hq_gemm_noalloc only: clear the scratch's status word and counters first. */
#define HQ_FLAG_NOALLOC_RESET 0x100u

/* Bytes of the fixed device scratch behind hq_gemm_noalloc (8 MiB). */
#define HQ_NOALLOC_SCRATCH_BYTES ((size_t)8 << 20)

/*
 * hq_gemm_noalloc — hq_gemm without a workspace argument.  The Humming pages
 * have no counterpart: this is an interface convenience of this library.
 *
 * For callers that cannot hand the library a workspace: code that holds only
 * its input and output pointers at the call site, with no device allocator
 * it may call there (a plugin or custom-op interface that passes tensors but
 * no scratch, or a runtime that forbids allocation once its memory plan is
 * fixed).  The status word, split-K counters and fp32 partials live instead
 * in one file-scope device array of HQ_NOALLOC_SCRATCH_BYTES per device,
 * zero at module load; no call allocates host or device memory.
 *
 * Arguments are hq_gemm's, less workspace/ws_bytes, plus:
 * flags          hq_gemm's flags, plus HQ_FLAG_NOALLOC_RESET: before the
 *                GEMM, clear the scratch's status word and split-K counters
 *                with cudaMemsetAsync on `stream` (allocates nothing).
 * device_status  optional 4-byte device word; if non-null, the scratch's
 *                status word is copied there on `stream` after the GEMM.
 *                That word is sticky: once a bounded device-side wait has run
 *                out it stays set (and the split-K counters may be stale)
 *                until a call passes HQ_FLAG_NOALLOC_RESET, which is the way
 *                back to correct results after such an error.
 *
 * Set-up: the first call with a given device current looks up the scratch's
 * address (cudaGetSymbolAddress) and caches it, keyed by the device and its
 * CUDA context (a context destroyed and created again, e.g. after
 * cudaDeviceReset, gets a fresh lookup); make that first call before any
 * stream capture.
 * Limit: a problem whose hq_gemm_workspace_size() exceeds
 * HQ_NOALLOC_SCRATCH_BYTES is rejected with HQ_ERR_WORKSPACE_TOO_SMALL before
 * anything is launched; use hq_gemm with a workspace for it.
 * Concurrency: all calls on one device share the scratch.  Calls whose GPU
 * work can overlap (different streams without an ordering event, or several
 * host threads) race on it and give wrong results; serialise them on one
 * stream or order them with events.
 */
hq_status hq_gemm_noalloc(const hq_weight_desc* wdesc, const void* w_t, int32_t m, int32_t atype,
                          const void* x, int64_t ldx, const void* x_scales, void* y, int64_t ldy,
                          uint32_t flags, int32_t* device_status, hq_stream_t stream);

/*
 * hq_moe_workspace_size — workspace for hq_moe_gemm (status word, routing
 * counts and offsets, permutation, per-pair fp32 outputs, and the routed
 * activation rows in expert order: T*topk rows of K bf16, or for
 * HQ_A_MXFP8_E4M3 T*topk rows of K e4m3 bytes and K/32 exponents in the same
 * space).  The size does not depend on atype.
 */
hq_status hq_moe_workspace_size(const hq_weight_desc* desc, int32_t tokens, int32_t topk,
                                int32_t atype, size_t* bytes);

/*
 * hq_moe_gemm — MoE grouped GEMM over routed tokens ([WIKI] "Device and
 * workload selection": indexed input gathered through routing indices,
 * grouped-contiguous execution per expert; [README] MoE GEMM).
 *
 * For flat pair f = t*topk + j with expert e = topk_ids[t][j]:
 *   route   counts, offsets[E+1] (exclusive prefix sum), and the stable
 *           permutation perm[offsets[e] + r] = r-th f (increasing) routed to e
 *   GEMM    Z[f] = a(X[t]) . dequant(W_e)^T     (N outputs)
 *   combine Y[t] = sum_j topk_w[t][j] * Z[t*topk + j], j in increasing order
 *
 * wdesc, w_t   expert weights [E][N][K] and their transform
 * tokens, topk T and top-k; topk_ids int32 [T][topk], topk_w float32 [T][topk]
 * x, ldx       activations [T][k]; y, ldy output [T][n] (bf16 for BF16 acts)
 * atype        HQ_A_BF16, or HQ_A_MXFP8_E4M3 for W4A8-MXFP4 (MXFP4 experts,
 *              k % 128 == 0): x still holds bf16 rows; each routed row is
 *              quantised to MXFP8 as it is gathered (e4m3 elements under one
 *              UE8M0 exponent per 32 along K, the conversion of
 *              hq_mxfp8_quantize) and multiplied on the block-scaled MMA,
 *              so a(X[t]) = mxfp8(X[t]); y is bf16
 * expert_offsets_out  optional int32 [E+1]; perm_out optional int32 [T*topk]
 * Limits (HQ_ERR_UNSUPPORTED beyond): E <= 1024, T*topk <= 2^24 and
 * (T*topk/16 + E + 1) * ceil(n/128) below 2^31.
 * An expert id outside [0, E) makes its pair contribute nothing and sets
 * HQ_ERR_INVALID_VALUE in the workspace status word.
 */
hq_status hq_moe_gemm(const hq_weight_desc* wdesc, const void* w_t, int32_t tokens, int32_t topk,
                      const int32_t* topk_ids, const float* topk_w, int32_t atype, const void* x,
                      int64_t ldx, void* y, int64_t ldy, int32_t* expert_offsets_out,
                      int32_t* perm_out, void* workspace, size_t ws_bytes, uint32_t flags,
                      hq_stream_t stream);

/*
 * hq_moe_ffn_workspace_size — workspace for hq_moe_ffn (status word, routing
 * offsets and permutation, the routed activation rows in expert order, the
 * bf16 gate/up rows and activations of every routed pair, and its fp32
 * weighted down-projection rows).
 */
hq_status hq_moe_ffn_workspace_size(const hq_weight_desc* w13, const hq_weight_desc* w2, int32_t tokens,
                                    int32_t topk, size_t* bytes);

/*
 * hq_moe_ffn — the MoE feed-forward block on routed tokens: the gate+up
 * grouped GEMM, the SiLU-gated product and the down grouped GEMM, then the
 * routing-weighted combine ([LAUNCH] MoE paragraph: the MoE measurement
 * covers the gate-up and the down GEMM).  For pair f = t*topk + j routed to
 * expert e = topk_ids[t][j]:
 *   H[f] = a(X[t]) . dequant(W13_e)^T         (2I outputs: gate, then up)
 *   A[f] = silu(H[f][0, I)) * H[f][I, 2I)      silu(g) = g / (1 + exp(-g))
 *   Y[t] = sum_j topk_w[t][j] * (A[t*topk + j] . dequant(W2_{e})^T)
 * A is held in bf16 (the activation type) between the GEMMs.  When I is a
 * multiple of 128 the gate+up GEMM computes A in its epilogue from the fp32
 * gate and up sums (H is never stored); otherwise H is stored in bf16 and an
 * elementwise kernel computes A from it.
 *
 * w13, w13_t   gate+up experts [E][2I][k] and their transform (I % 8 == 0)
 * w2, w2_t     down experts [E][n][I] and their transform (same E)
 * other arguments as hq_moe_gemm (bf16 activations; x [T][k], y [T][n]).
 * Invalid expert ids and limits: as hq_moe_gemm (the tile bound with the
 * larger of 2I and n).  Asynchronous.
 */
hq_status hq_moe_ffn(const hq_weight_desc* w13, const void* w13_t, const hq_weight_desc* w2, const void* w2_t,
                     int32_t tokens, int32_t topk, const int32_t* topk_ids, const float* topk_w, int32_t atype,
                     const void* x, int64_t ldx, void* y, int64_t ldy, void* workspace, size_t ws_bytes,
                     uint32_t flags, hq_stream_t stream);

/*
 * Grouped MoE input forms ([WIKI] "Device and workload selection": besides
 * the indexed form above, the rows of each expert can be handed over already
 * grouped, either back to back or in per-expert storage with a separate count
 * of valid rows).
 */
#define HQ_MOE_GROUPED_CONTIGUOUS 0 /* rows of expert e: [offsets[e], offsets[e+1]) of X and Y */
#define HQ_MOE_GROUPED_MASKED 1     /* rows of expert e: [e*rows, e*rows + counts[e]) of X and Y */

/*
 * hq_moe_grouped_workspace_size — workspace for hq_moe_grouped_gemm (status
 * word, compacted offsets, tile prefix and each expert's first X row, row map
 * of up to E*rows (masked) or rows (contiguous) entries).
 */
hq_status hq_moe_grouped_workspace_size(const hq_weight_desc* desc, int32_t form, int32_t rows, size_t* bytes);

/*
 * hq_moe_grouped_gemm — the per-expert GEMM on rows already grouped by
 * expert, no routing weights and no combine:
 *   Y[i] = a(X[i]) . dequant(W_e)^T   for every valid row i of expert e.
 *
 * form         HQ_MOE_GROUPED_CONTIGUOUS: expert_rows = int32 offsets[E+1]
 *              (device), nondecreasing, offsets[E] <= rows; X, Y have `rows`
 *              rows.  HQ_MOE_GROUPED_MASKED: expert_rows = int32 counts[E]
 *              (device), 0 <= counts[e] <= rows; X, Y are [E][rows] blocks.
 * expected_rows  rows per expert the caller expects (picks the tile width;
 *              the counts stay on the device); <= 0: derived from `rows`
 * x, ldx       activations (bf16); y, ldy output (bf16), 16-byte aligned rows
 * Limits (HQ_ERR_UNSUPPORTED beyond): E <= 1024, at most 2^24 rows of X (E*rows
 *              when masked), and (those rows/16 + E + 1) * ceil(n/128) below 2^31.
 * Rows outside every expert's range are neither read nor written.  Invalid
 * offsets or counts make that expert contribute nothing and set
 * HQ_ERR_INVALID_VALUE in the workspace status word.  Asynchronous.
 */
hq_status hq_moe_grouped_gemm(const hq_weight_desc* wdesc, const void* w_t, int32_t form, int32_t rows,
                              const int32_t* expert_rows, int32_t expected_rows, int32_t atype, const void* x,
                              int64_t ldx, void* y, int64_t ldy, void* workspace, size_t ws_bytes, uint32_t flags,
                              hq_stream_t stream);

/*
 * hq_selftest_wait_timeout — exercise the device-side failure path shared by
 * every kernel of the library, without a fault: one CTA waits on a barrier
 * that nothing completes, with the library's bounded wait (about 2 s); when
 * the wait runs out it records HQ_ERR_DEVICE_TIMEOUT in the status word of
 * `workspace` (16-byte aligned, at least 256 bytes, initialised) and exits
 * normally.  The context stays usable; hq_status_read reports and clears the
 * word.  For tests of failure detection.  Asynchronous.
 */
hq_status hq_selftest_wait_timeout(void* workspace, hq_stream_t stream);

/*
 * hq_mxfp8_quantize — activations to MXFP8, the activation side of the
 * W4A8-MXFP4 product ([LAUNCH] paragraph "Efficient W4A8-MXFP4 inference on
 * existing GPUs": MXFP4 weights with 8-bit floating-point activations).  OCP
 * MX v1.0 conversion with e4m3 elements, per row and per 32 along K:
 *   E = clamp(floor(log2(max |x|)) - 8 + 127, 0, 254)   (all-zero block: 0)
 *   q = e4m3(x / 2^(E - 127)), round to nearest even, saturating at +-448,
 *       the sign of zero kept
 *
 * m, k       rows and columns (k % 32 == 0; m = 0 is a no-op)
 * x, ldx     bf16 [m][k], row stride ldx elements (x 16-byte aligned, ldx % 8 == 0)
 * q, ldq     e4m3 bytes [m][k] out, row stride ldq bytes (q 8-byte aligned, ldq % 8 == 0)
 * e, lde     UE8M0 bytes [m][k/32] out, row stride lde bytes
 * Non-finite inputs give unspecified codes.  Asynchronous.
 */
hq_status hq_mxfp8_quantize(int32_t m, int32_t k, const void* x, int64_t ldx, void* q, int64_t ldq, void* e,
                            int64_t lde, hq_stream_t stream);

/*
 * hq_status_read — synchronise `stream` and read the device status word of a
 * workspace (HQ_OK when no device-side error was recorded).  With clear != 0
 * the word is reset to HQ_OK afterwards.
 */
hq_status hq_status_read(void* workspace, int32_t clear, hq_stream_t stream, int32_t* device_status);

/*
 * hq_last_plan — the launch plan of the most recent hq_gemm / hq_moe_gemm /
 * hq_moe_ffn / hq_moe_grouped_gemm call on this host thread.  For tests and
 * benchmarks.
 */
typedef struct {
  int32_t bn;          /* tokens per output tile (MMA N for WnA16, M side for FP8) */
  int32_t splits;      /* FP8: split-K factor; WnA16: 1 = whole tiles, 0 = stream-K, 2 = 2-CTA cluster split */
  int32_t grid;        /* CTAs of the GEMM kernel */
  int32_t launches;    /* kernels launched by the call */
  int32_t stages;      /* shared-memory pipeline stages */
  int32_t tile_class;  /* WnA16 tile-width class (0: bn <= 16, 1: <= 64, 2: <= 128, 3: <= 256) */
  int32_t groups;      /* WnA16 dequantiser groups of four warps */
  int32_t x_stages;    /* WnA16 activation ring stages (FP8: 0) */
} hq_plan_info;
hq_status hq_last_plan(hq_plan_info* info);

/*
 * hq_plan_query — the launch plan hq_gemm would choose for this weight, M,
 * activation type and flags on a device with `sms` SMs (1..192) and
 * `smem_optin` bytes of opt-in shared memory per block, computed on the host
 * alone: no device is queried and nothing is launched (for tests and capacity
 * planning).  Validation as hq_gemm's for the shape and types; m = 0 gives an
 * all-zero plan.  The plan of an actual call depends only on these inputs
 * (the device's SM count and opt-in shared memory), so it equals what
 * hq_last_plan reports after hq_gemm on such a device.
 */
hq_status hq_plan_query(const hq_weight_desc* wdesc, int32_t m, int32_t atype, int32_t sms, int64_t smem_optin,
                        uint32_t flags, hq_plan_info* info);

/*
 * hq_moe_plan_query — as hq_plan_query, for hq_moe_gemm with `tokens` tokens
 * routed to `topk` experts each: the expert tile width (tokens per tile, from
 * the mean routed rows per expert), its class, the ring stages and the grid
 * (one CTA per SM); launches = 4 (route, permute, grouped GEMM, combine).
 * Host only.
 */
hq_status hq_moe_plan_query(const hq_weight_desc* wdesc, int32_t tokens, int32_t topk, int32_t sms,
                            int64_t smem_optin, hq_plan_info* info);

/*
 * hq_tuning_reload — read the tuning switches again from the environment
 * (HQ_FORCE_BN, HQ_FORCE_SPLITK, HQ_FORCE_WSTAGES, HQ_FORCE_XSTAGES,
 * HQ_FORCE_X2D: one 2-D activation copy per slab instead of one per stage,
 * HQ_TRACE).  They are otherwise read once, at the first call that plans a
 * launch.  For sweeps and tests that compare plans in one process; call it
 * only while no other call of this library runs.  The pages have no
 * counterpart (their tuning configuration is an object passed to the layer,
 * aiwiki article, section "Configuration model").
 */
void hq_tuning_reload(void);

#ifdef __cplusplus
}
#endif

#endif /* HQ_H_ */
