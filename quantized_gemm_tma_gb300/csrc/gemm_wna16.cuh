// gemm_wna16.cuh — the weight-only-quantized GEMM kernel for sm_103a:
// low-bit weights (INT4 / INT6 / MXFP4 / NVFP4 / MXINT4) against BF16 or FP16
// activations (the MX and NVFP4 formats against BF16 only), in
// a dense form and an MoE grouped form ("WnA16": low-bit weights with 16-bit
// activations — Humming launch article, WnA16 paragraph; MoE GEMM — README
// "Key Features").
//
// Computes D[n, m] = sum_k W[n, k] * X[m, k] per output tile of 128 weight
// rows x BN tokens ("swap AB": the weights are the MMA's M side, so a
// decode-sized M only pads the MMA N dimension, down to 16).
//
// Work: the CTA walks a list of units (tile, K-block range).  A dense problem
// whose tiles fill most SMs twice over runs each tile on a 2-CTA cluster that
// splits K in halves (rank 1's fp32 sums reach rank 0 through distributed
// shared memory).  Dense problems with few tiles are split "stream-K": the
// tiles' K-blocks are dealt out in equal contiguous ranges, one per CTA, and
// a tile covered by several CTAs is finished by the last of them, which sums
// the fp32 partials in CTA order (deterministic).  Larger problems, and MoE,
// take whole tiles round-robin.
//
// Pipeline per CTA (one CTA per SM), warp roles:
//   warps 0-3    epilogue: one TMEM lane quarter each; wait for a unit's
//                accumulators, sum the issuers' partial accumulators, scale,
//                and store Y through shared-memory boxes and tensor stores
//                (or a partial, a cluster exchange, or MoE per-pair rows).
//   warps 4-19   dequantisers.  Two K-blocks per stage (bn <= 64, and dense
//                tiles of 128 tokens): four streams, stream t converting
//                K-block t & 1 of every stage of parity t >> 1 (a whole K-block
//                of its 32 rows per warp); tiles of 128 tokens with one
//                K-block per stage and W4A8 tiles of 256 tokens: four
//                streams, stream t taking every fourth stage.  A stream
//                publishes each K-block whole.  Otherwise (bf16/fp16 tiles of
//                256 tokens) all 16 warps on each K-block, one 32-column
//                chunk each.  A thread owns one weight row (its TMEM lane),
//                turns the packed codes into bf16x2/f16x2 pairs and writes
//                them into an A slot in TMEM with tcgen05.st.
//   warp 20      weight producer: per stage one bulk copy of up to KPS
//                consecutive weight tiles (one contiguous run of the tile
//                layout) into the weight ring, released once the dequantisers
//                have converted the codes.
//   warp 21      activation producer: per stage one tensor copy per 64-column
//                slab (128-byte swizzle) into the activation ring, released
//                by the MMA; MoE rows are gathered by routing index, four
//                rows per tile::gather4 tensor copy, the copies of a stage
//                issued by all 32 lanes.
//   warps 22..   MMA issuers: issuer p takes K-block p of every stage and
//                accumulates into its own TMEM accumulator, so two threads
//                issue tcgen05.mma.kind::f16 concurrently for narrow tiles
//                (one thread issues an M128 K16 MMA only every ~50 cycles).
//
// Every wait is bounded (2 s, or the CTA abort flag); on a timeout the CTA
// records HQ_ERR_DEVICE_TIMEOUT, drains its copies and MMAs, frees TMEM and
// exits.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>

#include "hq_internal.h"
#include "hq_ptx.cuh"

namespace hq {
namespace wna16 {

// Tile-width classes: maximum tokens per tile, K-blocks per stage (= MMA
// issuers), accumulator buffers.  With one K-block per stage the 16
// dequantiser warps share a ring of four A slots of 64 TMEM columns; with two
// they form four streams of four warps, each owning a ring of half slots of
// 32 TMEM columns (one K-block = two half slots).  TMEM: A slots in columns
// [0, acc_col0), accumulators (kDacc x kIss x kBnMax columns) from acc_col0 on.
template <int CLS>
struct Cls;
template <>
struct Cls<0> { static constexpr int kBnMax = 16, kKps = 2, kIss = 2, kDacc = 2; };
template <>
struct Cls<1> { static constexpr int kBnMax = 64, kKps = 2, kIss = 2, kDacc = 2; };
template <>
struct Cls<2> { static constexpr int kBnMax = 128, kKps = 1, kIss = 1, kDacc = 2; };
template <>
struct Cls<3> { static constexpr int kBnMax = 256, kKps = 1, kIss = 1, kDacc = 1; };
// Dense tiles of up to 128 tokens when every CTA runs one tile (2-CTA cluster
// split, or at most one whole tile per CTA): the streams and two issuers of
// the narrow classes, with one accumulator buffer, which a CTA with one unit
// does not need more of (N = K = 8192, M = 128: 24.8 against 27.4 us with
// class 2; class 2 keeps its second buffer for CTAs that run many units).
template <>
struct Cls<4> { static constexpr int kBnMax = 128, kKps = 2, kIss = 2, kDacc = 1; };

constexpr int kEpiWarps = 4;
constexpr int kDqWarps = 16;
constexpr int kASlots = 4;
constexpr int kDqWarp0 = kEpiWarps;                        // first dequant warp
constexpr int kProdWarp = kDqWarp0 + kDqWarps;             // weight producer warp
constexpr int kXProdWarp = kProdWarp + 1;                  // activation producer warp
constexpr int kIssWarp0 = kXProdWarp + 1;                  // first MMA issuer warp
constexpr uint32_t kACol0 = 0;
constexpr uint32_t kTmemCols = 512;

// Streams: half slots per stream; each K-block of a stream fills both and is
// published whole.  (A ring of three for the 16-token class, whose
// accumulators fit in the last 128 columns, let a stream's first half reuse
// the slot of K-block c - 2 instead of waiting for the MMA of K-block c - 1
// when halves were published separately; it measured no faster at M = 16:
// 18.2 against 17.8 us.)
template <int CLS>
constexpr int half_ring() { return 2; }
template <int CLS>
constexpr uint32_t acc_col0() { return static_cast<uint32_t>(4 * 64); }
// A-slot barriers of each kind: four streams' half slots (eight), of which
// the classes without streams use the first four (kASlots)
template <int CLS>
constexpr int a_bars() { return 4 * half_ring<CLS>(); }

template <int CLS>
constexpr int threads() { return 32 * (kIssWarp0 + Cls<CLS>::kIss); }

// Cluster split of a wide tile: rank 1's fp32 sums travel through rank 0's
// ring area as [128 rows][kXchgLd] (4 floats of padding per row keep the
// per-row 16-byte accesses of a warp on distinct banks).
template <int CLS>
constexpr int kXchgLd() { return Cls<CLS>::kBnMax + 4; }
template <int CLS>
constexpr uint32_t xchg_bytes() { return static_cast<uint32_t>(kTileN * kXchgLd<CLS>() * 4); }

// ---------------------------------------------------------------- packed math
template <bool BF16>
__device__ __forceinline__ uint32_t h2sub(uint32_t a, uint32_t b) {
  uint32_t r;
  if constexpr (BF16) {
    __nv_bfloat162 x = __hsub2(*reinterpret_cast<__nv_bfloat162*>(&a), *reinterpret_cast<__nv_bfloat162*>(&b));
    r = *reinterpret_cast<uint32_t*>(&x);
  } else {
    __half2 x = __hsub2(*reinterpret_cast<__half2*>(&a), *reinterpret_cast<__half2*>(&b));
    r = *reinterpret_cast<uint32_t*>(&x);
  }
  return r;
}

template <bool BF16>
__device__ __forceinline__ uint32_t h2mul(uint32_t a, uint32_t b) {
  uint32_t r;
  if constexpr (BF16) {
    __nv_bfloat162 x = __hmul2(*reinterpret_cast<__nv_bfloat162*>(&a), *reinterpret_cast<__nv_bfloat162*>(&b));
    r = *reinterpret_cast<uint32_t*>(&x);
  } else {
    __half2 x = __hmul2(*reinterpret_cast<__half2*>(&a), *reinterpret_cast<__half2*>(&b));
    r = *reinterpret_cast<uint32_t*>(&x);
  }
  return r;
}

template <bool BF16>
__device__ __forceinline__ constexpr uint32_t magic_half() {
  return BF16 ? 0x4300u : 0x6400u;  // 128.0 (bf16) / 1024.0 (fp16): unit spacing in the mantissa
}

template <bool BF16>
__device__ __forceinline__ uint32_t h2fma(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t r;
  if constexpr (BF16) {
    __nv_bfloat162 x = __hfma2(*reinterpret_cast<__nv_bfloat162*>(&a), *reinterpret_cast<__nv_bfloat162*>(&b),
                               *reinterpret_cast<__nv_bfloat162*>(&c));
    r = *reinterpret_cast<uint32_t*>(&x);
  } else {
    __half2 x = __hfma2(*reinterpret_cast<__half2*>(&a), *reinterpret_cast<__half2*>(&b),
                        *reinterpret_cast<__half2*>(&c));
    r = *reinterpret_cast<uint32_t*>(&x);
  }
  return r;
}

__device__ __forceinline__ uint32_t bf16x2_of(float f) {
  const uint32_t b = __bfloat16_as_ushort(__float2bfloat16_rn(f));
  return b | (b << 16);
}
__device__ __forceinline__ uint32_t f16x2_of(float f) {
  const uint32_t b = __half_as_ushort(__float2half_rn(f));
  return b | (b << 16);
}

// INT4 chunk of 32 codes (offset-binary u, zero point z) -> 16 pairs of
// (u - z) * s (SCALE) or of the unscaled difference (channelwise: bf16 gives
// (u - z) * 2^-7, fp16 gives u - z; the row scale follows in the epilogue).
// Word w of a chunk holds the pairs (w & 0x000F000F), (w & 0x00F000F0) and
// the same masks of w >> 8.
//   bf16: a byte b in the low half of a bf16 is the value b * 2^-133 (the
//         subnormal range and the first normal binade line up), so a masked
//         pair is u * 2^-133 or 16u * 2^-133; one FMA by 2^126 (2^122) minus
//         z * 2^-7 gives (u - z) * 2^-7 exactly, and one multiply by s * 2^7
//         rounds the product once, as (u - z) * s would be.
//   fp16: OR with 1024.0 (0x6400) puts u (16u) in the mantissa; one FMA with
//         1 (1/16) minus 1024 + z (64 + z) gives u - z exactly.
// The constants of one (zero point, scale) group, computed once and applied to
// every chunk of the group.
struct Int4Consts {
  uint32_t c_lo, c_hi, a_lo, a_hi, sc;
};
template <bool BF16, bool SCALE>
__device__ __forceinline__ Int4Consts int4_consts(uint32_t z, uint32_t s16) {
  Int4Consts k{};
  if constexpr (BF16) {
    k.c_lo = 0x7E807E80u;  // 2^126
    k.c_hi = 0x7C807C80u;  // 2^122
    // -z * 2^-7 and s * 2^7 are exact in bf16: take the top half of the fp32 bits
    const float zf = __uint_as_float(0x4B000000u | z) - 8388608.f;
    const uint32_t zb = __float_as_uint(zf * -0.0078125f) >> 16;
    k.a_lo = k.a_hi = zb | (zb << 16);
    if constexpr (SCALE) {
      const uint32_t sb = __float_as_uint(__uint_as_float(s16 << 16) * 128.f) >> 16;
      k.sc = sb | (sb << 16);
    }
  } else {
    k.c_lo = 0x3C003C00u;  // 1
    k.c_hi = 0x2C002C00u;  // 1/16
    k.a_lo = f16x2_of(-(1024.f + static_cast<float>(z)));
    k.a_hi = f16x2_of(-(64.f + static_cast<float>(z)));
    if constexpr (SCALE) k.sc = s16 * 0x00010001u;
  }
  return k;
}

template <bool BF16, bool SCALE>
__device__ __forceinline__ void dq_int4_apply(const uint4 q, const Int4Consts& k, uint32_t (&o)[16]) {
  const uint32_t w[4] = {q.x, q.y, q.z, q.w};
  constexpr uint32_t M = BF16 ? 0u : 0x64006400u;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const uint32_t w8 = w[j] >> 8;
    const uint32_t p[4] = {(w[j] & 0x000F000Fu) | M, (w[j] & 0x00F000F0u) | M, (w8 & 0x000F000Fu) | M,
                           (w8 & 0x00F000F0u) | M};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint32_t t = h2fma<BF16>(p[i], (i & 1) ? k.c_hi : k.c_lo, (i & 1) ? k.a_hi : k.a_lo);
      o[4 * j + i] = SCALE ? h2mul<BF16>(t, k.sc) : t;
    }
  }
}

template <bool BF16, bool SCALE>
__device__ __forceinline__ void dq_int4(const uint4 q, uint32_t z, uint32_t s16, uint32_t (&o)[16]) {
  dq_int4_apply<BF16, SCALE>(q, int4_consts<BF16, SCALE>(z, s16), o);
}
template <bool BF16, bool SCALE>
__device__ __forceinline__ void dq_int6(const uint4 q, const uint2 h, uint32_t c2, uint32_t s2, uint32_t (&o)[16]) {
  const uint32_t w[4] = {q.x, q.y, q.z, q.w};
  constexpr uint32_t M = magic_half<BF16>() * 0x00010001u;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const uint32_t H = (j < 2) ? h.x : h.y;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint32_t lo = (w[j] >> (4 * i)) & 0x000F000Fu;
      const uint32_t hi = __funnelshift_r(H, H, 4 * i + 2 * (j & 1)) & 0x00300030u;
      const uint32_t t = h2sub<BF16>(lo | hi | M, c2);
      o[4 * j + i] = SCALE ? h2mul<BF16>(t, s2) : t;
    }
  }
}

// MXFP4 chunk (32 e2m1 codes sharing one UE8M0 exponent E) -> bf16 pairs.
// Each e2m1 code S.EE.M is placed as the bf16 S | EE<<7 | M<<6, which equals
// e2m1 * 2^-126 exactly (EE = 0 gives the bf16 subnormal M * 2^-127); one
// multiply by 2^(E-1) then gives e2m1 * 2^(E-127), exact whenever it is
// representable.  For E > 128 the power is applied in two exact steps.
__device__ __forceinline__ void dq_mxfp4(const uint4 q, uint32_t E, uint32_t (&o)[16]) {
  const uint32_t w[4] = {q.x, q.y, q.z, q.w};
  const bool big = E > 128u;
  const uint32_t s1 = big ? (253u << 7) * 0x00010001u : ((E + 126u) << 7) * 0x00010001u;
  const uint32_t s2 = (E << 7) * 0x00010001u;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const uint32_t x = w[j];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int sm = 6 - 4 * i, ss = 12 - 4 * i;
      const uint32_t mag = (sm >= 0 ? (x << sm) : (x >> (-sm))) & 0x01C001C0u;
      const uint32_t sgn = (x << ss) & 0x80008000u;
      uint32_t v = h2mul<true>(mag | sgn, s1);
      if (big) v = h2mul<true>(v, s2);
      o[4 * j + i] = v;
    }
  }
}

// One e4m3 byte -> the same value as a bf16 pair (exact: 4 significant bits,
// exponents -9..8).
__device__ __forceinline__ uint32_t e4m3_to_bf16x2(uint32_t b) {
  const __half h(__nv_cvt_fp8_to_halfraw(static_cast<__nv_fp8_storage_t>(b), __NV_E4M3));
  const uint32_t x = __float_as_uint(__half2float(h)) >> 16;
  return x | (x << 16);
}

// NVFP4 chunk: 32 e2m1 codes, those of words 0-1 under the e4m3 scale in the
// low byte of s2, those of words 2-3 under the high byte.  The code placed as
// a bf16 (as for MXFP4) is e2m1 * 2^-126; one multiply by 2^126 makes it the
// e2m1 value, a second by the block scale gives e2m1 * s, at most 6
// significant bits, exact.  The tensor scale is applied to the fp32 sums.
__device__ __forceinline__ void dq_nvfp4(const uint4 q, uint32_t s2, uint32_t (&o)[16]) {
  const uint32_t w[4] = {q.x, q.y, q.z, q.w};
  constexpr uint32_t k2p126 = (253u << 7) * 0x00010001u;
  const uint32_t s_lo = e4m3_to_bf16x2(s2 & 0xFFu), s_hi = e4m3_to_bf16x2((s2 >> 8) & 0xFFu);
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const uint32_t x = w[j];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int sm = 6 - 4 * i, ss = 12 - 4 * i;
      const uint32_t mag = (sm >= 0 ? (x << sm) : (x >> (-sm))) & 0x01C001C0u;
      const uint32_t sgn = (x << ss) & 0x80008000u;
      o[4 * j + i] = h2mul<true>(h2mul<true>(mag | sgn, k2p126), j < 2 ? s_lo : s_hi);
    }
  }
}

// MXINT4 chunk: offset-binary codes u = q + 8 under one UE8M0 exponent E.
// The INT4 conversion gives (u - 8) * 2^-7 exactly; a multiply by 2^(E-120)
// gives q * 2^(E-127), exact whenever it is representable.  For E > 247 the
// power is applied in two exact steps (2^127, then 2^(E-247)).
__device__ __forceinline__ void dq_mxint4(const uint4 q, uint32_t E, uint32_t (&o)[16]) {
  dq_int4<true, false>(q, 8u, 0u, o);
  const bool big = E > 247u;
  const uint32_t s1 = big ? (254u << 7) * 0x00010001u : ((E + 7u) << 7) * 0x00010001u;
  const uint32_t s2 = ((E - 120u) << 7) * 0x00010001u;
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    uint32_t v = h2mul<true>(o[i], s1);
    if (big) v = h2mul<true>(v, s2);
    o[i] = v;
  }
}

// MXFP4 chunk for the 8-bit A operand (W4A8): 32 e2m1 codes -> 32 e4m3
// bytes in K order, four per 32-bit word (one TMEM column holds four
// consecutive K).  Every e2m1 value is exact in e4m3; the UE8M0 exponent is
// applied by the block-scaled MMA.  Word j of a chunk holds k = 8j + e, element
// e in nibble e / 2 + 4 (e % 2); the low three bits of a code index a byte
// table of e4m3 magnitudes, bit 3 is the sign (e4m3 bit 7).
__device__ __forceinline__ void dq_mxfp4_e4m3(const uint4 q, uint32_t (&o)[8]) {
  const uint32_t w[4] = {q.x, q.y, q.z, q.w};
  constexpr uint32_t kLo = 0x3C383000u, kHi = 0x4C484440u;  // e4m3 of 0, .5, 1, 1.5 | 2, 3, 4, 6
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const uint32_t a = w[j] & 0x0F0F0F0Fu, b = (w[j] >> 4) & 0x0F0F0F0Fu;  // nibbles 0,2,4,6 | 1,3,5,7
    const uint32_t v[2] = {__byte_perm(a, b, 0x6420u), __byte_perm(a, b, 0x7531u)};  // k = 8j + 0..3 | 4..7
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      uint32_t x = v[h] & 0x07070707u;
      x = (x | (x >> 4)) & 0x00FF00FFu;
      x = (x | (x >> 8)) & 0x0000FFFFu;  // the four table indices as byte selectors
      o[2 * j + h] = __byte_perm(kLo, kHi, x) | ((v[h] & 0x08080808u) << 4);
    }
  }
}

// The same conversion without a table: an e2m1 code placed at e4m3 bits
// [4:2] (sign at bit 7) is the e4m3 number of value x * 2^-6, exactly — e2m1's
// exponent bias is 6 below e4m3's, and e2m1's subnormal 0.5 lands on e4m3's
// subnormal grid.  The 2^6 goes into the sub-block's UE8M0 weight exponent
// (mx_fold, mx_fold_words).
__device__ __forceinline__ void dq_mxfp4_e4m3_s6(const uint4 q, uint32_t (&o)[8]) {
  const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    // nibbles 0,2,4,6 (elements 0,4,1,5) | 1,3,5,7 (elements 2,6,3,7), one per byte
    const uint32_t a = ((w[j] << 2) & 0x1C1C1C1Cu) | ((w[j] << 4) & 0x80808080u);
    const uint32_t b = ((w[j] >> 2) & 0x1C1C1C1Cu) | (w[j] & 0x80808080u);
    o[2 * j] = __byte_perm(a, b, 0x6420u);
    o[2 * j + 1] = __byte_perm(a, b, 0x7531u);
  }
}

// A UE8M0 weight exponent takes the 2^6 of dq_mxfp4_e4m3_s6 when it is at
// most 248; a larger one keeps its value and its sub-block is converted with
// the exact table instead.
__device__ __forceinline__ uint32_t mx_fold(uint32_t e) { return e <= 248u ? e + 6u : e; }

// W4A8 scale factors in the TMEM layout the block-scaled MMA reads
// (scale_vec::1X): for lane l of every lane quarter, column j of a group holds
// the word of row (or token) 32j + l whose byte s is the UE8M0 exponent of
// 32-K sub-block s; the MMA of sub-block s selects byte s by its scale-factor
// ids.  A group of 4 columns covers 128 rows.
//
// mx_fold_words: the weight words with mx_fold applied to every byte; the
// common case (no byte of the warp's words reaches 248) is one add per word.
__device__ __forceinline__ void mx_fold_words(uint32_t (&w)[4]) {
  uint32_t hi = 0;
#pragma unroll
  for (int j = 0; j < 4; ++j) hi |= w[j] & (w[j] << 1) & (w[j] << 2) & (w[j] << 3) & (w[j] << 4);
  if (!__any_sync(0xffffffffu, (hi & 0x80808080u) != 0u)) {
#pragma unroll
    for (int j = 0; j < 4; ++j) w[j] += 0x06060606u;
  } else {
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      uint32_t o = 0;
#pragma unroll
      for (int b = 0; b < 4; ++b) o |= mx_fold((w[j] >> (8 * b)) & 0xFFu) << (8 * b);
      w[j] = o;
    }
  }
}

// The MX instruction descriptor of sub-block s: scale-factor ids for B
// (bits 4-5) and A (bits 29-30).
__device__ __forceinline__ uint32_t mx_idesc_sub(uint32_t idesc, int s) {
  return idesc | (static_cast<uint32_t>(s) << 4) | (static_cast<uint32_t>(s) << 29);
}

// All lanes wait; the outcome is made warp-uniform so that the .sync.aligned
// tcgen05 instructions that follow are always executed by the full warp.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, volatile int* abort) {
  const bool got = dev::mbar_wait(bar, parity, abort);
  return __all_sync(0xffffffffu, got) != 0;
}

// Stage-ring position: slot and phase parity, advanced without division.
struct Ring {
  int s = 0;
  uint32_t ph = 0;
  __device__ __forceinline__ void next(int n) {
    if (++s == n) {
      s = 0;
      ph ^= 1u;
    }
  }
};

// L2 policy of the weight copies: a problem with one row of tiles (MoE: one
// per expert, on average) reads every weight byte once (evict first, keep the
// cache for activations); with several, each weight tile is read again by
// the next row of tiles.
template <bool MOE>
__device__ __forceinline__ uint64_t weight_policy(const GemmParams& p) {
  return p.m_tiles > 1 ? dev::policy_evict_normal() : dev::policy_evict_first();
}

// ---------------------------------------------------------------- work units
struct Unit {
  int e, nt, mt, tile, row0, rows, kb0, kb1;
  int xrow0;  // row of X (the tensor map's outer coordinate) of the unit's first token
};

// The CTA's list of units.  Every role walks the same list.
template <bool MOE>
struct Sched {
  long long it, it_end;  // stream-K: K-block iteration range of this CTA
  int w;                 // whole-tile / MoE: next work index
  int half = 0;          // MoE gated: the up tile of the last gate tile is next
  Unit gate;             // MoE gated: that gate tile's unit

  __device__ __forceinline__ void init(const GemmParams& p) {
    if (!MOE && p.stream_k) {
      it = static_cast<long long>(blockIdx.x) * p.iters / gridDim.x;
      it_end = static_cast<long long>(blockIdx.x + 1) * p.iters / gridDim.x;
    }
    w = blockIdx.x;
  }

  // MoE: s_tabs holds the m-tile prefix [E+1], the row prefix [E+1] and the
  // X row base of each expert [E], back to back in shared memory.
  __device__ __forceinline__ bool next(const GemmParams& p, const int* s_tabs, Unit& u) {
    if constexpr (!MOE) {
      if (p.cluster == 2) {
        // one tile per 2-CTA cluster: rank 0 the lower half of K, rank 1 the rest
        if (w != static_cast<int>(blockIdx.x)) return false;
        u.tile = blockIdx.x >> 1;
        const int kmid = p.k_tiles / 2;
        u.kb0 = (blockIdx.x & 1) ? kmid : 0;
        u.kb1 = (blockIdx.x & 1) ? p.k_tiles : kmid;
        w = -1;
      } else if (p.stream_k) {
        if (it >= it_end) return false;
        u.tile = static_cast<int>(it / p.k_tiles);
        u.kb0 = static_cast<int>(it - static_cast<long long>(u.tile) * p.k_tiles);
        const long long left = it_end - it;
        u.kb1 = (left < p.k_tiles - u.kb0) ? u.kb0 + static_cast<int>(left) : p.k_tiles;
        it += u.kb1 - u.kb0;
      } else {
        if (w >= p.num_tiles) return false;
        u.tile = w;
        u.kb0 = 0;
        u.kb1 = p.k_tiles;
        w += gridDim.x;
      }
      u.nt = u.tile % p.n_tiles;
      u.mt = u.tile / p.n_tiles;
      u.e = 0;
      u.row0 = u.mt * p.bn;
      u.xrow0 = u.row0;
      u.rows = min(p.bn, p.m - u.row0);
      return true;
    } else {
      const int* s_tile_off = s_tabs;
      const int* s_row_off = s_tabs + p.num_experts + 1;
      const int* s_xbase = s_row_off + p.num_experts + 1;
      // gated: work items are (expert, m-tile, gate n-tile), each run as the
      // gate tile and then the up tile I / 128 n-tiles further on
      const bool gated = p.moe_out == kMoeOutGated;
      const int nt_items = gated ? p.n_tiles / 2 : p.n_tiles;
      if (gated && half) {
        u = gate;
        u.nt += nt_items;
        half = 0;
        return true;
      }
      const int total = s_tile_off[p.num_experts] * nt_items;
      if (w >= total) return false;
      const int tile = w / nt_items;
      u.nt = w % nt_items;
      // expert e: last index with tile_off[e] <= tile
      int lo = 0, hi = p.num_experts;  // invariant tile_off[lo] <= tile < tile_off[hi]
      while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (s_tile_off[mid] <= tile) lo = mid; else hi = mid;
      }
      u.e = lo;
      u.mt = tile - s_tile_off[lo];
      u.tile = w;
      u.row0 = s_row_off[lo] + u.mt * p.bn;
      u.rows = min(p.bn, s_row_off[lo + 1] - u.row0);
      u.xrow0 = s_xbase[lo] + u.mt * p.bn;
      u.kb0 = 0;
      u.kb1 = p.k_tiles;
      w += gridDim.x;
      if (gated) {
        gate = u;
        half = 1;
      }
      return true;
    }
  }
};

// Stream-K: the CTAs whose iteration ranges meet tile t are [c_first, c_last];
// CTA c's range starts at floor(c * T / G).
__device__ __forceinline__ int sk_cta_of(long long x, long long T, int G) {
  // largest c with floor(c*T/G) <= x
  return static_cast<int>(((x + 1) * G - 1) / T);
}

// ---------------------------------------------------------------- the kernel
template <int FMT, bool BF16, int CLS, bool MOE>
__global__ void __launch_bounds__(threads<CLS>(), 1)
    wna16_kernel(const __grid_constant__ GemmParams p, const __grid_constant__ CUtensorMap tmap_x,
                 const __grid_constant__ CUtensorMap tmap_y) {
  using C = Cls<CLS>;
  constexpr int KPS = C::kKps, ISS = C::kIss, DACC = C::kDacc, BNMAX = C::kBnMax;
  constexpr int G = KPS;                 // dequantiser groups
  constexpr int WG = kDqWarps / G;        // warps per group
  constexpr int DA = kASlots / G;         // A slots per group
  // W4A8: e4m3 activations (one 128-byte swizzled slab per K-block instead of
  // two of bf16), e4m3 weights in TMEM (32 columns per K-block: A at columns
  // [0, 32) of each 64-column A slot, UE8M0 scale factors in [32, 64)), and
  // block-scaled K32 MMAs.
  constexpr bool A8 = FMT == static_cast<int>(WFmt::MXFP4_A8);
  // Streams: the dequantisers work as four streams of four warps, a whole
  // K-block of its rows per warp, so the four warps sharing a scheduler are at
  // different points of their pipelines instead of in lock step, and the
  // per-K-block waits and hand-offs are paid by four warps instead of sixteen.
  // With two K-blocks per stage stream t takes K-block (t & 1) of every stage
  // of parity (t >> 1); tiles of 128 tokens with one K-block per stage (MoE,
  // and dense problems with several tiles per CTA) and W4A8 tiles of 256
  // tokens (an MMA block twice as fast as bf16's) have stream t take every
  // fourth stage.
  constexpr bool kStream = KPS == 2 || CLS == 2 || (CLS == 3 && A8);
  constexpr int NSTG = kStream ? 4 / KPS : 1;  // stream period in stages
  // A stream publishes its K-block once, both half slots together, on the
  // barrier pair of its first half slot, and the issuer waits and commits
  // once per K-block (the W4A8 scale factors then live in the first half
  // slot only): every wait and commit costs the single issuing thread about
  // 100-300 cycles, more than publishing the first half early gains
  // (N = K = 8192: M = 16 16.3 -> 15.4 us, M = 64 19.8 -> 18.6 us; W4A8
  // M = 4096 263 -> 233 us).
  // The single issuing thread pays for every wait and commit on its own
  // (about 100-300 cycles each against 500 cycles of MMA per W4A8 K-block),
  // so for W4A8 tiles of 256 tokens the stream also waits for the stage's
  // activations before it publishes, and the activation producer refills a
  // slot once the K-block that read it has released its stream's A slot: the
  // issuer waits once and commits once per K-block.  Both parity waits are
  // unambiguous with an activation ring of exactly four stages, one stream
  // period: the producer's on the release (the stream's next K-block needs
  // activations not yet loaded) and the stream's on the activations (below).
  // (The 128-token MoE tiles keep the issuer's activation waits: four 32 KB
  // activation stages would leave their weights half the ring.)
  constexpr bool kXMerge = kStream && CLS == 3;
  constexpr uint32_t kSlabsKb = A8 ? 1u : 2u;  // activation slabs per K-block
  // With streams, issuer p takes K-block p of every stage, i.e. the K-blocks
  // of streams p and 2 + p alternately.
  extern __shared__ uint8_t smem_raw[];
  // 1024-byte aligned base, derived from smem_raw by an offset so that the
  // compiler keeps shared-memory addressing for every access through it
  uint8_t* smem = smem_raw + ((1024u - (dev::smem_u32(smem_raw) & 1023u)) & 1023u);

  const int SW = p.stages;    // weight ring (KPS tiles per stage)
  const int SX = p.x_stages;  // activation ring (2 KPS slabs per stage)
  const int bn = p.bn;
  const uint32_t tile_bytes = p.tile_bytes;
  const uint32_t w_stage = (KPS * tile_bytes + 1023u) & ~1023u;
  const uint32_t slab = static_cast<uint32_t>(bn) * 128u;  // bn rows x 64 K (128 bytes, swizzled)
  const uint32_t x_stage = kSlabsKb * KPS * slab;
  uint8_t* x_st = smem;                    // slabs first: 1024-byte aligned at any bn
  uint8_t* w_st = smem + SX * x_stage;
  // W4A8: the activation exponent words of each weight stage, [stage][K-block
  // of the stage][token], copied in by the weight producer
  uint32_t* e_st = reinterpret_cast<uint32_t*>(w_st + SW * w_stage);
  constexpr uint32_t kETok = BNMAX > 128 ? BNMAX : 128;  // token words per K-block
  constexpr uint32_t kEStage = A8 ? KPS * kETok : 0u;    // words per stage
  uint64_t* w_full = reinterpret_cast<uint64_t*>(e_st + SW * kEStage);
  uint64_t* w_empty = w_full + SW;
  uint64_t* x_full = w_empty + SW;
  uint64_t* x_empty = x_full + SX;
  uint64_t* a_full = x_empty + SX;
  constexpr int NAB = a_bars<CLS>();  // A-slot barriers of each kind
  constexpr int HR = half_ring<CLS>();  // streams: half slots per stream
  static_assert(HR == 2, "a stream publishes whole K-blocks: its ring holds one K-block");
  constexpr uint32_t ACC0 = acc_col0<CLS>();
  uint64_t* a_empty = a_full + NAB;
  uint64_t* acc_full = a_empty + NAB;
  uint64_t* acc_empty = acc_full + DACC;
  uint64_t* tear = acc_empty + DACC;
  uint64_t* red_full = tear + 1;  // cluster split: the peer's half arrived
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(red_full + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  // cluster split, class 0: rank 1's sums [128][16] fp32, 16-byte aligned
  float* s_red = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(tmem_slot) + 16 +
                                          ((16u - (dev::smem_u32(tmem_slot) & 15u)) & 15u));
  // MoE: m-tile prefix [E+1], row prefix [E+1], X row base per expert [E]
  int* s_tabs = reinterpret_cast<int*>(s_red + (CLS == 0 ? kTileN * 16 : 0));
  int* s_tabs_end = s_tabs + (MOE ? 3 * p.num_experts + 2 : 0);
  // dense Y stores: per epilogue warp two staging boxes of 16 tokens x 32 rows
  // (16-bit), 128-byte aligned
  uint16_t* y_stage = reinterpret_cast<uint16_t*>(
      reinterpret_cast<uint8_t*>(s_tabs_end) + ((128u - (dev::smem_u32(s_tabs_end) & 127u)) & 127u));

  const int warp = threadIdx.x >> 5;
  const uint32_t lane = dev::lane_id();
  // A stream skips the stages of the other streams, so a weight ring slot
  // must always carry stages of one residue modulo the stream period (a depth
  // that is a multiple of it); otherwise a stream's parity wait could pass
  // one phase early.  W4A8 256-token tiles also need an activation ring of
  // exactly four stages (above).  The planner never asks for anything else;
  // refuse it before any barrier, TMEM or copy exists.
  if ((kStream && (SW % NSTG)) || (kXMerge && SX != 4)) {
    if (threadIdx.x == 0 && p.status) atomicCAS(p.status, 0, static_cast<int>(HQ_ERR_INVALID_ARG));
    return;
  }
  if (threadIdx.x == 0) HQ_TRACE_CTA(0);

  if (threadIdx.x == 0) {
    for (int s = 0; s < SW; ++s) {
      // W4A8: the tensor copy's arrival, then one per producer lane when its
      // exponent copies have landed
      dev::mbar_init(&w_full[s], A8 ? 33 : 1);
      dev::mbar_init(&w_empty[s], kStream ? 4 * KPS : kDqWarps);  // streams: the warps of those that take it
    }
    for (int s = 0; s < SX; ++s) {
      dev::mbar_init(&x_full[s], 1);
      dev::mbar_init(&x_empty[s], ISS);
    }
    for (int a = 0; a < NAB; ++a) {
      dev::mbar_init(&a_full[a], kStream ? 4 : WG);
      dev::mbar_init(&a_empty[a], 1);
    }
    for (int b = 0; b < DACC; ++b) {
      dev::mbar_init(&acc_full[b], ISS);
      dev::mbar_init(&acc_empty[b], kEpiWarps);
    }
    dev::mbar_init(tear, ISS);
    dev::mbar_init(red_full, kEpiWarps);
    *abort_flag = 0;
    dev::fence_barrier_init();
  }
  if (warp == 0) {
    dev::tmem_alloc(tmem_slot, kTmemCols);
    dev::tmem_relinquish();
  }
  if (warp == kXProdWarp && lane == 0) dev::prefetch_tmap(&tmap_x);
  dev::tc_fence_before();
  __syncthreads();
  dev::tc_fence_after();
  // 2-CTA cluster: the peer's barriers must be initialised before the first
  // remote arrive; the epilogue waits on this before touching the peer
  if (!MOE && p.cluster == 2) dev::cluster_arrive();
  const uint32_t tmem = *tmem_slot;
  [[maybe_unused]] int tr0 = 0;
  if (threadIdx.x == 0) HQ_TRACE(15, tr0, 0);

  // Weights are constant while the GEMM runs (hq_transform is synchronous), so
  // the first ring of weight copies is issued before waiting on the previous
  // grid; activations and everything else only after the wait.
  int n_pre = 0;
  if constexpr (!MOE) {
    if (warp == kProdWarp) {
      if (lane == 0) {
        Sched<MOE> sc;
        sc.init(p);
        const uint64_t pol = weight_policy<MOE>(p);
        Unit u;
        while (n_pre < SW && sc.next(p, s_tabs, u)) {
          const uint8_t* wt = p.tiles + static_cast<uint64_t>(u.nt) * p.k_tiles * tile_bytes;
          for (int kb = u.kb0; kb < u.kb1 && n_pre < SW; kb += KPS, ++n_pre) {
            const uint32_t wbytes = static_cast<uint32_t>(min(KPS, u.kb1 - kb)) * tile_bytes;
            dev::mbar_arrive_expect_tx(&w_full[n_pre], wbytes);
            dev::bulk_load_hint(w_st + n_pre * w_stage, wt + static_cast<uint64_t>(kb) * tile_bytes, wbytes,
                                &w_full[n_pre], pol);
          }
        }
      }
      n_pre = __shfl_sync(0xffffffffu, n_pre, 0);
    }
  }
  dev::grid_dep_wait();
  dev::grid_dep_launch();
  if (threadIdx.x == 0) HQ_TRACE_CTA(1);
  if constexpr (MOE) {
    const int E = p.num_experts;
    for (int i = threadIdx.x; i <= E; i += blockDim.x) {
      s_tabs[i] = p.tile_offsets[i];
      s_tabs[E + 1 + i] = p.expert_offsets[i];
      if (i < E) s_tabs[2 * E + 2 + i] = p.x_base[i];
    }
    __syncthreads();
  }

  if (warp == kProdWarp) {
    // ============================================================ weight producer
    Sched<MOE> sc;
    sc.init(p);
    Ring rg;
    int issued = 0;
    bool ok = true;
    const uint64_t pol = weight_policy<MOE>(p);
    [[maybe_unused]] int tr = 0;
    Unit u;
    while (ok && sc.next(p, s_tabs, u)) {
      const uint8_t* wt = p.tiles + static_cast<uint64_t>(u.e) * p.expert_stride +
                          static_cast<uint64_t>(u.nt) * p.k_tiles * tile_bytes;
      for (int kb = u.kb0; kb < u.kb1; kb += KPS) {
        if (issued >= n_pre) {
          if (!warp_wait(&w_empty[rg.s], rg.ph ^ 1u, abort_flag)) {
            ok = false;
            break;
          }
          if (lane == 0) {
            const uint32_t wbytes = static_cast<uint32_t>(min(KPS, u.kb1 - kb)) * tile_bytes;
            dev::mbar_arrive_expect_tx(&w_full[rg.s], wbytes);
            dev::bulk_load_hint(w_st + rg.s * w_stage, wt + static_cast<uint64_t>(kb) * tile_bytes, wbytes,
                                &w_full[rg.s], pol);
          }
        }
        if constexpr (A8) {
          // one exponent word (four 32-K sub-blocks) per token and K-block of
          // the stage; tokens past the unit get zero exponents (their
          // activation rows are zero-filled and their columns never stored)
          const int cnt = min(KPS, u.kb1 - kb);
          uint32_t* es = e_st + rg.s * kEStage;
#pragma unroll
          for (int i = 0; i < KPS; ++i) {
            if (i < cnt) {
#pragma unroll
              for (int j = 0; j < static_cast<int>(kETok / 32); ++j) {
                const int tok = 32 * j + static_cast<int>(lane);
                const bool in = tok < u.rows;
                const uint8_t* src = p.x_mx + (in ? static_cast<int64_t>(u.xrow0 + tok) * p.ld_mx + (kb + i) * 4 : 0);
                dev::cp_async4(es + i * kETok + tok, src, in ? 4u : 0u);
              }
            }
          }
          dev::cp_async_arrive(&w_full[rg.s]);
        }
        if (lane == 0) HQ_TRACE(0, tr, (1ull << 24) | issued);
        rg.next(SW);
        ++issued;
      }
    }
    if (!ok && lane == 0) dev::raise_error(p.status, abort_flag, HQ_ERR_DEVICE_TIMEOUT);
    // drain: every copy this warp issued has landed before the CTA can exit
    if constexpr (A8) dev::cp_async_wait_all();
    if (lane == 0) {
      for (int s = 0; s < SW && s < issued; ++s) {
        const int last = ((issued - 1 - s) / SW) * SW + s;
        const uint32_t ph = (last / SW) & 1;
        const uint64_t t0 = dev::globaltimer();
        while (!dev::mbar_try_wait(&w_full[s], ph) && dev::globaltimer() - t0 < dev::kWaitTimeoutNs) {
        }
      }
    }
  } else if (warp == kXProdWarp) {
    // ============================================================ activation producer
    Sched<MOE> sc;
    sc.init(p);
    Ring rg;
    int issued = 0;
    bool ok = true;
    [[maybe_unused]] int tr = 0;
    Unit u;
    while (ok && sc.next(p, s_tabs, u)) {
      for (int kb = u.kb0; kb < u.kb1; kb += KPS) {
        const int cnt = min(KPS, u.kb1 - kb);
        if constexpr (kXMerge) {
          // the slot's previous stage, issued - SX, was read by the MMAs of
          // K-block (issued - SX) / 4 of stream (issued - SX) % 4; their
          // completion releases that stream's A slot
          if (issued >= SX) {
            const int prev = issued - SX;
            if (!warp_wait(&a_empty[(prev & 3) * HR], static_cast<uint32_t>(prev >> 2) & 1u, abort_flag)) {
              ok = false;
              break;
            }
          }
        } else if (!warp_wait(&x_empty[rg.s], rg.ph ^ 1u, abort_flag)) {
          ok = false;
          break;
        }
        uint8_t* xs = x_st + rg.s * x_stage;
        if (lane == 0) {
          // one 64-column slab of bn rows per copy, from X row xrow0 on (MoE:
          // the expert's rows stand together in X); columns past K and rows
          // past the end of X are zero-filled by the tensor copy, and rows
          // past the unit belong to other experts: their output columns are
          // never stored
          if (p.x3d) {
            // every slab of the stage in one box (slabs past K read as zeros)
            dev::mbar_arrive_expect_tx(&x_full[rg.s], x_stage);
            dev::tma_load_3d(xs, &tmap_x, &x_full[rg.s], 0, u.xrow0, static_cast<int>(kSlabsKb) * kb);
          } else {
            const int zs = static_cast<int>(kSlabsKb) * cnt;
            dev::mbar_arrive_expect_tx(&x_full[rg.s], static_cast<uint32_t>(zs) * slab);
            for (int z = 0; z < zs; ++z)
              dev::tma_load_2d(xs + z * slab, &tmap_x, &x_full[rg.s], A8 ? (kb + z) * 128 : (2 * kb + z) * 64,
                               u.xrow0);
          }
          HQ_TRACE(3, tr, (16ull << 24) | issued);
        }
        rg.next(SX);
        ++issued;
      }
    }
    if (!ok && lane == 0) dev::raise_error(p.status, abort_flag, HQ_ERR_DEVICE_TIMEOUT);
    if (lane == 0) {
      for (int s = 0; s < SX && s < issued; ++s) {
        const int last = ((issued - 1 - s) / SX) * SX + s;
        const uint32_t ph = (last / SX) & 1;
        const uint64_t t0 = dev::globaltimer();
        while (!dev::mbar_try_wait(&x_full[s], ph) && dev::globaltimer() - t0 < dev::kWaitTimeoutNs) {
        }
      }
    }
  } else if (warp >= kIssWarp0) {
    // ============================================================ MMA issuers
    // One thread per issuer warp walks the schedule, waits and issues.
    const int pidx = warp - kIssWarp0;
    if (lane == 0) {
      Sched<MOE> sc;
      sc.init(p);
      Ring rx;
      uint32_t cu = 0;
      const uint32_t idesc = p.idesc;
      bool ok = true;
      int ui = 0;
      [[maybe_unused]] int tr = 0, ts = 0;
      [[maybe_unused]] uint32_t S = 0;           // streams: stage counter
      [[maybe_unused]] uint32_t cs0 = 0, cs1 = 0;  // two K-blocks per stage: K-blocks taken from streams pidx, 2 + pidx
      Unit u;
      while (ok && sc.next(p, s_tabs, u)) {
        // whole-unit accumulator (double-buffered across units where TMEM allows)
        const int buf = DACC == 1 ? 0 : (ui & 1);
        {
          const uint32_t accph = static_cast<uint32_t>(DACC == 1 ? ui : (ui >> 1)) & 1u;
          if (!dev::mbar_wait(&acc_empty[buf], accph ^ 1u, abort_flag)) {
            ok = false;
            break;
          }
          dev::tc_fence_after();
        }
        bool first = true;
        for (int kb = u.kb0; kb < u.kb1; kb += KPS) {
          const int cnt = min(KPS, u.kb1 - kb);
          // W4A8 256-token tiles: the stream's publish covers the activations
          if (!kXMerge && !dev::mbar_wait(&x_full[rx.s], rx.ph, abort_flag)) {
            ok = false;
            break;
          }
          HQ_TRACE(1 + pidx, tr, (2ull << 24) | ts);
          // stream mode: K-block pidx of this stage comes from stream
          // 2 (S & 1) + pidx (one K-block per stage: stream S & 3), published
          // whole
          const int q = pidx;
          if (kStream && q < cnt) {
            const int t = KPS == 2 ? 2 * static_cast<int>(S & 1u) + q : static_cast<int>(S & 3u);
            // K-blocks taken from stream t so far: one per stream period with
            // one K-block per stage; with two, a unit's last stage may carry
            // one K-block only, so the issuer counts them per stage parity
            const uint32_t cst = KPS == 1 ? S / static_cast<uint32_t>(NSTG) : ((S & 1u) ? cs1 : cs0);
            const uint32_t xs = dev::smem_u32(x_st + rx.s * x_stage) + kSlabsKb * q * slab;
            const uint32_t d_tmem = tmem + ACC0 + static_cast<uint32_t>((buf * ISS + pidx) * BNMAX);
            const bool fresh = first;
            // the stream's K-block cst: one wait, its two half slots' MMAs,
            // one release (descriptor of 32-byte step k: base + 2k)
            const int hs = t * HR;
            if (!dev::mbar_wait(&a_full[hs], cst & 1u, abort_flag)) {
              ok = false;
              break;
            }
            HQ_TRACE(1 + pidx, tr, (3ull << 24) | ts);
            dev::tc_fence_after();
            const uint32_t a_tmem = tmem + kACol0 + static_cast<uint32_t>(hs * 32);
            const uint64_t bd0 = dev::sw128_desc(xs);
            if constexpr (A8) {
#pragma unroll
              for (int c = 0; c < 4; ++c)
                dev::mma_mx_ts(d_tmem, a_tmem + (c >> 1) * 32 + (c & 1) * 8, bd0 + 2u * c, mx_idesc_sub(idesc, c),
                               a_tmem + 16u, a_tmem + 20u, (fresh && c == 0) ? 0u : 1u);
            } else {
#pragma unroll
              for (int c = 0; c < 8; ++c)
                dev::mma_f16_ts(d_tmem, a_tmem + (c >> 2) * 32 + (c & 3) * 8,
                                bd0 + static_cast<uint64_t>(((c >> 2) * slab + (c & 3) * 32) >> 4), idesc,
                                (fresh && c == 0) ? 0u : 1u);
            }
            dev::tc_commit(&a_empty[hs]);
            if (!ok) break;
            if (KPS == 2) {
              if (S & 1u) ++cs1;
              else ++cs0;
            }
            first = false;
          } else if (!kStream && pidx < cnt) {
            const int slot = pidx * DA + static_cast<int>(cu % DA);
            if (!dev::mbar_wait(&a_full[slot], (cu / DA) & 1u, abort_flag)) {
              ok = false;
              break;
            }
            HQ_TRACE(1 + pidx, tr, (3ull << 24) | ts);
            dev::tc_fence_after();
            const uint32_t xs = dev::smem_u32(x_st + rx.s * x_stage) + kSlabsKb * pidx * slab;
            const uint32_t a_tmem = tmem + kACol0 + static_cast<uint32_t>(slot) * 64u;
            const uint32_t d_tmem = tmem + ACC0 + static_cast<uint32_t>((buf * ISS + pidx) * BNMAX);
            const bool fresh = first;
            if constexpr (A8) {
              // 32-K sub-block c: A at slot*64 + 8c, scale factors at slot*64 + 32 (A) and + 36 (B)
#pragma unroll
              for (int c = 0; c < 4; ++c) {
                const uint64_t bdesc = dev::sw128_desc(xs + c * 32);
                dev::mma_mx_ts(d_tmem, a_tmem + c * 8, bdesc, mx_idesc_sub(idesc, c), a_tmem + 32u, a_tmem + 36u,
                               (fresh && c == 0) ? 0u : 1u);
              }
            } else {
#pragma unroll
              for (int kk = 0; kk < 8; ++kk) {
                const uint64_t bdesc = dev::sw128_desc(xs + (kk >> 2) * slab + (kk & 3) * 32);
                dev::mma_f16_ts(d_tmem, a_tmem + kk * 8, bdesc, idesc, (fresh && kk == 0) ? 0u : 1u);
              }
            }
            dev::tc_commit(&a_empty[slot]);
            ++cu;
            first = false;
          }
          if constexpr (!kXMerge) dev::tc_commit(&x_empty[rx.s]);  // else: the A-slot release frees it
          HQ_TRACE(1 + pidx, tr, (4ull << 24) | ts);
          ++ts;
          ++S;
          rx.next(SX);
        }
        if (!ok) break;
        dev::tc_commit(&acc_full[buf]);
        ++ui;
      }
      if (!ok) dev::raise_error(p.status, abort_flag, HQ_ERR_DEVICE_TIMEOUT);
      dev::tc_commit(tear);  // arrives once every MMA this thread issued has completed
    }
  } else if (kStream && warp >= kDqWarp0) {
    // ============================================================ dequantisers (streams)
    const int dw = warp - kDqWarp0;
    const int t = dw >> 2;                  // stream
    // the stages it takes (S % NSTG == sg) and the K-block of them it converts
    const uint32_t sg = KPS == 2 ? static_cast<uint32_t>(t >> 1) : static_cast<uint32_t>(t);
    const int pos = KPS == 2 ? (t & 1) : 0;
    const int quarter = warp & 3;
    const int r = quarter * 32 + static_cast<int>(lane);  // weight row within the tile (TMEM lane)
    // this lane's row in the stream's ring of half slots (32 columns each)
    const uint32_t a_lane =
        tmem + (static_cast<uint32_t>(quarter * 32) << 16) + kACol0 + static_cast<uint32_t>(t * HR * 32);
    // the weight-tile layout fields this role reads per K-block, in registers
    const uint32_t q_scale_off = p.scale_off, q_zero_off = p.zero_off, q_hi_off = p.hi_off;
    const int q_g_kb = p.g_kb, q_group_k = p.group_k, q_has_zeros = p.has_zeros, q_channel = p.channel;
    Sched<MOE> sc;
    sc.init(p);
    Ring rg;
    uint32_t ca = 0;    // this stream's K-blocks so far (one use of each half slot per K-block)
    uint32_t S = 0;     // stage counter
    bool ok = true;
    [[maybe_unused]] int tr = 0, ts = 0;
    const bool trace_me = quarter == 0 && lane == 0;
    uint32_t zrow = 0;
    // INT4 with one scale group per tile (group 128): the group's constants are
    // computed once per K-block (gk_valid), not per chunk
    [[maybe_unused]] Int4Consts gk{};
    [[maybe_unused]] bool gk_valid = false;
    // chunks c0, c0 + 1 (64 K) of this row -> 2 x 16 pairs
    auto convert2 = [&](const uint8_t* wsm, int c0, uint32_t (&o)[2][16]) {
      if constexpr (FMT == static_cast<int>(WFmt::INT4)) {
        if (!q_channel && q_g_kb == 1) {
          if (!gk_valid) {
            const uint32_t s16 = reinterpret_cast<const uint16_t*>(wsm + q_scale_off)[r];
            const uint32_t z = q_has_zeros ? wsm[q_zero_off + r] : zrow;
            gk = int4_consts<BF16, true>(z, s16);
            gk_valid = true;
          }
          const uint4 q0 = *reinterpret_cast<const uint4*>(wsm + (c0 * kTileN + r) * 16);
          const uint4 q1 = *reinterpret_cast<const uint4*>(wsm + ((c0 + 1) * kTileN + r) * 16);
          dq_int4_apply<BF16, true>(q0, gk, o[0]);
          dq_int4_apply<BF16, true>(q1, gk, o[1]);
          return;
        }
      }
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const int c = c0 + i;
        const uint4 q = *reinterpret_cast<const uint4*>(wsm + (c * kTileN + r) * 16);
        uint32_t z = zrow, sc16 = 0;
        if constexpr (FMT == static_cast<int>(WFmt::MXFP4) || FMT == static_cast<int>(WFmt::MXINT4)) {
          sc16 = wsm[q_scale_off + r * 4 + c];
        } else if constexpr (FMT == static_cast<int>(WFmt::NVFP4)) {
          sc16 = reinterpret_cast<const uint16_t*>(wsm + q_scale_off + r * 8)[c];
        } else if (!q_channel) {
          const int g = (q_g_kb > 1) ? (32 * c) / q_group_k : 0;
          sc16 = reinterpret_cast<const uint16_t*>(wsm + q_scale_off)[r * q_g_kb + g];
          if (q_has_zeros) z = wsm[q_zero_off + r * q_g_kb + g];
        }
        if constexpr (FMT == static_cast<int>(WFmt::INT4)) {
          if (q_channel) dq_int4<BF16, false>(q, z, sc16, o[i]);
          else dq_int4<BF16, true>(q, z, sc16, o[i]);
        } else if constexpr (FMT == static_cast<int>(WFmt::INT6)) {
          const uint2 qh = *reinterpret_cast<const uint2*>(wsm + q_hi_off + (c * kTileN + r) * 8);
          const uint32_t c2 = (magic_half<BF16>() + z) * 0x00010001u;
          if (q_channel) dq_int6<BF16, false>(q, qh, c2, 0, o[i]);
          else dq_int6<BF16, true>(q, qh, c2, sc16 * 0x00010001u, o[i]);
        } else if constexpr (FMT == static_cast<int>(WFmt::NVFP4)) {
          dq_nvfp4(q, sc16, o[i]);
        } else if constexpr (FMT == static_cast<int>(WFmt::MXINT4)) {
          dq_mxint4(q, sc16, o[i]);
        } else {
          dq_mxfp4(q, sc16, o[i]);
        }
      }
    };
    // W4A8 256-token tiles: the stage's activations have landed (the issuer
    // waits on this stream's publish only).  With a ring of exactly four
    // activation stages the parity wait is unambiguous: the stream has seen
    // the MMA of its previous K-block (stage S - 4, the slot's previous
    // stage) complete, and stage S + 4 cannot load before this publish.
    auto x_landed = [&]() -> bool {
      if constexpr (!kXMerge) return true;
      return warp_wait(&x_full[S & 3u], (S >> 2) & 1u, abort_flag);
    };
    // issued stores -> visible to the MMA, then count in on the half slot
    auto publish = [&](int hs) {
      dev::tmem_st_wait();
      dev::tc_fence_before();
      __syncwarp();
      if (lane == 0) dev::mbar_arrive(&a_full[hs]);
    };
    Unit u;
    while (ok && sc.next(p, s_tabs, u)) {
      const int n = u.nt * kTileN + r;
      zrow = static_cast<uint32_t>(p.zero_sym);
      if (q_channel && q_has_zeros) zrow = p.row_zero[static_cast<size_t>(u.e) * p.n_pad + n];
      for (int kb = u.kb0; kb < u.kb1; kb += KPS, ++S) {
        const int cnt = min(KPS, u.kb1 - kb);
        if ((S % NSTG) == sg) {
          if (!warp_wait(&w_full[rg.s], rg.ph, abort_flag)) {
            ok = false;
            break;
          }
          if (trace_me) HQ_TRACE(5 + t, tr, (5ull << 24) | ts);
          if (pos < cnt) {
            const uint8_t* wsm = w_st + rg.s * w_stage + pos * tile_bytes;
            // The K-block fills the stream's two half slots (the first half
            // is stored while the second is converted) once the MMAs of the
            // stream's previous K-block have released them, and is published
            // whole on the first slot's barrier pair.
            constexpr int j0 = 0, j1 = 1;
            const uint32_t eph0 = (ca & 1u) ^ 1u;  // release parity of the previous K-block
            if constexpr (A8) {
              // scale exponents of this K-block: weight rows 32j + lane (from
              // the tile; the conversion's 2^6 is folded in when they are
              // stored) and tokens 32j + lane (staged beside the tile by the
              // weight producer)
              constexpr int kXW = static_cast<int>(kETok / 32);  // token words: 4, or 8 for 256 tokens
              uint32_t ww[4], xw[kXW];
              const uint32_t* es = e_st + rg.s * kEStage + pos * kETok;
#pragma unroll
              for (int j = 0; j < 4; ++j) ww[j] = *reinterpret_cast<const uint32_t*>(wsm + q_scale_off + (32 * j + lane) * 4);
#pragma unroll
              for (int j = 0; j < kXW; ++j) xw[j] = es[32 * j + lane];
              mx_fold_words(ww);
              // this lane's row: sub-blocks whose exponent cannot take the fold
              // are converted exactly (rare: a block scale above 2^121); the
              // warp checks for bytes of 248 and up (top five bits set) first
              const uint32_t own = *reinterpret_cast<const uint32_t*>(wsm + q_scale_off + r * 4);
              const bool any_big =
                  __any_sync(0xffffffffu, (own & (own << 1) & (own << 2) & (own << 3) & (own << 4) & 0x80808080u) != 0u);
              uint32_t o8[2][8];
              auto conv8 = [&](int c0) {
#pragma unroll
                for (int i = 0; i < 2; ++i) {
                  const uint4 q = *reinterpret_cast<const uint4*>(wsm + ((c0 + i) * kTileN + r) * 16);
                  dq_mxfp4_e4m3_s6(q, o8[i]);
                  if (any_big && ((own >> (8 * (c0 + i))) & 0xFFu) > 248u) dq_mxfp4_e4m3(q, o8[i]);
                }
              };
              // half slot j: e4m3 codes of two sub-blocks in columns
              // [0, 16), its own copy of the scale factors at 16 (A, 4
              // columns) and 20 (B, 4 columns per 128 tokens)
              auto st_half = [&](int j, bool sf) {
                uint32_t o16[16];
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                  o16[i] = o8[0][i];
                  o16[8 + i] = o8[1][i];
                }
                dev::tmem_st16(a_lane + j * 32, o16);
                if (sf) {
                  dev::tmem_st4(a_lane + j * 32 + 16, ww[0], ww[1], ww[2], ww[3]);
                  dev::tmem_st4(a_lane + j * 32 + 20, xw[0], xw[1], xw[2], xw[3]);
                  if constexpr (kXW == 8) dev::tmem_st4(a_lane + j * 32 + 24, xw[4], xw[5], xw[6], xw[7]);
                }
              };
              conv8(0);
              if (trace_me) HQ_TRACE(5 + t, tr, (12ull << 24) | ts);
              if (!warp_wait(&a_empty[t * HR + j0], eph0, abort_flag) || !x_landed()) {
                ok = false;
                break;
              }
              if (trace_me) HQ_TRACE(5 + t, tr, (6ull << 24) | ts);
              dev::tc_fence_after();
              st_half(j0, true);
              conv8(2);
              __syncwarp();
              if (lane == 0) dev::mbar_arrive(&w_empty[rg.s]);
              st_half(j1, false);  // the MMAs of both halves read the first half's scale factors
              publish(t * HR + j0);
              if (trace_me) HQ_TRACE(5 + t, tr, (7ull << 24) | ts);
              ++ca;
              ++ts;
              rg.next(SW);
              continue;
            }
            uint32_t o[2][16];
            gk_valid = false;
            convert2(wsm, 0, o);
            if (trace_me) HQ_TRACE(5 + t, tr, (12ull << 24) | ts);
            if (!warp_wait(&a_empty[t * HR + j0], eph0, abort_flag) || !x_landed()) {
              ok = false;
              break;
            }
            if (trace_me) HQ_TRACE(5 + t, tr, (6ull << 24) | ts);
            dev::tc_fence_after();
            dev::tmem_st16(a_lane + j0 * 32, o[0]);
            dev::tmem_st16(a_lane + j0 * 32 + 16, o[1]);
            convert2(wsm, 2, o);
            // every lane's codes are consumed: the stage may be refilled
            __syncwarp();
            if (lane == 0) dev::mbar_arrive(&w_empty[rg.s]);
            dev::tmem_st16(a_lane + j1 * 32, o[0]);
            dev::tmem_st16(a_lane + j1 * 32 + 16, o[1]);
            publish(t * HR + j0);
            if (trace_me) HQ_TRACE(5 + t, tr, (7ull << 24) | ts);
            ++ca;
          } else {
            __syncwarp();
            if (lane == 0) dev::mbar_arrive(&w_empty[rg.s]);
          }
        }
        ++ts;
        rg.next(SW);
      }
    }
    dev::tmem_st_wait();  // a wait that gave up may leave stores of this warp in flight
    if (!ok && lane == 0) dev::raise_error(p.status, abort_flag, HQ_ERR_DEVICE_TIMEOUT);
  } else if (warp >= kDqWarp0) {
    // ============================================================ dequantisers
    const int dw = warp - kDqWarp0;
    const int gi = dw / WG;                 // group = position within each stage
    const int quarter = warp & 3;
    const int sub = (dw % WG) >> 2;         // which G chunks of the 4 this warp converts
    const int r = quarter * 32 + static_cast<int>(lane);  // weight row within the tile (TMEM lane)
    const uint32_t a_lane = tmem + (static_cast<uint32_t>(quarter * 32) << 16) + kACol0;
    // the weight-tile layout fields this role reads per K-block, in registers
    const uint32_t q_scale_off = p.scale_off, q_zero_off = p.zero_off, q_hi_off = p.hi_off;
    const int q_g_kb = p.g_kb, q_group_k = p.group_k, q_has_zeros = p.has_zeros, q_channel = p.channel;
    Sched<MOE> sc;
    sc.init(p);
    Ring rg;
    uint32_t ca = 0;
    int pend = -1;  // A slot whose stores were issued but not yet published
    bool ok = true;
    [[maybe_unused]] int tr = 0, ts = 0;
    const bool trace_me = (dw % WG) == 0 && lane == 0;
    Unit u;
    while (ok && sc.next(p, s_tabs, u)) {
      const int n = u.nt * kTileN + r;
      uint32_t zrow = static_cast<uint32_t>(p.zero_sym);
      if (q_channel && q_has_zeros) zrow = p.row_zero[static_cast<size_t>(u.e) * p.n_pad + n];
      for (int kb = u.kb0; kb < u.kb1; kb += KPS) {
        const int cnt = min(KPS, u.kb1 - kb);
        if (!warp_wait(&w_full[rg.s], rg.ph, abort_flag)) {
          ok = false;
          break;
        }
        if (trace_me) HQ_TRACE(5 + gi, tr, (5ull << 24) | ts);
        const bool real = gi < cnt;
        uint4 qc[G];
        uint2 qh[G];
        uint32_t zz[G], ss[G];
        [[maybe_unused]] uint32_t ww[4], xw[4];  // W4A8: weight / token scale exponent words of the K-block
        if (real) {
          const uint8_t* wsm = w_st + rg.s * w_stage + gi * tile_bytes;
          if constexpr (A8) {
            // the scale factors of the K-block are stored by three of the four
            // warps of each lane quarter: sub 0 the weight words (with the
            // conversion's 2^6 folded in), sub 1 and 2 the token words of
            // tokens 0..127 and 128..255 (staged beside the tile by the
            // weight producer)
            const uint32_t* es = e_st + rg.s * kEStage + gi * kETok;
            if (sub == 0) {
#pragma unroll
              for (int j = 0; j < 4; ++j) ww[j] = *reinterpret_cast<const uint32_t*>(wsm + q_scale_off + (32 * j + lane) * 4);
              mx_fold_words(ww);
            } else if (sub == 1 || (sub == 2 && kETok > 128)) {
#pragma unroll
              for (int j = 0; j < 4; ++j) xw[j] = es[32 * (j + 4 * (sub - 1)) + lane];
            }
          }
#pragma unroll
          for (int i = 0; i < G; ++i) {
            const int c = sub * G + i;
            qc[i] = *reinterpret_cast<const uint4*>(wsm + (c * kTileN + r) * 16);
            if constexpr (FMT == static_cast<int>(WFmt::INT6))
              qh[i] = *reinterpret_cast<const uint2*>(wsm + q_hi_off + (c * kTileN + r) * 8);
            if constexpr (FMT == static_cast<int>(WFmt::MXFP4) || FMT == static_cast<int>(WFmt::MXINT4) || A8) {
              ss[i] = wsm[q_scale_off + r * 4 + c];
              zz[i] = 0;
            } else if constexpr (FMT == static_cast<int>(WFmt::NVFP4)) {
              ss[i] = reinterpret_cast<const uint16_t*>(wsm + q_scale_off + r * 8)[c];
              zz[i] = 0;
            } else {
              zz[i] = zrow;
              ss[i] = 0;
              if (!q_channel) {
                const int g = (q_g_kb > 1) ? (32 * c) / q_group_k : 0;
                ss[i] = reinterpret_cast<const uint16_t*>(wsm + q_scale_off)[r * q_g_kb + g];
                if (q_has_zeros) zz[i] = wsm[q_zero_off + r * q_g_kb + g];
              }
            }
          }
        }
        // convert first: the arithmetic covers the previous K-block's TMEM
        // stores still in flight and the MMA that frees this K-block's slot
        uint32_t o[G][16];
        [[maybe_unused]] uint32_t o8[8];
        if (real && A8) {
          // exact table for a sub-block whose exponent cannot take the fold
          dq_mxfp4_e4m3_s6(qc[0], o8);
          if (__any_sync(0xffffffffu, ss[0] > 248u) && ss[0] > 248u) dq_mxfp4_e4m3(qc[0], o8);
        } else if (real) {
#pragma unroll
          for (int i = 0; i < G; ++i) {
            if constexpr (FMT == static_cast<int>(WFmt::INT4)) {
              if (q_channel) dq_int4<BF16, false>(qc[i], zz[i], ss[i], o[i]);
              else dq_int4<BF16, true>(qc[i], zz[i], ss[i], o[i]);
            } else if constexpr (FMT == static_cast<int>(WFmt::INT6)) {
              const uint32_t c2 = (magic_half<BF16>() + zz[i]) * 0x00010001u;
              if (q_channel) dq_int6<BF16, false>(qc[i], qh[i], c2, 0, o[i]);
              else dq_int6<BF16, true>(qc[i], qh[i], c2, ss[i] * 0x00010001u, o[i]);
            } else if constexpr (FMT == static_cast<int>(WFmt::NVFP4)) {
              dq_nvfp4(qc[i], ss[i], o[i]);
            } else if constexpr (FMT == static_cast<int>(WFmt::MXINT4)) {
              dq_mxint4(qc[i], ss[i], o[i]);
            } else {
              dq_mxfp4(qc[i], ss[i], o[i]);
            }
          }
        }
        if (trace_me) HQ_TRACE(5 + gi, tr, (12ull << 24) | ts);
        // The weight stage is free once every lane has consumed its codes: the
        // conversion above used them, so no lane's shared-memory load can still
        // be in flight when lane 0 releases the stage to the next tensor copy.
        __syncwarp();
        if (lane == 0) dev::mbar_arrive(&w_empty[rg.s]);
        // publish the previous K-block's A slot
        if (pend >= 0) {
          dev::tmem_st_wait();
          dev::tc_fence_before();
          __syncwarp();
          if (lane == 0) dev::mbar_arrive(&a_full[pend]);
          pend = -1;
          if (trace_me) HQ_TRACE(5 + gi, tr, (13ull << 24) | ts);
        }
        if (real) {
          const int slot = gi * DA + static_cast<int>(ca % DA);
          if (!warp_wait(&a_empty[slot], ((ca / DA) & 1u) ^ 1u, abort_flag)) {
            ok = false;
            break;
          }
          if (trace_me) HQ_TRACE(5 + gi, tr, (6ull << 24) | ts);
          dev::tc_fence_after();
          if constexpr (A8) {
            // 32-K sub-block `sub` (one per warp, G = 1): e4m3 codes; scale
            // factors A at slot*64 + 32 (4 columns), B at slot*64 + 36 (4 or 8)
            dev::tmem_st8(a_lane + slot * 64 + sub * 8, o8);
            if (sub == 0) dev::tmem_st4(a_lane + slot * 64 + 32, ww[0], ww[1], ww[2], ww[3]);
            else if (sub == 1) dev::tmem_st4(a_lane + slot * 64 + 36, xw[0], xw[1], xw[2], xw[3]);
            else if (sub == 2 && kETok > 128) dev::tmem_st4(a_lane + slot * 64 + 40, xw[0], xw[1], xw[2], xw[3]);
          } else {
#pragma unroll
            for (int i = 0; i < G; ++i) dev::tmem_st16(a_lane + slot * 64 + (sub * G + i) * 16, o[i]);
          }
          pend = slot;
          if (trace_me) HQ_TRACE(5 + gi, tr, (7ull << 24) | ts);
          ++ca;
        }
        ++ts;
        rg.next(SW);
      }
    }
    if (pend >= 0) {
      dev::tmem_st_wait();
      dev::tc_fence_before();
      __syncwarp();
      if (lane == 0) dev::mbar_arrive(&a_full[pend]);
    }
    if (!ok && lane == 0) dev::raise_error(p.status, abort_flag, HQ_ERR_DEVICE_TIMEOUT);
  } else {
    // ============================================================ epilogue
    const int quarter = warp;
    const int r = quarter * 32 + static_cast<int>(lane);
    const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
    Sched<MOE> sc;
    sc.init(p);
    bool ok = true;
    int ui = 0;
    [[maybe_unused]] uint32_t ystg = 0;  // dense: tensor stores of Y issued by this warp
    [[maybe_unused]] int tr = 0;
    const bool trace_me = quarter == 0 && lane == 0;
    // INT4 bf16 operands without a folded scale carry an extra 2^-7
    constexpr float kOpFix = (FMT == static_cast<int>(WFmt::INT4) && BF16) ? 128.f : 1.f;
    const bool gated = MOE && p.moe_out == kMoeOutGated;
    // MoE gated: this CTA's gate sums [BNMAX columns][128 rows] in global
    // memory (L2-resident); a thread reads back only what it wrote
    float* const gbuf = gated ? p.gate_buf + static_cast<size_t>(blockIdx.x) * BNMAX * kTileN + r : nullptr;
    const int half_n = p.n_tiles / 2 * kTileN;  // gated: I, the first up row
    Unit u;
    while (ok && sc.next(p, s_tabs, u)) {
      const int n = u.nt * kTileN + r;
      const bool n_ok = n < p.n;
      // gated units come in pairs: the gate tile (even unit), then its up tile
      const bool gate_half = gated && (ui & 1) == 0;
      float rs = (p.channel && n_ok) ? p.row_scale[static_cast<size_t>(u.e) * p.n_pad + n] * kOpFix : 1.f;
      if constexpr (FMT == static_cast<int>(WFmt::NVFP4)) rs = p.tensor_scale[u.e];  // the per-expert tensor scale
      // gated, up tile: the row scale of the matching gate row
      float rs_gate = rs;
      if (gated && !gate_half && p.channel)
        rs_gate = p.row_scale[static_cast<size_t>(u.e) * p.n_pad + n - half_n] * kOpFix;
      // silu(gate) * up of 16 columns of this row, stored at routed row p,
      // output column n - I (the gate row)
      [[maybe_unused]] auto emit_gated16 = [&](int ch, const float (&g)[16], const float (&v)[16]) {
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const int col = ch * 16 + i;
          if (col < u.rows && n_ok) {
            const float gs = g[i] * rs_gate;
            const float a = gs / (1.f + expf(-gs)) * (v[i] * rs);
            const size_t off = static_cast<size_t>(u.row0 + col) * p.ldy + (n - half_n);
            reinterpret_cast<__nv_bfloat16*>(p.y)[off] = __float2bfloat16_rn(a);
          }
        }
      };
      const bool partial = !MOE && p.stream_k && (u.kb0 > 0 || u.kb1 < p.k_tiles);
      float* pslot = partial ? p.partials + static_cast<size_t>(2 * blockIdx.x + (ui == 0 ? 0 : 1)) * bn * kTileN
                             : nullptr;
      // MoE: the unit's routed pairs and their weights, column 32k + lane in
      // register k of each lane (loaded once per unit, broadcast per column)
      constexpr int kMoeRegs = MOE ? BNMAX / 32 + (BNMAX % 32 ? 1 : 0) : 1;
      [[maybe_unused]] int f_reg[kMoeRegs];
      [[maybe_unused]] float w_reg[kMoeRegs];
      if constexpr (MOE) {
#pragma unroll
        for (int k = 0; k < kMoeRegs; ++k) {
          const int col = 32 * k + static_cast<int>(lane);
          f_reg[k] = col < u.rows ? p.perm[u.row0 + col] : 0;
        }
#pragma unroll
        for (int k = 0; k < kMoeRegs; ++k) {
          const int col = 32 * k + static_cast<int>(lane);
          w_reg[k] = (col < u.rows && p.moe_out == kMoeOutZ) ? p.topk_w[f_reg[k]] : 0.f;
        }
      }
      // columns [16 ch, 16 ch + 16) of this row: partial, MoE row or Y
      auto emit16 = [&](int ch, const float (&vin)[16]) {
        float v[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) v[i] = vin[i];
        if constexpr (CLS == 0 && !MOE) {
          if (p.cluster == 2) {
            dev::cluster_wait();
            // bn <= 16: one chunk.  Rank 1 hands its half-K sums to rank 0
            // through distributed shared memory; rank 0 adds them after its
            // own (K order) and writes Y.
            const uint32_t red_row = dev::smem_u32(s_red + r * 16);
            if (blockIdx.x & 1) {
              const uint32_t dst = dev::map_shared(red_row, 0);
#pragma unroll
              for (int i = 0; i < 4; ++i) dev::st_cluster_v4(dst + 16 * i, v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
              dev::fence_acq_rel_cluster();
              __syncwarp();
              if (lane == 0) dev::mbar_arrive_remote(dev::map_shared(dev::smem_u32(red_full), 0));
              return;
            }
            bool got = dev::mbar_wait_cluster(red_full, 0, abort_flag);
            got = __all_sync(0xffffffffu, got) != 0;
            if (!got) {
              if (lane == 0) dev::raise_error(p.status, abort_flag, HQ_ERR_DEVICE_TIMEOUT);
              return;
            }
#pragma unroll
            for (int i = 0; i < 16; ++i) v[i] += s_red[r * 16 + i];
          }
        }
        if (partial) {
          float4* dst = reinterpret_cast<float4*>(pslot + static_cast<size_t>(r) * bn + ch * 16);
#pragma unroll
          for (int i = 0; i < 4; ++i) dst[i] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
          return;
        }
        if constexpr (!MOE) {
          if (p.y_tma) {
            // tokens 16 ch .. 16 ch + 15 of rows quarter * 32 .. + 31: staged as
            // [token][row] 16-bit, then one tensor store (clipped at M and N)
            uint16_t* buf = y_stage + (quarter * 2 + (ystg & 1)) * (16 * 32);
            if (ystg >= 2 && lane == 0) dev::bulk_wait_read<1>();  // the store two boxes back has read it
            __syncwarp();
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              if constexpr (BF16) buf[i * 32 + lane] = __bfloat16_as_ushort(__float2bfloat16_rn(v[i] * rs));
              else buf[i * 32 + lane] = __half_as_ushort(__float2half_rn(v[i] * rs));
            }
            dev::fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              dev::tma_store_2d(&tmap_y, buf, u.nt * kTileN + quarter * 32, u.row0 + ch * 16);
              dev::bulk_commit();
            }
            ++ystg;
            return;
          }
        }
        [[maybe_unused]] int fr = 0;
        [[maybe_unused]] float wr = 0.f;
        if constexpr (MOE) {
          // columns 16 ch .. 16 ch + 15 live in register ch / 2, lanes 16 (ch & 1) + i
#pragma unroll
          for (int k = 0; k < kMoeRegs; ++k)
            if ((ch >> 1) == k) {
              fr = f_reg[k];
              wr = w_reg[k];
            }
        }
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const int col = ch * 16 + i;
          if constexpr (MOE) {
            const int f = __shfl_sync(0xffffffffu, fr, ((ch & 1) << 4) + i);
            const float wf = __shfl_sync(0xffffffffu, wr, ((ch & 1) << 4) + i);
            if (col < u.rows && n_ok) {
              if (p.moe_out != kMoeOutZ) {  // a 16-bit Y row: f (grouped forms) or the routed position
                const size_t row = p.moe_out == kMoeOutRowMap ? static_cast<size_t>(f)
                                                               : static_cast<size_t>(u.row0 + col);
                const size_t off = row * p.ldy + n;
                if constexpr (BF16) reinterpret_cast<__nv_bfloat16*>(p.y)[off] = __float2bfloat16_rn(v[i] * rs);
                else reinterpret_cast<__half*>(p.y)[off] = __float2half_rn(v[i] * rs);
              } else {
                p.zbuf[static_cast<size_t>(f) * p.n_pad + n] = v[i] * rs * wf;
              }
            }
            continue;
          }
          if (col >= u.rows) continue;
          if (partial) {
            // stored below, 16 at a time
          } else if (n_ok) {
            if constexpr (MOE) {
            } else {
              const size_t off = static_cast<size_t>(u.row0 + col) * p.ldy + n;
              if constexpr (BF16) reinterpret_cast<__nv_bfloat16*>(p.y)[off] = __float2bfloat16_rn(v[i] * rs);
              else reinterpret_cast<__half*>(p.y)[off] = __float2half_rn(v[i] * rs);
            }
          }
        }
      };
      {
        const int buf = DACC == 1 ? 0 : (ui & 1);
        const uint32_t accph = static_cast<uint32_t>(DACC == 1 ? ui : (ui >> 1)) & 1u;
        if (!warp_wait(&acc_full[buf], accph, abort_flag)) {
          ok = false;
          break;
        }
        if (trace_me) HQ_TRACE(9, tr, (8ull << 24) | ui);
        dev::tc_fence_after();
        // issuers that took at least one K-block of the unit; their partial
        // accumulators are summed in issuer order
        const uint32_t parts = (1u << min(ISS, u.kb1 - u.kb0)) - 1u;
        const int is0 = __ffs(parts) - 1;
        const uint32_t acc0 = tmem + lane_base + ACC0 + static_cast<uint32_t>(buf * ISS * BNMAX);
        // the issuers' partial accumulators of 16 columns, summed in issuer order
        auto acc16 = [&](int ch, float (&v)[16]) {
          uint32_t a[16];
          dev::tmem_ld16(acc0 + is0 * BNMAX + ch * 16, a);
          dev::tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(a[i]);
          for (int is = is0 + 1; is < ISS; ++is) {
            if (!((parts >> is) & 1u)) continue;
            dev::tmem_ld16(acc0 + is * BNMAX + ch * 16, a);
            dev::tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 16; ++i) v[i] += __uint_as_float(a[i]);
          }
        };
        bool xchg = false;
        if constexpr (CLS >= 1 && !MOE) xchg = p.cluster == 2;
        if (gate_half) {
          // the gate tile's sums wait in the CTA's gate buffer for its up tile
          for (int ch = 0; ch < (bn >> 4); ++ch) {
            float v[16];
            acc16(ch, v);
#pragma unroll
            for (int i = 0; i < 16; ++i) __stcg(gbuf + (ch * 16 + i) * kTileN, v[i]);
          }
        } else if (gated) {
          // the gate sums of chunk ch + 1 are loaded while chunk ch is combined
          float g[16], gn[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) g[i] = __ldcg(gbuf + i * kTileN);
          for (int ch = 0; ch < (bn >> 4); ++ch) {
            if ((ch + 1) * 16 < bn) {
#pragma unroll
              for (int i = 0; i < 16; ++i) gn[i] = __ldcg(gbuf + ((ch + 1) * 16 + i) * kTileN);
            }
            float v[16];
            acc16(ch, v);
            emit_gated16(ch, g, v);
#pragma unroll
            for (int i = 0; i < 16; ++i) g[i] = gn[i];
          }
        } else if (!xchg) {
          for (int ch = 0; ch < (bn >> 4); ++ch) {
            float v[16];
            acc16(ch, v);
            emit16(ch, v);
          }
        } else if constexpr (CLS >= 1 && !MOE) {
          // Cluster split, wide tiles: rank 1 writes its half-K sums into
          // rank 0's shared memory (rank 0's rings are idle once its MMAs are
          // done, which it signals first); rank 0 adds them after its own and
          // stores Y.
          dev::cluster_wait();
          const uint32_t local = dev::smem_u32(smem);
          if (blockIdx.x & 1) {
            bool got = dev::mbar_wait_cluster(red_full, 0, abort_flag);  // rank 0 is ready
            if (__all_sync(0xffffffffu, got) == 0) {
              ok = false;
              break;
            }
            const uint32_t xremote = dev::map_shared(local, 0);
            for (int ch = 0; ch < (bn >> 4); ++ch) {
              float v[16];
              acc16(ch, v);
              const uint32_t dst = xremote + static_cast<uint32_t>((r * kXchgLd<CLS>() + ch * 16) * 4);
#pragma unroll
              for (int i = 0; i < 4; ++i)
                dev::st_cluster_v4(dst + 16 * i, v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
            }
            dev::fence_acq_rel_cluster();
            __syncwarp();
            if (lane == 0) dev::mbar_arrive_remote(dev::map_shared(dev::smem_u32(red_full), 0));
          } else {
            __syncwarp();
            if (lane == 0) dev::mbar_arrive_remote(dev::map_shared(dev::smem_u32(red_full), 1));
            bool got = dev::mbar_wait_cluster(red_full, 0, abort_flag);  // rank 1's sums arrived
            if (__all_sync(0xffffffffu, got) == 0) {
              ok = false;
              break;
            }
            const float* xbuf = reinterpret_cast<const float*>(smem);
            for (int ch = 0; ch < (bn >> 4); ++ch) {
              float v[16];
              acc16(ch, v);
              const float4* src = reinterpret_cast<const float4*>(xbuf + r * kXchgLd<CLS>() + ch * 16);
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                const float4 t4 = src[i];
                v[4 * i] += t4.x;
                v[4 * i + 1] += t4.y;
                v[4 * i + 2] += t4.z;
                v[4 * i + 3] += t4.w;
              }
              emit16(ch, v);
            }
          }
        }
        dev::tc_fence_before();
        __syncwarp();
        if (lane == 0) dev::mbar_arrive(&acc_empty[buf]);
        if (trace_me) HQ_TRACE(9, tr, (9ull << 24) | ui);
      }
      if (partial) {
        // The last of the tile's CTAs sums every partial in CTA (= K) order.
        // Partials are [slot][row][bn] fp32, one contiguous run per row.  Every
        // lane fences its own stores before lane 0 counts the warp in, and
        // fences again before reading the other CTAs' partials.
        dev::fence_acq_rel_gpu();
        __syncwarp();
        const long long T = p.iters;
        const int Gc = static_cast<int>(gridDim.x);
        const long long x0 = static_cast<long long>(u.tile) * p.k_tiles;
        const int cf = sk_cta_of(x0, T, Gc);
        const int cl = sk_cta_of(x0 + p.k_tiles - 1, T, Gc);
        int* ctr = p.counters + u.tile * 4 + quarter;
        int last = 0;
        if (lane == 0) last = (dev::atom_add_acq_rel_gpu(ctr, 1) == cl - cf) ? 1 : 0;
        last = __shfl_sync(0xffffffffu, last, 0);
        if (last) {
          dev::fence_acq_rel_gpu();
          // 16 columns at a time, contributors summed in CTA order; two
          // contributors' loads are in flight together
          for (int ch = 0; ch * 16 < u.rows; ++ch) {
            float v[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) v[i] = 0.f;
            auto part = [&](int c) {
              const long long begin = static_cast<long long>(c) * T / Gc;
              const int slot = 2 * c + (begin >= x0 ? 0 : 1);
              return reinterpret_cast<const float4*>(p.partials + (static_cast<size_t>(slot) * kTileN + r) * bn + ch * 16);
            };
#pragma unroll 1
            for (int c = cf; c <= cl; c += 2) {
              const bool two = c + 1 <= cl;
              const float4* sa = part(c);
              const float4* sb = part(two ? c + 1 : c);
              float4 ta[4], tb[4];
#pragma unroll
              for (int i = 0; i < 4; ++i) ta[i] = __ldcg(sa + i);
#pragma unroll
              for (int i = 0; i < 4; ++i) tb[i] = __ldcg(sb + i);
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                v[4 * i + 0] = (c == cf) ? ta[i].x : v[4 * i + 0] + ta[i].x;
                v[4 * i + 1] = (c == cf) ? ta[i].y : v[4 * i + 1] + ta[i].y;
                v[4 * i + 2] = (c == cf) ? ta[i].z : v[4 * i + 2] + ta[i].z;
                v[4 * i + 3] = (c == cf) ? ta[i].w : v[4 * i + 3] + ta[i].w;
              }
              if (two) {
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                  v[4 * i + 0] += tb[i].x;
                  v[4 * i + 1] += tb[i].y;
                  v[4 * i + 2] += tb[i].z;
                  v[4 * i + 3] += tb[i].w;
                }
              }
            }
            if (n_ok) {
#pragma unroll
              for (int i = 0; i < 16; ++i) {
                const int col = ch * 16 + i;
                if (col < u.rows) {
                  const size_t off = static_cast<size_t>(u.row0 + col) * p.ldy + n;
                  if constexpr (BF16) reinterpret_cast<__nv_bfloat16*>(p.y)[off] = __float2bfloat16_rn(v[i] * rs);
                  else reinterpret_cast<__half*>(p.y)[off] = __float2half_rn(v[i] * rs);
                }
              }
            }
          }
          if (lane == 0) *ctr = 0;  // ready for the next call
        }
        if (trace_me) HQ_TRACE(9, tr, ((10ull + last) << 24) | ui);
      }
      ++ui;
    }
    // every tensor store of Y has completed before the CTA exits
    if constexpr (!MOE) {
      if (p.y_tma && lane == 0) dev::bulk_wait<0>();
    }
    if (!ok && lane == 0) dev::raise_error(p.status, abort_flag, HQ_ERR_DEVICE_TIMEOUT);
  }

  // ---------------------------------------------------------------- teardown
  dev::tc_fence_before();
  __syncthreads();
  if (threadIdx.x == 0) HQ_TRACE(15, tr0, 1);
  if (threadIdx.x == 0) HQ_TRACE_CTA(2);
  if (warp == 0) {
    if (lane == 0) {
      const uint64_t t0 = dev::globaltimer();
      while (!dev::mbar_try_wait(tear, 0) && dev::globaltimer() - t0 < dev::kWaitTimeoutNs) {
      }
    }
    __syncwarp();
    dev::tc_fence_after();
    dev::tmem_dealloc(tmem, kTmemCols);
    if (lane == 0) HQ_TRACE_CTA(3);
  }
}

// Dynamic shared memory bytes for a launch of class CLS.
template <int CLS>
inline uint32_t smem_bytes(int w_stages, int x_stages, uint32_t tile_bytes, int bn, int num_experts, bool a8) {
  using C = Cls<CLS>;
  const uint32_t w = static_cast<uint32_t>(w_stages) * ((C::kKps * tile_bytes + 1023u) & ~1023u) +
                     (a8 ? static_cast<uint32_t>(w_stages) * C::kKps * 4u * (C::kBnMax > 128 ? C::kBnMax : 128)
                         : 0u);  // W4A8 token exponent words
  const uint32_t x = static_cast<uint32_t>(x_stages) * (a8 ? 1u : 2u) * C::kKps * static_cast<uint32_t>(bn) * 128u;
  const uint32_t bars =
      (2u * w_stages + 2u * x_stages + 2u * a_bars<CLS>() + 2u * C::kDacc + 1u +
       1u) * 8u + 16u;
  const uint32_t scales = CLS == 0 ? 4u * kTileN * 16u : 0u;  // cluster split exchange of class 0
  const uint32_t moe = num_experts ? 4u * (3u * num_experts + 2u) : 0u;
  const uint32_t ystage = num_experts == 0 ? kEpiWarps * 2u * 16u * 32u * 2u + 128u : 0u;  // dense Y boxes
  return w + x + bars + scales + moe + ystage + 1024u /* alignment slack */;
}

}  // namespace wna16
}  // namespace hq
