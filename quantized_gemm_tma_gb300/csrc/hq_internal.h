// hq_internal.h — the sm_103 tile layout of transformed weights and the
// parameter blocks shared by the host API (hq_api.cpp) and the kernels.
//
// Transformed weight buffer (output of hq_transform):
//
//   [ header: 256 bytes ]
//   [ tiles:  E x n_tiles x k_tiles tiles of tile_bytes, ordered (e, nt, kt)
//             so that one CTA streams contiguous memory along K ]
//   [ row region (channelwise INT): fp32 scale [E][n_pad], u8 zero [E][n_pad] ]
//   [ block region (FP8): fp32 block scales [E][n_tiles][k_tiles] ]
//   [ tensor region (NVFP4): fp32 tensor scale [E] ]
//
// A tile covers 128 weight rows (n) x 128 reduction columns (k).  Rows and K
// are padded to multiples of 128 with codes that decode to zero.
//
// Inside a tile (all parts 16-byte aligned, one bulk copy per tile):
//   4-bit formats (INT4 offset-binary u = q+8 for symmetric, MXFP4 e2m1):
//     codes [chunk c = 0..3][row r = 0..127][16 bytes]; chunk c holds k in
//     [32c, 32c+32) of row r as four 32-bit words; word j holds k = 32c+8j+e,
//     e = 0..7, element e in nibble (e/2) + 4*(e%2).  So (word >> 4i) &
//     0x000F000F yields elements 2i (low half) and 2i+1 (high half): one
//     bf16x2 / f16x2 pair of the MMA A operand, which keeps K pairs packed in
//     one 32-bit TMEM column.
//   INT6 (u = q+32 offset-binary for symmetric): low nibbles as the 4-bit
//     layout (8192 bytes), then the top two bits [chunk][row][8 bytes]: two
//     32-bit words per chunk, word h serving low words 2h and 2h+1; the top
//     bits of element e of low word w sit at bits (4 + 16*(e%2) + 4*(e/2) +
//     2*(w%2)) mod 32, so rotating right by 4*(e/2) + 2*(w%2) and masking
//     0x00300030 lands them next to the low nibbles.
//   scales (groupwise INT): 16-bit [row][g], g_kb = groups per tile
//   zeros (groupwise INT with zero points): u8 [row][g]
//   MXFP4 scales: UE8M0 u8 [row][4] (one per 32-column chunk)
//   NVFP4: codes as MXFP4; scales e4m3 u8 [row][8] (one per 16 columns:
//     words 0-1 of chunk c use scale 2c, words 2-3 scale 2c+1)
//   MXINT4: codes as symmetric INT4 (offset-binary u = q+8); scales as MXFP4
//   FP8: the 128 x 128-byte A-operand image in the 128-byte swizzled K-major
//     layout: row r at r*128, 16-byte chunk j stored at chunk j ^ (r % 8).
#pragma once

#include <cstddef>
#include <cstdint>

#include "hq.h"

struct __nv_bfloat16;

namespace hq {

constexpr int kTileN = 128;
constexpr int kTileK = 128;
constexpr uint32_t kHeaderBytes = 256;
constexpr uint32_t kMagic = 0x31545148u;  // "HQT1"
constexpr uint32_t kLayoutVersion = 1;

// Head of every GEMM workspace: the status word region, then a fixed region
// of split-K / stream-K counters (8 per tile, at most kMaxSplitTiles tiles),
// then the fp32 partials.
constexpr size_t kWsStatusBytes = 256;
constexpr int kMaxSplitTiles = 512;
constexpr size_t kWsCounterBytes = sizeof(int) * kMaxSplitTiles * 8;

// Device-side header of a transformed weight.
struct TileHeader {
  uint32_t magic;
  uint32_t version;
  int32_t wtype, stype, n, k, num_experts, group_k, signed_codes, has_zeros;
  uint32_t invalid_count;  // NaN scales / codes seen by hq_transform
  uint32_t pad[53];
};
static_assert(sizeof(TileHeader) == kHeaderBytes, "header must be 256 bytes");

struct Layout {
  int wtype, stype, n, k, num_experts, group_k, signed_codes, has_zeros;
  int n_pad, k_pad, n_tiles, k_tiles;
  int channel;  // INT with group_k == 0: scale (and zero) per row, scale applied in the epilogue
  int g_kb;     // INT groupwise: scale groups stored per tile (1, 2 or 4)
  int groups;   // scale groups per row in the standard format (INT)
  uint32_t codes_bytes, hi_off, scale_off, scale_bytes, zero_off, zero_bytes, tile_bytes;
  uint64_t tiles_off, expert_stride, row_off, row_zero_off, blk_off, ts_off, total;
};

// Fill L from a descriptor; returns HQ_OK or the validation error.
hq_status make_layout(const hq_weight_desc& d, Layout* L);

#if defined(__CUDACC__)
#define HQ_HD __host__ __device__
#else
#define HQ_HD
#endif

// tcgen05 // Instruction descriptors: D fp32 (bits 4-5 = 1), A/B format (bits 7-9,
// 10-12), both operands K-major, N >> 3 at bit 17, M >> 4 at bit 24.
HQ_HD constexpr uint32_t idesc_f16(bool bf16, int m, int n) {
  return (1u << 4) | ((bf16 ? 1u : 0u) << 7) | ((bf16 ? 1u : 0u) << 10) |
         (static_cast<uint32_t>(n >> 3) << 17) | (static_cast<uint32_t>(m >> 4) << 24);
}
// Block-scaled MMA (kind::mxf8f6f4.block_scale.scale_vec::1X), e4m3 x e4m3
// with UE8M0 scale factors: A/B format 0 (E4M3) at bits 7-9 / 10-12, both
// K-major, N >> 3 at bit 17, scale format E8M0 (bit 23), M >> 4 at bit 24,
// scale-factor ids 0 (bits 4-5 for B, 29-30 for A), K = 32.
HQ_HD constexpr uint32_t idesc_mx_e4m3(int m, int n) {
  return (static_cast<uint32_t>(n >> 3) << 17) | (1u << 23) | (static_cast<uint32_t>(m >> 4) << 24);
}
HQ_HD constexpr uint32_t idesc_e4m3(int m, int n) {
  return (1u << 4) | (0u << 7) | (0u << 10) | (static_cast<uint32_t>(n >> 3) << 17) |
         (static_cast<uint32_t>(m >> 4) << 24);
}

// ------------------------------------------------------------------ GEMM
// MXFP4_A8: MXFP4 weights against MXFP8 activations (e4m3 codes with one
// UE8M0 exponent per 32 along K), block-scaled MMA.
enum class WFmt : int { INT4 = 0, INT6 = 1, MXFP4 = 2, NVFP4 = 3, MXINT4 = 4, MXFP4_A8 = 5 };

struct GemmParams {
  const uint8_t* tiles;     // tile (e=0, nt=0, kt=0)
  uint64_t expert_stride;   // bytes between experts
  uint32_t tile_bytes, hi_off, scale_off, zero_off;
  int g_kb, group_k, has_zeros, channel, zero_sym;  // zero_sym: implicit zero for symmetric codes
  const float* row_scale;   // channel: [E][n_pad]
  const uint8_t* row_zero;  // channel with zeros: [E][n_pad]
  const float* tensor_scale;// NVFP4: [E], applied to the fp32 sums
  int n, n_pad, k, k_tiles, n_tiles;
  int m;                    // dense: rows of X / Y
  int bn;                   // MMA N (tokens per tile), multiple of 16
  int m_tiles, num_tiles;   // dense: token tiles, output tiles (m_tiles * n_tiles); MoE: m_tiles = 2
                            // when the routed rows average more than a tile per expert, else 1
  int stages, x_stages;     // weight-ring and activation-ring stages
  int groups;               // dequantiser groups (for reporting)
  int stream_k;             // dense: deal K-blocks out in equal ranges (1) or whole tiles (0)
  int cluster;              // dense: 2 = a 2-CTA cluster per tile, each CTA half of K, combined in shared memory
  int x3d;                  // activation map is 3-D: one box = every slab of a stage
  long long iters;          // stream-K: tiles * k_tiles
  uint32_t idesc;
  // output
  void* y;
  int64_t ldy;
  int y_tma;                // dense: Y written by tensor stores of 16 x 32 boxes through shared memory
  float* partials;          // stream-K: [2 * grid][bn][128] fp32 (head and tail unit of each CTA)
  int* counters;            // stream-K: [tiles][4], zero between calls
  int* status;
  // MoE (grouped mode)
  int num_experts, topk;
  const int* tile_offsets;  // [E+1] m-tile prefix over experts
  const int* expert_offsets;// [E+1] row prefix
  const int* perm;          // [rows]: routed position -> pair index f (indexed) or X/Y row (grouped forms)
  const float* topk_w;      // [T*topk]
  const int* x_base;        // [E]: X row of each expert's first routed row (its rows stand together in X)
  float* zbuf;              // [T*topk][n_pad] weighted per-pair outputs
  float* gate_buf;          // gated: [grid][bn max of the class][128] fp32 gate sums, one block per CTA
  const uint8_t* x_mx;      // MXFP4_A8: activation UE8M0 exponents [m][k/32] (rows 4-byte aligned)
  int64_t ld_mx;            // MXFP4_A8: row stride of x_mx in bytes
  int moe_out;              // kMoeOutZ, kMoeOutRowMap or kMoeOutRouted
};

// MoE output modes: the weighted fp32 row zbuf[perm[p]] (combined afterwards),
// the 16-bit Y row perm[p] (grouped forms), the 16-bit Y row p itself (rows in
// routed order, the feed-forward block's gate+up output), or, gated, the
// 16-bit row p of silu(gate) * up: the weight holds 2I rows (gate rows, then
// up rows, I a multiple of 128) and each CTA takes a gate tile and the
// matching up tile as two consecutive units, writing I outputs per row; the
// gate tile's fp32 sums wait for the up tile in the CTA's block of gate_buf.
constexpr int kMoeOutZ = 0, kMoeOutRowMap = 1, kMoeOutRouted = 2, kMoeOutGated = 3;

struct Fp8Params {
  const uint8_t* tiles;
  uint64_t expert_stride;
  uint32_t tile_bytes;
  const float* blk_scale;   // [n_tiles][k_tiles]
  const float* x_scale;     // [m][k_tiles]
  int n, n_pad, k_tiles, n_tiles, m, bn, m_tiles, stages;
  int splits, kb_per_split;
  uint32_t idesc;
  void* y;
  int64_t ldy;
  float* partials;          // split-K: [splits][m][n_pad] fp32
  int* counters;            // split-K: [m_tiles * n_groups * 8]
  int* status;
};

}  // namespace hq
