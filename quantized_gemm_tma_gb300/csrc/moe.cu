// moe.cu — MoE routing and combine around the grouped GEMM (Humming aiwiki
// article, "Device and workload selection": indexed input gathered through
// routing indices; grouped-contiguous execution places each expert's rows
// together).
//
// route:   a stable counting sort of the T*topk (token, slot) pairs by expert
//          in one CTA: per-warp histograms over contiguous segments, an
//          exclusive prefix over experts and warps, then an in-order scatter
//          (ranks inside a 32-pair step from __match_any_sync).  Also emits
//          the prefix of m-tiles per expert for the grouped GEMM scheduler.
// combine: Y[t, :] = sum_j Z[t*topk + j, :] in slot order (Z already carries
//          the routing weight), rounded once to bf16.
// permute: the routed activation rows in expert order (the grouped-contiguous
//          organisation of an indexed input): Xg[p, :] = X[perm[p] / topk, :],
//          so that the grouped GEMM loads whole tiles of an expert's rows;
//          for W4A8 the gathered rows are quantised to MXFP8 on the way.
// grouped: the grouped-contiguous and grouped-masked input forms (rows per
//          expert given by the caller): offsets, tile prefix, row map and the
//          X row where each expert's rows start.
// act:     silu(gate) * up between the gate+up and down GEMMs of the MoE
//          feed-forward block.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>

#include "hq_internal.h"
#include "hq_launch.h"
#include "hq_ptx.cuh"
#include "mxfp8.cuh"

namespace hq {
namespace {

constexpr int kRouteThreads = 1024;
constexpr int kRouteWarps = kRouteThreads / 32;
constexpr int kRouteChunk = 8;  // expert ids per lane loaded together
constexpr int kCountThreads = 256;

// Block-wide exclusive scan of one value per thread (threads >= count hold 0).
__device__ __forceinline__ int block_exclusive_scan(int v, int* warp_tot, int& total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int inc = v;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const int t = __shfl_up_sync(0xffffffffu, inc, d);
    if (lane >= d) inc += t;
  }
  if (lane == 31) warp_tot[warp] = inc;
  __syncthreads();
  if (warp == 0) {
    int w = warp_tot[lane];
    int winc = w;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int t = __shfl_up_sync(0xffffffffu, winc, d);
      if (lane >= d) winc += t;
    }
    warp_tot[lane] = winc - w;           // exclusive prefix of warp totals
    if (lane == 31) warp_tot[32] = winc;  // grand total
  }
  __syncthreads();
  total = warp_tot[32];
  const int r = warp_tot[warp] + inc - v;
  __syncthreads();
  return r;
}

// Many pairs: block b counts the experts of its contiguous segment of
// blk_seg pairs into counts[b][E]; the route kernel below, one block per
// segment, turns the table into each block's write base.
__global__ void __launch_bounds__(kCountThreads)
    moe_route_count_kernel(const int* __restrict__ ids, int pairs, int num_experts, int blk_seg,
                           int* __restrict__ counts, int* __restrict__ status) {
  extern __shared__ int cnt_s[];  // [E]
  const int E = num_experts;
  for (int e = threadIdx.x; e < E; e += blockDim.x) cnt_s[e] = 0;
  __syncthreads();
  const int g0 = blockIdx.x * blk_seg, g1 = min(pairs, g0 + blk_seg);
  bool bad = false;
  for (int f = g0 + static_cast<int>(threadIdx.x); f < g1; f += blockDim.x) {
    const int e = ids[f];
    if (e >= 0 && e < E) atomicAdd(&cnt_s[e], 1);
    else bad = true;
  }
  if (bad) atomicCAS(status, 0, static_cast<int>(HQ_ERR_INVALID_VALUE));
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) counts[static_cast<size_t>(blockIdx.x) * E + e] = cnt_s[e];
}

// Block b routes the pairs [b blk_seg, (b + 1) blk_seg): per-warp histograms
// of its segment, then a stable scatter.  With one block (counts == nullptr)
// the expert totals are the block's own; with several, counts[gridDim.x][E]
// gives the totals and the pairs of earlier blocks, so every pair lands
// where the stable counting sort over all pairs puts it.
__global__ void __launch_bounds__(kRouteThreads, 1)
    moe_route_kernel(const int* __restrict__ ids, int pairs, int num_experts, int bn, int blk_seg,
                     const int* __restrict__ counts, int* __restrict__ exp_off, int* __restrict__ tile_off,
                     int* __restrict__ perm, int* __restrict__ off_out, int* __restrict__ perm_out,
                     int* __restrict__ status) {
  // launched with programmatic dependent launch: the previous grid and its
  // memory are complete before anything here touches global memory
  dev::grid_dep_wait();
  dev::grid_dep_launch();
  extern __shared__ int sm[];
  int* wcnt = sm;                                  // [warps][E]: per-warp counts, then write cursors
  int* warp_tot = sm + kRouteWarps * num_experts;  // [33]
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int E = num_experts;
  const int g0 = blockIdx.x * blk_seg, g1 = min(pairs, g0 + blk_seg);
  const int seg = (g1 - g0 + kRouteWarps - 1) / kRouteWarps;
  const int f0 = g0 + warp * seg, f1 = min(g1, f0 + seg);

  for (int i = tid; i < kRouteWarps * E; i += kRouteThreads) wcnt[i] = 0;
  __syncthreads();
  // ids are read kRouteChunk per lane at a time, so one load latency covers
  // 32 x kRouteChunk pairs of the warp's segment
  bool bad = false;
  for (int b = f0; b < f1; b += 32 * kRouteChunk) {
    int ev[kRouteChunk];
#pragma unroll
    for (int j = 0; j < kRouteChunk; ++j) {
      const int f = b + 32 * j + lane;
      ev[j] = f < f1 ? ids[f] : 0;
    }
#pragma unroll
    for (int j = 0; j < kRouteChunk; ++j) {
      if (b + 32 * j + lane >= f1) continue;
      if (ev[j] >= 0 && ev[j] < E) atomicAdd(&wcnt[warp * E + ev[j]], 1);
      else bad = true;
    }
  }
  if (bad && counts == nullptr) atomicCAS(status, 0, static_cast<int>(HQ_ERR_INVALID_VALUE));
  __syncthreads();

  // per-expert totals (and the pairs of earlier blocks), exclusive prefix
  // over experts (rows and m-tiles)
  int cnt = 0, before = 0;
  if (tid < E) {
    if (counts == nullptr) {
      for (int w = 0; w < kRouteWarps; ++w) cnt += wcnt[w * E + tid];
    } else {
      for (int b = 0; b < static_cast<int>(gridDim.x); ++b) {
        const int c = counts[static_cast<size_t>(b) * E + tid];
        cnt += c;
        if (b < static_cast<int>(blockIdx.x)) before += c;
      }
    }
  }
  int rows_total = 0, tiles_total = 0;
  const int row_base = block_exclusive_scan(tid < E ? cnt : 0, warp_tot, rows_total);
  const int tile_base = block_exclusive_scan(tid < E ? (cnt + bn - 1) / bn : 0, warp_tot, tiles_total);
  if (tid < E) {
    if (blockIdx.x == 0) {
      exp_off[tid] = row_base;
      tile_off[tid] = tile_base;
      if (off_out) off_out[tid] = row_base;
    }
    // write cursor of each warp for this expert: the pairs routed to it by
    // earlier blocks and by this block's earlier warps come first
    int run = row_base + before;
    for (int w = 0; w < kRouteWarps; ++w) {
      const int c = wcnt[w * E + tid];
      wcnt[w * E + tid] = run;
      run += c;
    }
  }
  if (tid == 0 && blockIdx.x == 0) {
    exp_off[E] = rows_total;
    tile_off[E] = tiles_total;
    if (off_out) off_out[E] = rows_total;
  }
  __syncthreads();

  // stable scatter: each warp walks its segment in order, 32 pairs per step
  int* cur = wcnt + warp * E;
  for (int b = f0; b < f1; b += 32 * kRouteChunk) {
    int ev[kRouteChunk];
#pragma unroll
    for (int j = 0; j < kRouteChunk; ++j) {
      const int f = b + 32 * j + lane;
      ev[j] = f < f1 ? ids[f] : -1;
    }
#pragma unroll
    for (int j = 0; j < kRouteChunk; ++j) {
      const int f = b + 32 * j + lane;
      int e = ev[j];
      if (e < 0 || e >= E) e = -1;
      const unsigned peers = __match_any_sync(0xffffffffu, e);
      const int rank = __popc(peers & ((1u << lane) - 1u));
      int pos = 0;
      if (e >= 0) pos = cur[e] + rank;
      __syncwarp();
      if (e >= 0) {
        perm[pos] = f;
        if (perm_out) perm_out[pos] = f;
        if (rank == 0) cur[e] += __popc(peers);
      }
      __syncwarp();
    }
  }
}

// Grouped input forms: the rows of expert e are given, either contiguously
// (rows [offs[e], offs[e+1]) of X and Y) or masked (rows [e*max_rows,
// e*max_rows + counts[e]) of an [E][max_rows] block).  Writes the compacted
// offsets, the m-tile prefix and, for compacted position p of expert e, the
// X / Y row perm[p].  Invalid counts or offsets make the expert contribute
// nothing and set HQ_ERR_INVALID_VALUE.
__global__ void __launch_bounds__(kRouteThreads, 1)
    moe_grouped_route_kernel(const int* __restrict__ rows_in, int masked, int rows, int num_experts, int bn,
                             int* __restrict__ exp_off, int* __restrict__ tile_off, int* __restrict__ perm,
                             int* __restrict__ x_base, int* __restrict__ status) {
  // launched with programmatic dependent launch: the previous grid and its
  // memory are complete before anything here touches global memory
  dev::grid_dep_wait();
  dev::grid_dep_launch();
  __shared__ int warp_tot[33];
  __shared__ int s_off[kRouteThreads];
  __shared__ int s_base[kRouteThreads];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int E = num_experts;
  int cnt = 0, base = 0;
  if (tid < E) {
    if (masked) {
      cnt = rows_in[tid];
      base = tid * rows;
      if (cnt < 0 || cnt > rows) {
        atomicCAS(status, 0, static_cast<int>(HQ_ERR_INVALID_VALUE));
        cnt = 0;
      }
    } else {
      base = rows_in[tid];
      const int end = rows_in[tid + 1];
      cnt = end - base;
      if (base < 0 || cnt < 0 || end > rows) {
        atomicCAS(status, 0, static_cast<int>(HQ_ERR_INVALID_VALUE));
        cnt = 0;
        base = 0;
      }
    }
  }
  int rows_total = 0, tiles_total = 0;
  const int row_base = block_exclusive_scan(cnt, warp_tot, rows_total);
  const int tile_base = block_exclusive_scan((cnt + bn - 1) / bn, warp_tot, tiles_total);
  if (tid < E) {
    exp_off[tid] = row_base;
    tile_off[tid] = tile_base;
    x_base[tid] = base;
    s_off[tid] = row_base;
    s_base[tid] = base;
  }
  if (tid == 0) {
    exp_off[E] = rows_total;
    tile_off[E] = tiles_total;
  }
  __syncthreads();
  for (int e = warp; e < E; e += kRouteWarps) {
    const int o = s_off[e], b = s_base[e], c = (e + 1 < E ? s_off[e + 1] : rows_total) - o;
    for (int r = lane; r < c; r += 32) perm[o + r] = b + r;
  }
}

// Xg[p, :] = X[perm[p] / topk, :] for the routed positions p < *routed (the
// route's row total: pairs with an invalid expert id are not routed), K bf16
// values per row (K a multiple of 8): one thread per 16-byte chunk, rows of X
// read through L2 (each token's row serves its topk pairs), Xg written once.
__global__ void moe_permute_kernel(const uint4* __restrict__ x, int64_t ldx16, int tokens,
                                   const int* __restrict__ perm, const int* __restrict__ routed, int topk,
                                   int chunks, uint4* __restrict__ xg, int64_t ldg16) {
  const int64_t total = static_cast<int64_t>(*routed) * chunks;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t p = i / chunks;
    const int c = static_cast<int>(i - p * chunks);
    const int t = perm[p] / topk;
    if (t < 0 || t >= tokens) continue;
    xg[p * ldg16 + c] = __ldg(x + t * ldx16 + c);
  }
}

// The same gather quantising each row to MXFP8 (W4A8): Q[p][:k] e4m3 and
// Ex[p][:k/32] UE8M0 of X[perm[p] / topk], the conversion of the standalone
// quantiser.  One thread per 8 elements of every slot up to `pairs` (the four
// lanes of a 32-element block are consecutive: k % 32 == 0); slots past the
// device count *routed are left alone, and every lane takes part in the
// block's shuffles.
__global__ void __launch_bounds__(256) moe_permute_mxfp8_kernel(const __nv_bfloat16* __restrict__ x, int64_t ldx,
                                                                int tokens, const int* __restrict__ perm,
                                                                const int* __restrict__ routed, int pairs, int topk,
                                                                int k, uint8_t* __restrict__ q, int64_t ldq,
                                                                uint8_t* __restrict__ ex, int64_t lde) {
  const int per_row = k / 8;
  const int64_t idx = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int64_t rows = min(*routed, pairs);
  const bool live = idx < rows * per_row;
  const int64_t p = live ? idx / per_row : 0;
  const int j = live ? static_cast<int>(idx - p * per_row) : 0;
  const int t = live ? perm[p] / topk : -1;
  uint4 raw = make_uint4(0, 0, 0, 0);
  if (t >= 0 && t < tokens) raw = __ldg(reinterpret_cast<const uint4*>(x + static_cast<int64_t>(t) * ldx + 8 * j));
  int E = 0;
  const uint2 packed = dev::mxfp8_quantize8(raw, &E);
  if (live) {
    *reinterpret_cast<uint2*>(q + p * ldq + 8 * j) = packed;
    if ((j & 3) == 0) ex[p * lde + j / 4] = static_cast<uint8_t>(E);
  }
}

// MoE feed-forward activation between the two grouped GEMMs:
//   A[f][i] = silu(H[f][i]) * H[f][inter + i],  silu(g) = g / (1 + e^-g),
// computed in fp32 from the bf16 gate and up halves and rounded once to bf16.
// One thread per (pair, 8 consecutive outputs): 16-byte loads and stores.
__global__ void moe_act_kernel(const __nv_bfloat16* __restrict__ h, int64_t ldh, int pairs, int inter,
                               __nv_bfloat16* __restrict__ a, int64_t lda) {
  dev::grid_dep_wait();
  dev::grid_dep_launch();
  const int groups = inter / 8;
  const int64_t idx = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (idx >= static_cast<int64_t>(pairs) * groups) return;
  const int64_t f = idx / groups;
  const int i0 = static_cast<int>(idx % groups) * 8;
  const uint4 g4 = *reinterpret_cast<const uint4*>(h + f * ldh + i0);
  const uint4 u4 = *reinterpret_cast<const uint4*>(h + f * ldh + inter + i0);
  const __nv_bfloat162* g2 = reinterpret_cast<const __nv_bfloat162*>(&g4);
  const __nv_bfloat162* u2 = reinterpret_cast<const __nv_bfloat162*>(&u4);
  uint4 o;
  __nv_bfloat162* o2 = reinterpret_cast<__nv_bfloat162*>(&o);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 g = __bfloat1622float2(g2[i]);
    const float2 u = __bfloat1622float2(u2[i]);
    o2[i] = __floats2bfloat162_rn(g.x / (1.f + expf(-g.x)) * u.x, g.y / (1.f + expf(-g.y)) * u.y);
  }
  *reinterpret_cast<uint4*>(a + f * lda + i0) = o;
}

// One thread per (token, 8 consecutive outputs).
__global__ void moe_combine_kernel(const float* __restrict__ z, const int* __restrict__ ids, int tokens, int topk,
                                   int num_experts, int n, int n_pad, __nv_bfloat16* __restrict__ y, int64_t ldy) {
  dev::grid_dep_wait();
  dev::grid_dep_launch();
  const int groups = (n + 7) / 8;
  const int64_t idx = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (idx >= static_cast<int64_t>(tokens) * groups) return;
  const int t = static_cast<int>(idx / groups);
  const int n0 = static_cast<int>(idx % groups) * 8;
  float acc[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) acc[i] = 0.f;
  for (int j = 0; j < topk; ++j) {
    const int f = t * topk + j;
    const int e = ids[f];
    if (e < 0 || e >= num_experts) continue;
    const float4* src = reinterpret_cast<const float4*>(z + static_cast<size_t>(f) * n_pad + n0);
    const float4 a = __ldcs(src), b = __ldcs(src + 1);
    acc[0] += a.x; acc[1] += a.y; acc[2] += a.z; acc[3] += a.w;
    acc[4] += b.x; acc[5] += b.y; acc[6] += b.z; acc[7] += b.w;
  }
  __nv_bfloat16* yr = y + static_cast<size_t>(t) * ldy + n0;
  if (n0 + 8 <= n) {
    uint4 o;
    __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&o);
#pragma unroll
    for (int i = 0; i < 4; ++i) h[i] = __floats2bfloat162_rn(acc[2 * i], acc[2 * i + 1]);
    *reinterpret_cast<uint4*>(yr) = o;
  } else {
    for (int i = 0; i < 8 && n0 + i < n; ++i) yr[i] = __float2bfloat16_rn(acc[i]);
  }
}

}  // namespace

int moe_route_blocks(int pairs) {
  if (pairs <= kRouteSinglePairs) return 1;
  return std::min(kRouteMaxBlocks, (pairs + kRoutePairsPerBlock - 1) / kRoutePairsPerBlock);
}

cudaError_t launch_moe_route(const int* topk_ids, int pairs, int num_experts, int bn, int* expert_offsets,
                             int* tile_offsets, int* perm, int* offsets_out, int* perm_out, int* counts,
                             int* status, cudaStream_t stream) {
  const size_t smem = sizeof(int) * (static_cast<size_t>(kRouteWarps) * num_experts + 33);
  cudaError_t e = ensure_smem_optin(reinterpret_cast<const void*>(moe_route_kernel));
  if (e != cudaSuccess) return e;
  const int blocks = moe_route_blocks(pairs);
  const int blk_seg = (pairs + blocks - 1) / blocks;
  if (blocks > 1) {
    moe_route_count_kernel<<<blocks, kCountThreads, sizeof(int) * num_experts, stream>>>(topk_ids, pairs,
                                                                                       num_experts, blk_seg,
                                                                                       counts, status);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  const int* block_counts = blocks > 1 ? counts : nullptr;
  return launch_pdl(reinterpret_cast<const void*>(moe_route_kernel), blocks, kRouteThreads,
                    static_cast<uint32_t>(smem), stream, 1, topk_ids, pairs, num_experts, bn, blk_seg, block_counts,
                    expert_offsets, tile_offsets, perm, offsets_out, perm_out, status);
}

cudaError_t launch_moe_grouped_route(const int* rows_in, bool masked, int rows, int num_experts, int bn,
                                     int* expert_offsets, int* tile_offsets, int* perm, int* x_base, int* status,
                                     cudaStream_t stream) {
  if (num_experts > kRouteThreads) return cudaErrorInvalidValue;
  const int masked_i = masked ? 1 : 0;
  return launch_pdl(reinterpret_cast<const void*>(moe_grouped_route_kernel), 1, kRouteThreads, 0u, stream, 1,
                    rows_in, masked_i, rows, num_experts, bn, expert_offsets, tile_offsets, perm, x_base, status);
}

cudaError_t launch_moe_permute(const void* x, int64_t ldx, int tokens, const int* perm, const int* routed,
                               int pairs, int topk, int k, void* xg, int64_t ldg, int sms, cudaStream_t stream) {
  if (pairs == 0) return cudaSuccess;
  if (k % 8 || ldx % 8 || ldg % 8) return cudaErrorInvalidValue;
  const int chunks = k / 8;
  const int64_t total = static_cast<int64_t>(pairs) * chunks;  // at most this many routed chunks
  const int block = 256;
  const int64_t want = (total + block - 1) / block;
  const int grid = static_cast<int>(std::min<int64_t>(want, static_cast<int64_t>(sms) * 8));
  moe_permute_kernel<<<grid, block, 0, stream>>>(static_cast<const uint4*>(x), ldx / 8, tokens, perm, routed, topk,
                                                 chunks, static_cast<uint4*>(xg), ldg / 8);
  return cudaGetLastError();
}

cudaError_t launch_moe_permute_mxfp8(const void* x, int64_t ldx, int tokens, const int* perm, const int* routed,
                                     int pairs, int topk, int k, void* q, int64_t ldq, void* ex, int64_t lde,
                                     cudaStream_t stream) {
  if (pairs == 0) return cudaSuccess;
  if (k % 32 || ldx % 8 || ldq % 8) return cudaErrorInvalidValue;
  const int64_t threads = static_cast<int64_t>(pairs) * (k / 8);
  const int block = 256;
  moe_permute_mxfp8_kernel<<<static_cast<unsigned>((threads + block - 1) / block), block, 0, stream>>>(
      static_cast<const __nv_bfloat16*>(x), ldx, tokens, perm, routed, pairs, topk, k, static_cast<uint8_t*>(q), ldq,
      static_cast<uint8_t*>(ex), lde);
  return cudaGetLastError();
}

cudaError_t launch_moe_act(const void* h, int64_t ldh, int pairs, int inter, void* a, int64_t lda,
                           cudaStream_t stream) {
  const int64_t threads = static_cast<int64_t>(pairs) * (inter / 8);
  if (threads == 0) return cudaSuccess;
  const int block = 256;
  const __nv_bfloat16* hp = static_cast<const __nv_bfloat16*>(h);
  __nv_bfloat16* ap = static_cast<__nv_bfloat16*>(a);
  return launch_pdl(reinterpret_cast<const void*>(moe_act_kernel), static_cast<int>((threads + block - 1) / block),
                    block, 0u, stream, 1, hp, ldh, pairs, inter, ap, lda);
}

cudaError_t launch_moe_combine(const float* zbuf, const int* topk_ids, int tokens, int topk, int num_experts, int n,
                               int n_pad, void* y, int64_t ldy, bool bf16, cudaStream_t stream) {
  (void)bf16;
  const int64_t threads = static_cast<int64_t>(tokens) * ((n + 7) / 8);
  const int block = 256;
  __nv_bfloat16* yp = static_cast<__nv_bfloat16*>(y);
  return launch_pdl(reinterpret_cast<const void*>(moe_combine_kernel), static_cast<int>((threads + block - 1) / block),
                    block, 0u, stream, 1, zbuf, topk_ids, tokens, topk, num_experts, n, n_pad, yp, ldy);
}

}  // namespace hq
