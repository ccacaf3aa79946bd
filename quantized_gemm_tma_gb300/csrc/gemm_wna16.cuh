// gemm_wna16.cuh — the weight-only-quantized GEMM kernel for sm_103a:
// low-bit weights (INT4 / INT6 / MXFP4) against BF16 or FP16 activations, in
// a dense form and an MoE grouped form ("WnA16": low-bit weights with 16-bit
// activations — Humming launch article, WnA16 paragraph; MoE GEMM — README
// Key Features).
//
// Computes D[n, m] = sum_k W[n, k] * X[m, k] per tile of 128 weight rows x BN
// tokens ("swap AB": the weights are the MMA's M side, so decode-sized M only
// pads the MMA N dimension, down to 16).
//
// Warp roles (320 threads, one CTA per SM):
//   warp 0     TMA producer: one bulk copy per weight tile (codes, scales and
//              zeros are contiguous in the transformed layout) and a 2-D
//              tensor copy of the activation tile (128-byte swizzle) into a
//              multi-stage shared-memory ring.  MoE: activation rows are
//              gathered by routing index with cp.async into the same swizzled
//              layout.
//   warp 1     TMEM allocator and MMA issuer: one thread issues
//              tcgen05.mma.kind::f16 with the A operand (dequantised weights)
//              read from tensor memory and B (activations) from shared memory,
//              fp32 accumulation in TMEM.
//   warps 2-9  dequantisers: each thread owns one weight row (TMEM lane) and
//              two 32-column chunks of every 128-column K block; it turns the
//              packed codes into bf16x2/f16x2 pairs with magic-number integer
//              to float conversion, applies zero point and scale, and writes
//              them into the A ring in TMEM with tcgen05.st.  After the K loop
//              the same warps run the epilogue (tcgen05.ld -> scale -> store,
//              split-K partials with a deterministic last-arriver reduction,
//              or the MoE per-pair weighted outputs).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "hq_internal.h"
#include "hq_ptx.cuh"

namespace hq {
namespace wna16 {

constexpr int kDqWarps = kWna16DqWarps;
constexpr int kThreads = 64 + 32 * kDqWarps;
constexpr int kAStages = kWna16AStages;

template <int BN_MAX>
struct Cfg {
  static constexpr int kTmemCols = (BN_MAX + 64 * kAStages) <= 256 ? 256 : 512;
  static constexpr int kAccCol = 0;
  static constexpr int kACol = BN_MAX;
};

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

// INT4 chunk of 32 codes (offset-binary u) -> 16 pairs of (u - z) [* s].
template <bool BF16, bool SCALE>
__device__ __forceinline__ void dq_int4(const uint4 q, uint32_t c2, uint32_t s2, uint32_t (&o)[16]) {
  const uint32_t w[4] = {q.x, q.y, q.z, q.w};
  constexpr uint32_t M = magic_half<BF16>() * 0x00010001u;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint32_t v = ((w[j] >> (4 * i)) & 0x000F000Fu) | M;
      const uint32_t t = h2sub<BF16>(v, c2);
      o[4 * j + i] = SCALE ? h2mul<BF16>(t, s2) : t;
    }
  }
}

// INT6 chunk: low nibbles as INT4, top two bits from the rotated hi words.
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

// All lanes wait; the outcome is made warp-uniform so that the .sync.aligned
// tcgen05 instructions that follow are always executed by the full warp.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, volatile int* abort) {
  const bool got = dev::mbar_wait(bar, parity, abort);
  return __all_sync(0xffffffffu, got) != 0;
}

// ---------------------------------------------------------------- work items
struct Work {
  int e, nt, row0, rows, kb0, kb1, split, mt;
};

template <bool MOE>
__device__ __forceinline__ Work decode_work(const GemmParams& p, int w, const int* s_tile_off, const int* s_row_off) {
  Work r;
  if constexpr (!MOE) {
    r.split = w % p.splits;
    const int t = w / p.splits;
    r.nt = t % p.n_tiles;
    r.mt = t / p.n_tiles;
    r.e = 0;
    r.row0 = r.mt * p.bn;
    r.rows = min(p.bn, p.m - r.row0);
    r.kb0 = r.split * p.kb_per_split;
    r.kb1 = min(p.k_tiles, r.kb0 + p.kb_per_split);
  } else {
    const int tile = w / p.n_tiles;
    r.nt = w % p.n_tiles;
    // expert e: last index with tile_off[e] <= tile
    int lo = 0, hi = p.num_experts;  // invariant tile_off[lo] <= tile < tile_off[hi]
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (s_tile_off[mid] <= tile) lo = mid; else hi = mid;
    }
    r.e = lo;
    r.mt = tile - s_tile_off[lo];
    r.row0 = s_row_off[lo] + r.mt * p.bn;
    r.rows = min(p.bn, s_row_off[lo + 1] - r.row0);
    r.kb0 = 0;
    r.kb1 = p.k_tiles;
    r.split = 0;
  }
  return r;
}

// ---------------------------------------------------------------- the kernel
template <int FMT, bool BF16, int BN_MAX, bool MOE>
__global__ void __launch_bounds__(kThreads, (BN_MAX <= 64 ? 2 : 1))
    wna16_kernel(const __grid_constant__ GemmParams p, const __grid_constant__ CUtensorMap tmap_x,
                 const __nv_bfloat16* __restrict__ x_rows /* MoE: activations [T][ldx] */, int64_t ldx) {
  using C = Cfg<BN_MAX>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

  const int S = p.stages;
  const int bn = p.bn;
  const uint32_t tile_bytes = p.tile_bytes;
  const uint32_t w_stage_bytes = (tile_bytes + 127u) & ~127u;
  const uint32_t x_stage_bytes = static_cast<uint32_t>(bn) * 256u;  // two 128-byte-wide K halves
  uint8_t* w_st = smem;
  uint8_t* x_st = smem + ((S * w_stage_bytes + 1023u) & ~1023u);
  uint64_t* bars = reinterpret_cast<uint64_t*>(x_st + S * x_stage_bytes);
  uint64_t* full = bars;
  uint64_t* empty = bars + S;
  uint64_t* a_full = bars + 2 * S;
  uint64_t* a_empty = a_full + kAStages;
  uint64_t* acc_full = a_empty + kAStages;
  uint64_t* acc_empty = acc_full + 1;
  uint64_t* tear = acc_empty + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(tear + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  int* s_tile_off = reinterpret_cast<int*>(tmem_slot + 4);
  int* s_row_off = s_tile_off + (MOE ? p.num_experts + 1 : 0);

  const int warp = threadIdx.x >> 5;
  const uint32_t lane = dev::lane_id();

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      dev::mbar_init(&full[s], MOE ? 33u : 1u);
      dev::mbar_init(&empty[s], kDqWarps + 1);
    }
    for (int j = 0; j < kAStages; ++j) {
      dev::mbar_init(&a_full[j], kDqWarps);
      dev::mbar_init(&a_empty[j], 1);
    }
    dev::mbar_init(acc_full, 1);
    dev::mbar_init(acc_empty, kDqWarps);
    dev::mbar_init(tear, 1);
    *abort_flag = 0;
    dev::fence_barrier_init();
  }
  if constexpr (MOE) {
    for (int i = threadIdx.x; i <= p.num_experts; i += blockDim.x) {
      s_tile_off[i] = p.tile_offsets[i];
      s_row_off[i] = p.expert_offsets[i];
    }
  }
  if (warp == 1) {
    dev::tmem_alloc(tmem_slot, C::kTmemCols);
    dev::tmem_relinquish();
  }
  if (warp == 0 && lane == 0 && !MOE) dev::prefetch_tmap(&tmap_x);
  dev::tc_fence_before();
  __syncthreads();
  dev::tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  const int total = MOE ? s_tile_off[p.num_experts] * p.n_tiles : p.n_tiles * p.m_tiles * p.splits;
  const uint8_t* tiles_base = p.tiles;

  if (warp == 0) {
    // ============================================================ producer
    int it = 0;
    bool ok = true;
    if (MOE || lane == 0) {
      const uint64_t pol = dev::policy_evict_first();
      for (int w = blockIdx.x; ok && w < total; w += gridDim.x) {
        const Work wk = decode_work<MOE>(p, w, s_tile_off, s_row_off);
        const uint8_t* wt = tiles_base + static_cast<uint64_t>(wk.e) * p.expert_stride +
                            static_cast<uint64_t>(wk.nt) * p.k_tiles * tile_bytes;
        // MoE: this lane's gathered activation rows (token index per row)
        int tok[BN_MAX / 32 > 0 ? BN_MAX / 32 : 1];
        if constexpr (MOE) {
#pragma unroll
          for (int q = 0; q < (BN_MAX / 32 > 0 ? BN_MAX / 32 : 1); ++q) {
            const int r = static_cast<int>(lane) + 32 * q;
            tok[q] = (r < wk.rows) ? p.perm[wk.row0 + r] / p.topk : -1;
          }
        }
        for (int kb = wk.kb0; kb < wk.kb1; ++kb, ++it) {
          const int s = it % S;
          const uint32_t ph = (it / S) & 1;
          bool got;
          if constexpr (MOE) got = warp_wait(&empty[s], ph ^ 1u, abort_flag);
          else got = dev::mbar_wait(&empty[s], ph ^ 1u, abort_flag);
          if (!got) {
            ok = false;
            break;
          }
          uint8_t* xs = x_st + s * x_stage_bytes;
          if (!MOE || lane == 0) {
            dev::mbar_arrive_expect_tx(&full[s], tile_bytes + (MOE ? 0u : x_stage_bytes));
            dev::bulk_load_hint(w_st + s * w_stage_bytes, wt + static_cast<uint64_t>(kb) * tile_bytes, tile_bytes,
                                &full[s], pol);
          }
          if constexpr (!MOE) {
            dev::tma_load_2d(xs, &tmap_x, &full[s], kb * kTileK, wk.row0);
            dev::tma_load_2d(xs + bn * 128, &tmap_x, &full[s], kb * kTileK + 64, wk.row0);
          } else {
            __syncwarp();
            // rows r = lane + 32q; 16 chunks of 16 bytes per row (two 128-byte K halves)
#pragma unroll
            for (int q = 0; q < (BN_MAX / 32 > 0 ? BN_MAX / 32 : 1); ++q) {
              const int r = static_cast<int>(lane) + 32 * q;
              if (r < bn && tok[q] >= 0) {
                const __nv_bfloat16* src = x_rows + static_cast<int64_t>(tok[q]) * ldx + kb * kTileK;
#pragma unroll
                for (int c = 0; c < 16; ++c) {
                  const int half = c >> 3, j = c & 7;
                  uint8_t* dst = xs + half * bn * 128 + r * 128 + ((j ^ (r & 7)) << 4);
                  // columns at or beyond K are zero-filled (source size 0)
                  const uint32_t src_bytes = (kb * kTileK + half * 64 + j * 8 < p.k) ? 16u : 0u;
                  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dev::smem_u32(dst)),
                               "l"(src + (src_bytes ? half * 64 + j * 8 : 0)), "r"(src_bytes)
                               : "memory");
                }
              }
            }
            asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(dev::smem_u32(&full[s]))
                         : "memory");
          }
        }
      }
      if (!ok) dev::raise_error(p.status, abort_flag, HQ_ERR_DEVICE_TIMEOUT);
      // drain: wait until every copy this warp issued has landed
      if constexpr (MOE) asm volatile("cp.async.wait_all;" ::: "memory");
      if (!MOE || lane == 0) {
        for (int s = 0; s < S && s < it; ++s) {
          const int last = ((it - 1 - s) / S) * S + s;
          const uint32_t ph = (last / S) & 1;
          const uint64_t t0 = dev::globaltimer();
          while (!dev::mbar_try_wait(&full[s], ph) && dev::globaltimer() - t0 < dev::kWaitTimeoutNs) {
          }
        }
      }
    }
  } else if (warp == 1) {
    // ============================================================ MMA issuer
    if (lane == 0) {
      int it = 0, ia = 0, item = 0;
      bool ok = true;
      const uint32_t idesc = p.idesc;
      for (int w = blockIdx.x; ok && w < total; w += gridDim.x, ++item) {
        const Work wk = decode_work<MOE>(p, w, s_tile_off, s_row_off);
        if (!dev::mbar_wait(acc_empty, (item & 1) ^ 1u, abort_flag)) {
          ok = false;
          break;
        }
        dev::tc_fence_after();
        for (int kb = wk.kb0; kb < wk.kb1; ++kb, ++it, ++ia) {
          const int s = it % S;
          const int j = ia % kAStages;
          if (!dev::mbar_wait(&full[s], (it / S) & 1, abort_flag) ||
              !dev::mbar_wait(&a_full[j], (ia / kAStages) & 1, abort_flag)) {
            ok = false;
            break;
          }
          if constexpr (MOE) dev::fence_proxy_async_smem();  // cp.async rows -> tensor-core reads
          dev::tc_fence_after();
          const uint32_t xs = dev::smem_u32(x_st + s * x_stage_bytes);
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            const uint64_t bdesc = dev::sw128_desc(xs + (kk >> 2) * bn * 128 + (kk & 3) * 32);
            dev::mma_f16_ts(tmem + C::kAccCol, tmem + C::kACol + j * 64 + kk * 8, bdesc, idesc,
                            (kb > wk.kb0 || kk > 0) ? 1u : 0u);
          }
          dev::tc_commit(&empty[s]);
          dev::tc_commit(&a_empty[j]);
        }
        if (!ok) break;
        dev::tc_commit(acc_full);
      }
      if (!ok) dev::raise_error(p.status, abort_flag, HQ_ERR_DEVICE_TIMEOUT);
      // drain: all MMAs issued by this thread complete before TMEM is freed
      dev::tc_commit(tear);
      const uint64_t t0 = dev::globaltimer();
      while (!dev::mbar_try_wait(tear, 0) && dev::globaltimer() - t0 < dev::kWaitTimeoutNs) {
      }
    }
  } else {
    // ============================================================ dequant + epilogue
    const int dq = warp - 2;            // 0..7
    const int quarter = warp & 3;       // TMEM lane quarter this warp may access
    const int half = dq >> 2;           // which two 32-column chunks of each K block
    const int r = quarter * 32 + static_cast<int>(lane);  // weight row within the tile (TMEM lane)
    const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
    int it = 0, ia = 0, item = 0;
    bool ok = true;
    for (int w = blockIdx.x; ok && w < total; w += gridDim.x, ++item) {
      const Work wk = decode_work<MOE>(p, w, s_tile_off, s_row_off);
      const int n = wk.nt * kTileN + r;
      uint32_t zrow = static_cast<uint32_t>(p.zero_sym);
      if (p.channel && p.has_zeros) zrow = p.row_zero[static_cast<size_t>(wk.e) * p.n_pad + n];
      for (int kb = wk.kb0; kb < wk.kb1; ++kb, ++it, ++ia) {
        const int s = it % S;
        if (!warp_wait(&full[s], (it / S) & 1, abort_flag)) {
          ok = false;
          break;
        }
        const uint8_t* wsm = w_st + s * w_stage_bytes;
        uint4 qc[2];
        uint2 qh[2];
        uint32_t c2[2], s2[2];
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
          const int c = 2 * half + cc;
          qc[cc] = *reinterpret_cast<const uint4*>(wsm + (c * kTileN + r) * 16);
          if constexpr (FMT == static_cast<int>(WFmt::INT6))
            qh[cc] = *reinterpret_cast<const uint2*>(wsm + p.hi_off + (c * kTileN + r) * 8);
          if constexpr (FMT == static_cast<int>(WFmt::MXFP4)) {
            s2[cc] = wsm[p.scale_off + r * 4 + c];
            c2[cc] = 0;
          } else {
            uint32_t z = zrow;
            uint32_t sc = 0;
            if (!p.channel) {
              const int g = (p.g_kb > 1) ? (32 * c) / p.group_k : 0;
              sc = reinterpret_cast<const uint16_t*>(wsm + p.scale_off)[r * p.g_kb + g];
              if (p.has_zeros) z = wsm[p.zero_off + r * p.g_kb + g];
            }
            c2[cc] = (magic_half<BF16>() + z) * 0x00010001u;
            s2[cc] = sc * 0x00010001u;
          }
        }
        __syncwarp();
        if (lane == 0) dev::mbar_arrive(&empty[s]);
        const int j = ia % kAStages;
        if (!warp_wait(&a_empty[j], ((ia / kAStages) & 1) ^ 1u, abort_flag)) {
          ok = false;
          break;
        }
        dev::tc_fence_after();
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
          const int c = 2 * half + cc;
          uint32_t o[16];
          if constexpr (FMT == static_cast<int>(WFmt::INT4)) {
            if (p.channel) dq_int4<BF16, false>(qc[cc], c2[cc], 0, o);
            else dq_int4<BF16, true>(qc[cc], c2[cc], s2[cc], o);
          } else if constexpr (FMT == static_cast<int>(WFmt::INT6)) {
            if (p.channel) dq_int6<BF16, false>(qc[cc], qh[cc], c2[cc], 0, o);
            else dq_int6<BF16, true>(qc[cc], qh[cc], c2[cc], s2[cc], o);
          } else {
            dq_mxfp4(qc[cc], s2[cc], o);
          }
          dev::tmem_st16(tmem + lane_base + C::kACol + j * 64 + c * 16, o);
        }
        dev::tmem_st_wait();
        dev::tc_fence_before();
        __syncwarp();
        if (lane == 0) dev::mbar_arrive(&a_full[j]);
      }
      if (!ok) break;

      // ---------------------------------------------------------- epilogue
      if (!warp_wait(acc_full, item & 1, abort_flag)) {
        ok = false;
        break;
      }
      dev::tc_fence_after();
      const bool n_ok = n < p.n;
      const float rs = (p.channel && n_ok) ? p.row_scale[static_cast<size_t>(wk.e) * p.n_pad + n] : 1.f;
      const int nchunks = bn >> 4;
      if constexpr (MOE) {
        for (int ch = half; ch < nchunks; ch += 2) {
          uint32_t v[16];
          dev::tmem_ld16(tmem + lane_base + C::kAccCol + ch * 16, v);
          dev::tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const int col = ch * 16 + i;
            if (col < wk.rows && n_ok) {
              const int f = p.perm[wk.row0 + col];
              p.zbuf[static_cast<size_t>(f) * p.n_pad + n] = __uint_as_float(v[i]) * rs * p.topk_w[f];
            }
          }
        }
      } else if (p.splits == 1) {
        for (int ch = half; ch < nchunks; ch += 2) {
          uint32_t v[16];
          dev::tmem_ld16(tmem + lane_base + C::kAccCol + ch * 16, v);
          dev::tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const int col = ch * 16 + i;
            if (col < wk.rows && n_ok) {
              const float f = __uint_as_float(v[i]) * rs;
              const size_t off = static_cast<size_t>(wk.row0 + col) * p.ldy + n;
              if constexpr (BF16) reinterpret_cast<__nv_bfloat16*>(p.y)[off] = __float2bfloat16_rn(f);
              else reinterpret_cast<__half*>(p.y)[off] = __float2half_rn(f);
            }
          }
        }
      } else {
        // split-K: store this split's fp32 partial, then the last of the
        // `splits` warps covering the same (rows, columns) slice sums all
        // partials in split order (deterministic) and writes Y.
        for (int ch = half; ch < nchunks; ch += 2) {
          uint32_t v[16];
          dev::tmem_ld16(tmem + lane_base + C::kAccCol + ch * 16, v);
          dev::tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const int col = ch * 16 + i;
            if (col < wk.rows)
              p.partials[(static_cast<size_t>(wk.split) * p.m + wk.row0 + col) * p.n_pad + n] = __uint_as_float(v[i]);
          }
        }
        __threadfence();
        __syncwarp();
        int* ctr = p.counters + ((wk.mt * p.n_tiles + wk.nt) * kDqWarps + dq);
        int last = 0;
        if (lane == 0) last = (atomicAdd(ctr, 1) == p.splits - 1) ? 1 : 0;
        last = __shfl_sync(0xffffffffu, last, 0);
        if (last) {
          __threadfence();
          for (int ch = half; ch < nchunks; ch += 2) {
            uint32_t v[16];
            dev::tmem_ld16(tmem + lane_base + C::kAccCol + ch * 16, v);
            dev::tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const int col = ch * 16 + i;
              if (col < wk.rows && n_ok) {
                float acc = 0.f;
                for (int sp = 0; sp < p.splits; ++sp) {
                  const float part = (sp == wk.split)
                                         ? __uint_as_float(v[i])
                                         : __ldcg(&p.partials[(static_cast<size_t>(sp) * p.m + wk.row0 + col) * p.n_pad + n]);
                  acc = (sp == 0) ? part : acc + part;
                }
                const float f = acc * rs;
                const size_t off = static_cast<size_t>(wk.row0 + col) * p.ldy + n;
                if constexpr (BF16) reinterpret_cast<__nv_bfloat16*>(p.y)[off] = __float2bfloat16_rn(f);
                else reinterpret_cast<__half*>(p.y)[off] = __float2half_rn(f);
              }
            }
          }
          if (lane == 0) *ctr = 0;  // ready for the next call
        }
      }
      dev::tc_fence_before();
      __syncwarp();
      if (lane == 0) dev::mbar_arrive(acc_empty);
    }
    if (!ok) dev::raise_error(p.status, abort_flag, HQ_ERR_DEVICE_TIMEOUT);
  }

  dev::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    dev::tc_fence_after();
    dev::tmem_dealloc(tmem, C::kTmemCols);
  }
}

// Dynamic shared memory bytes for a launch.
inline uint32_t smem_bytes(int stages, uint32_t tile_bytes, int bn, int num_experts) {
  const uint32_t w = static_cast<uint32_t>(stages) * ((tile_bytes + 127u) & ~127u);
  const uint32_t x = static_cast<uint32_t>(stages) * static_cast<uint32_t>(bn) * 256u;
  const uint32_t bars = (2u * stages + 2u * kAStages + 3u) * 8u + 16u + 8u * (num_experts + 1);
  return ((w + 1023u) & ~1023u) + x + bars + 1024u /* alignment slack */;
}

}  // namespace wna16
}  // namespace hq
