// gemm_fp8.cu — W8A8 FP8 GEMM with 128x128 float32 weight block scales and
// per-token, per-128-K-group float32 activation scales ("FP8 W8A8" — Humming
// launch/alphasignal pages; the block-scaled form of the quantized GEMM):
//
//   Y[m, n] = sum_kb  s_x[m, kb] * s_w[n/128, kb] * sum_{k in kb} x[m, k] w[n, k]
//
// The fp32 block scales are not a native tensor-core scale format, so each
// 128-K block is multiplied on the tensor core (tcgen05.mma.kind::f8f6f4,
// e4m3 x e4m3 -> fp32 in TMEM) into a fresh partial, and the epilogue warps
// promote it: acc += s_x * s_w * partial, in registers.  Two TMEM partial
// buffers ping-pong so the MMA of block kb+1 overlaps the promotion of kb.
//
// Orientation: tokens are the MMA M side (TMEM lanes), weights the N side, so
// one thread (one token row) applies a single scalar s_x[m, kb] * s_w[., kb]
// per 128 columns of weights.
//
// Warps: 0 = TMA producer (bulk copy of the pre-swizzled weight image, 2-D
// tensor copy of the activation tile), 1 = TMEM allocator + MMA issuer,
// 2..9 = promotion + epilogue (two warps per TMEM lane quarter, each owning
// half of the columns).
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "hq_internal.h"
#include "hq_launch.h"
#include "hq_ptx.cuh"

namespace hq {
namespace fp8 {

constexpr int kEpiWarps = 8;
constexpr int kThreads = 64 + 32 * kEpiWarps;
constexpr int kTokTile = 128;  // tokens per tile (MMA M)

__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, volatile int* abort) {
  const bool got = dev::mbar_wait(bar, parity, abort);
  return __all_sync(0xffffffffu, got) != 0;
}

// BN = weights per tile (MMA N): 128 or 256 (one or two 128-row weight tiles)
template <int BN>
__global__ void __launch_bounds__(kThreads, 1)
    fp8_kernel(const __grid_constant__ Fp8Params p, const __grid_constant__ CUtensorMap tmap_x) {
  constexpr int kTmemCols = 2 * BN <= 256 ? 256 : 512;
  constexpr int kHalfCols = BN / 2;  // columns per epilogue warp
  constexpr int kNT = BN / 128;      // weight tiles per stage
  extern __shared__ uint8_t smem_raw[];
  // 1024-byte aligned base, derived from smem_raw by an offset so that the
  // compiler keeps shared-memory addressing for every access through it
  uint8_t* smem = smem_raw + ((1024u - (dev::smem_u32(smem_raw) & 1023u)) & 1023u);
  const int S = p.stages;
  constexpr uint32_t kWBytes = 16384u * kNT;
  constexpr uint32_t kXBytes = kTokTile * 128u;
  uint8_t* w_st = smem;
  uint8_t* x_st = smem + S * kWBytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(x_st + S * kXBytes);
  uint64_t* full = bars;
  uint64_t* empty = bars + S;
  uint64_t* p_full = bars + 2 * S;   // [2]
  uint64_t* p_empty = p_full + 2;    // [2]
  uint64_t* tear = p_empty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(tear + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const uint32_t lane = dev::lane_id();
  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      dev::mbar_init(&full[s], 1);
      dev::mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      dev::mbar_init(&p_full[b], 1);
      dev::mbar_init(&p_empty[b], kEpiWarps);
    }
    dev::mbar_init(tear, 1);
    *abort_flag = 0;
    dev::fence_barrier_init();
  }
  if (warp == 1) {
    dev::tmem_alloc(tmem_slot, kTmemCols);
    dev::tmem_relinquish();
  }
  if (warp == 0 && lane == 0) dev::prefetch_tmap(&tmap_x);
  dev::tc_fence_before();
  __syncthreads();
  dev::tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  const int n_groups = p.n_tiles / kNT + (p.n_tiles % kNT ? 1 : 0);
  const int total = p.m_tiles * n_groups * p.splits;
  // work item w -> (split, n group, m tile); split fastest
  auto item_of = [&](int w, int& sp, int& ng, int& mt, int& kb0, int& kb1) {
    sp = w % p.splits;
    const int t = w / p.splits;
    ng = t % n_groups;
    mt = t / n_groups;
    kb0 = sp * p.kb_per_split;
    kb1 = min(p.k_tiles, kb0 + p.kb_per_split);
  };

  if (warp == 0) {
    if (lane == 0) {
      const uint64_t pol = dev::policy_evict_first();
      int it = 0;
      bool ok = true;
      for (int w = blockIdx.x; ok && w < total; w += gridDim.x) {
        int sp, ng, mt, kb0, kb1;
        item_of(w, sp, ng, mt, kb0, kb1);
        for (int kb = kb0; kb < kb1; ++kb, ++it) {
          const int s = it % S;
          if (!dev::mbar_wait(&empty[s], ((it / S) & 1) ^ 1u, abort_flag)) {
            ok = false;
            break;
          }
          uint32_t bytes = kXBytes;
          for (int t = 0; t < kNT; ++t)
            if (ng * kNT + t < p.n_tiles) bytes += 16384u;
          dev::mbar_arrive_expect_tx(&full[s], bytes);
          for (int t = 0; t < kNT; ++t) {
            const int nt = ng * kNT + t;
            if (nt < p.n_tiles)
              dev::bulk_load_hint(w_st + s * kWBytes + t * 16384u,
                                  p.tiles + (static_cast<uint64_t>(nt) * p.k_tiles + kb) * p.tile_bytes, 16384u,
                                  &full[s], pol);
          }
          dev::tma_load_2d(x_st + s * kXBytes, &tmap_x, &full[s], kb * 128, mt * kTokTile);
        }
      }
      if (!ok) dev::raise_error(p.status, abort_flag, HQ_ERR_DEVICE_TIMEOUT);
      for (int s = 0; s < S && s < it; ++s) {
        const int last = ((it - 1 - s) / S) * S + s;
        const uint64_t t0 = dev::globaltimer();
        while (!dev::mbar_try_wait(&full[s], (last / S) & 1) && dev::globaltimer() - t0 < dev::kWaitTimeoutNs) {
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      int it = 0, ip = 0;
      bool ok = true;
      for (int w = blockIdx.x; ok && w < total; w += gridDim.x) {
        int sp, ng, mt, kb0, kb1;
        item_of(w, sp, ng, mt, kb0, kb1);
        for (int kb = kb0; kb < kb1; ++kb, ++it, ++ip) {
          const int s = it % S, b = ip & 1;
          if (!dev::mbar_wait(&full[s], (it / S) & 1, abort_flag) ||
              !dev::mbar_wait(&p_empty[b], ((ip >> 1) & 1) ^ 1u, abort_flag)) {
            ok = false;
            break;
          }
          dev::tc_fence_after();
          const uint32_t xa = dev::smem_u32(x_st + s * kXBytes);
          const uint32_t wa = dev::smem_u32(w_st + s * kWBytes);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            // A = activations [128 tokens x 128 B], B = weights [BN rows x 128 B]; K step 32 bytes
            dev::mma_f8_ss(tmem + b * BN, dev::sw128_desc(xa + kk * 32), dev::sw128_desc(wa + kk * 32), p.idesc,
                           kk > 0 ? 1u : 0u);
          }
          dev::tc_commit(&empty[s]);
          dev::tc_commit(&p_full[b]);
        }
      }
      if (!ok) dev::raise_error(p.status, abort_flag, HQ_ERR_DEVICE_TIMEOUT);
      dev::tc_commit(tear);
      const uint64_t t0 = dev::globaltimer();
      while (!dev::mbar_try_wait(tear, 0) && dev::globaltimer() - t0 < dev::kWaitTimeoutNs) {
      }
    }
  } else {
    const int ew = warp - 2;
    const int quarter = warp & 3;
    const int half = ew >> 2;
    const int row = quarter * 32 + static_cast<int>(lane);   // token row within the tile
    const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
    int ip = 0;
    bool ok = true;
    for (int w = blockIdx.x; ok && w < total; w += gridDim.x) {
      int sp, ng, mt, kb0, kb1;
      item_of(w, sp, ng, mt, kb0, kb1);
      const int m = mt * kTokTile + row;
      const bool m_ok = m < p.m;
      float acc[kHalfCols];
#pragma unroll
      for (int i = 0; i < kHalfCols; ++i) acc[i] = 0.f;
      // this warp's columns [half*kHalfCols, +kHalfCols) lie in weight tile t_own
      const int t_own = (half * kHalfCols) / 128;
      const int nt_own = ng * kNT + t_own;
      for (int kb = kb0; kb < kb1; ++kb, ++ip) {
        const int b = ip & 1;
        const float sx = m_ok ? __ldg(&p.x_scale[static_cast<size_t>(m) * p.k_tiles + kb]) : 0.f;
        const float sw = (nt_own < p.n_tiles) ? __ldg(&p.blk_scale[static_cast<size_t>(nt_own) * p.k_tiles + kb]) : 0.f;
        const float sc = sx * sw;
        if (!warp_wait(&p_full[b], (ip >> 1) & 1, abort_flag)) {
          ok = false;
          break;
        }
        dev::tc_fence_after();
#pragma unroll
        for (int ch = 0; ch < kHalfCols / 16; ++ch) {
          uint32_t v[16];
          dev::tmem_ld16(tmem + lane_base + b * BN + half * kHalfCols + ch * 16, v);
          dev::tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 16; ++i) acc[ch * 16 + i] = fmaf(sc, __uint_as_float(v[i]), acc[ch * 16 + i]);
        }
        dev::tc_fence_before();
        __syncwarp();
        if (lane == 0) dev::mbar_arrive(&p_empty[b]);
      }
      if (!ok) break;
      const int n0 = ng * BN + half * kHalfCols;
      bool write = true;
      if (p.splits > 1) {
        // store this split's fp32 partial; the last of the `splits` warps
        // owning this (rows, columns) slice sums them in split order
        if (m_ok && n0 < p.n_pad) {
          float* dst = p.partials + (static_cast<size_t>(sp) * p.m + m) * p.n_pad + n0;
#pragma unroll
          for (int i = 0; i < kHalfCols; i += 4)
            *reinterpret_cast<float4*>(dst + i) = make_float4(acc[i], acc[i + 1], acc[i + 2], acc[i + 3]);
        }
        __threadfence();
        __syncwarp();
        int* ctr = p.counters + ((mt * n_groups + ng) * kEpiWarps + ew);
        int last = 0;
        if (lane == 0) last = (atomicAdd(ctr, 1) == p.splits - 1) ? 1 : 0;
        last = __shfl_sync(0xffffffffu, last, 0);
        write = last != 0;
        if (last) {
          __threadfence();
          if (m_ok && n0 < p.n_pad) {
#pragma unroll
            for (int i = 0; i < kHalfCols; ++i) acc[i] = 0.f;
            for (int q = 0; q < p.splits; ++q) {
              const float* src = p.partials + (static_cast<size_t>(q) * p.m + m) * p.n_pad + n0;
#pragma unroll
              for (int i = 0; i < kHalfCols; i += 4) {
                const float4 v = __ldcg(reinterpret_cast<const float4*>(src + i));
                acc[i] += v.x; acc[i + 1] += v.y; acc[i + 2] += v.z; acc[i + 3] += v.w;
              }
            }
          }
          if (lane == 0) *ctr = 0;
        }
      }
      if (write && m_ok) {
        __nv_bfloat16* yr = reinterpret_cast<__nv_bfloat16*>(p.y) + static_cast<size_t>(m) * p.ldy;
#pragma unroll
        for (int i = 0; i < kHalfCols; i += 2) {
          const int n = n0 + i;
          if (n + 1 < p.n) {
            *reinterpret_cast<__nv_bfloat162*>(yr + n) = __floats2bfloat162_rn(acc[i], acc[i + 1]);
          } else if (n < p.n) {
            yr[n] = __float2bfloat16_rn(acc[i]);
          }
        }
      }
    }
    if (!ok) dev::raise_error(p.status, abort_flag, HQ_ERR_DEVICE_TIMEOUT);
  }

  dev::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    dev::tc_fence_after();
    dev::tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace fp8

uint32_t fp8_smem_bytes(int stages, int bn) {
  const uint32_t nt = bn <= 128 ? 1u : 2u;
  return static_cast<uint32_t>(stages) * (16384u * nt + fp8::kTokTile * 128u) + (2u * stages + 5u) * 8u + 16u + 1024u;
}

cudaError_t launch_fp8(const Fp8Params& p, const CUtensorMap& tmap, int bn, int grid, uint32_t smem,
                       cudaStream_t stream) {
  if (bn <= 128) {
    auto k = fp8::fp8_kernel<128>;
    cudaError_t e = ensure_smem_optin(reinterpret_cast<const void*>(k));
    if (e != cudaSuccess) return e;
    k<<<grid, fp8::kThreads, smem, stream>>>(p, tmap);
  } else {
    auto k = fp8::fp8_kernel<256>;
    cudaError_t e = ensure_smem_optin(reinterpret_cast<const void*>(k));
    if (e != cudaSuccess) return e;
    k<<<grid, fp8::kThreads, smem, stream>>>(p, tmap);
  }
  return cudaGetLastError();
}

}  // namespace hq
