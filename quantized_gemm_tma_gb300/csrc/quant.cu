// quant.cu — activation quantisation to MXFP8 for the W4A8-MXFP4 product:
// e4m3 elements under one UE8M0 exponent per 32 along K (OCP Microscaling
// v1.0 conversion; the Humming launch article's W4A8-MXFP4 paragraph pairs
// MXFP4 weights with 8-bit floating-point activations).
//
//   E  = clamp(floor(log2(max |x| of the block)) - 8 + 127, 0, 254)
//        (8 is the largest exponent of a normal e4m3 value; an all-zero
//        block gives 0)
//   q  = e4m3(x / 2^(E - 127)), round to nearest even, saturating at 448
//
// For bf16 inputs the block maximum is exact in fp32 and floor(log2) is its
// exponent field less the bias (a maximum that is zero or an fp32 subnormal
// gives E = 0 after the clamp).  The scale is an exact power of two, so each
// code is decided on the exact value; a product that underflows fp32 is far
// below half the smallest e4m3 subnormal and rounds to a signed zero either
// way.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "hq_launch.h"

namespace hq {
namespace {

// One thread per 8 consecutive elements of a row; the four threads of a
// 32-element block are consecutive lanes (K % 32 == 0, so no block straddles
// two rows).
__global__ void __launch_bounds__(256) mxfp8_quantize_kernel(const __nv_bfloat16* __restrict__ x, int64_t ldx,
                                                             int m, int k, uint8_t* __restrict__ q, int64_t ldq,
                                                             uint8_t* __restrict__ e, int64_t lde) {
  const int per_row = k / 8;
  const int64_t idx = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const bool live = idx < static_cast<int64_t>(m) * per_row;
  const int row = live ? static_cast<int>(idx / per_row) : 0;
  const int j = live ? static_cast<int>(idx - static_cast<int64_t>(row) * per_row) : 0;
  uint4 raw = make_uint4(0, 0, 0, 0);
  if (live) raw = *reinterpret_cast<const uint4*>(x + static_cast<int64_t>(row) * ldx + 8 * j);
  const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
  float v[8];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    v[2 * i] = __uint_as_float(w[i] << 16);            // element 2i (low half)
    v[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);  // element 2i + 1
  }
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(v[i]));
  // block of 32 = lanes 4b .. 4b+3 (every lane takes part, dead ones with 0)
  amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
  amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
  const int ef = static_cast<int>((__float_as_uint(amax) >> 23) & 0xFFu);  // exponent field of the block maximum
  const int E = ef == 0 ? 0 : min(max(ef - 8, 0), 254);
  const float scale = __uint_as_float(static_cast<uint32_t>(254 - E) << 23);  // 2^(127 - E), normal for E <= 253
  uint32_t packed[2];
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    uint32_t word = 0;
#pragma unroll
    for (int p = 0; p < 2; ++p) {
      const float lo = v[4 * h + 2 * p] * scale, hi = v[4 * h + 2 * p + 1] * scale;
      uint16_t pair;
      asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(pair) : "f"(hi), "f"(lo));
      word |= static_cast<uint32_t>(pair) << (16 * p);
    }
    packed[h] = word;
  }
  if (live) {
    *reinterpret_cast<uint2*>(q + static_cast<int64_t>(row) * ldq + 8 * j) = make_uint2(packed[0], packed[1]);
    if ((j & 3) == 0) e[static_cast<int64_t>(row) * lde + j / 4] = static_cast<uint8_t>(E);
  }
}

}  // namespace

cudaError_t launch_mxfp8_quantize(const void* x, int64_t ldx, int m, int k, void* q, int64_t ldq, void* e,
                                  int64_t lde, cudaStream_t stream) {
  const int64_t threads = static_cast<int64_t>(m) * (k / 8);
  if (threads == 0) return cudaSuccess;
  const int block = 256;
  mxfp8_quantize_kernel<<<static_cast<unsigned>((threads + block - 1) / block), block, 0, stream>>>(
      static_cast<const __nv_bfloat16*>(x), ldx, m, k, static_cast<uint8_t*>(q), ldq, static_cast<uint8_t*>(e), lde);
  return cudaGetLastError();
}

}  // namespace hq
