// mxfp8.cuh — the MXFP8 conversion of activations (OCP Microscaling v1.0:
// e4m3 elements under one UE8M0 exponent per 32 along K), shared by the
// standalone quantiser and the quantising MoE gather.
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
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace hq {
namespace dev {

// Eight consecutive bf16 of a row (raw, element 2i in the low half of word i)
// -> eight e4m3 bytes in order, and the UE8M0 exponent E of the 32-element
// block that four consecutive lanes 4b .. 4b+3 hold.  Every lane of the warp
// calls it (a lane without data passes zeros).
__device__ __forceinline__ uint2 mxfp8_quantize8(const uint4 raw, int* e_out) {
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
  amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
  amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
  const int ef = static_cast<int>((__float_as_uint(amax) >> 23) & 0xFFu);  // exponent field of the block maximum
  const int E = ef == 0 ? 0 : min(max(ef - 8, 0), 254);
  // 2^(127 - E): normal for every E a finite bf16 block gives (E <= 246)
  const float scale = __uint_as_float(static_cast<uint32_t>(254 - E) << 23);
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
  *e_out = E;
  return make_uint2(packed[0], packed[1]);
}

}  // namespace dev
}  // namespace hq
