// quant.cu — activation quantisation to MXFP8 for the W4A8-MXFP4 product:
// e4m3 elements under one UE8M0 exponent per 32 along K (OCP Microscaling
// v1.0 conversion; the Humming launch article's W4A8-MXFP4 paragraph pairs
// MXFP4 weights with 8-bit floating-point activations).  The conversion
// itself is dev::mxfp8_quantize8.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "hq_launch.h"
#include "mxfp8.cuh"

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
  int E = 0;
  const uint2 packed = dev::mxfp8_quantize8(raw, &E);
  if (live) {
    *reinterpret_cast<uint2*>(q + static_cast<int64_t>(row) * ldq + 8 * j) = packed;
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
