// wna16_int4.cu — instantiations and launcher of the WnA16 kernel for
// INT4 weights (kept in their own translation unit so the formats compile
// in parallel).
#include "gemm_wna16.cuh"
#include "hq_launch.h"

namespace hq {
namespace {

template <bool BF16, int BN_MAX, bool MOE>
cudaError_t run(const Wna16Launch& l, const GemmParams& p, const CUtensorMap& tmap, const void* x_rows, int64_t ldx,
                cudaStream_t stream) {
  auto k = wna16::wna16_kernel<0, BF16, BN_MAX, MOE>;
  cudaError_t e = ensure_smem_optin(reinterpret_cast<const void*>(k));
  if (e != cudaSuccess) return e;
  k<<<l.grid, wna16::kThreads, l.smem, stream>>>(p, tmap, static_cast<const __nv_bfloat16*>(x_rows), ldx);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_wna16_int4(const Wna16Launch& l, const GemmParams& p, const CUtensorMap& tmap, const void* x_rows,
                             int64_t ldx, cudaStream_t stream) {
  if (l.bf16 == true && l.bn_max == 64 && l.moe == false) return run<true, 64, false>(l, p, tmap, x_rows, ldx, stream);
  if (l.bf16 == true && l.bn_max == 64 && l.moe == true) return run<true, 64, true>(l, p, tmap, x_rows, ldx, stream);
  if (l.bf16 == true && l.bn_max == 256 && l.moe == false) return run<true, 256, false>(l, p, tmap, x_rows, ldx, stream);
  if (l.bf16 == true && l.bn_max == 256 && l.moe == true) return run<true, 256, true>(l, p, tmap, x_rows, ldx, stream);
  if (l.bf16 == false && l.bn_max == 64 && l.moe == false) return run<false, 64, false>(l, p, tmap, x_rows, ldx, stream);
  if (l.bf16 == false && l.bn_max == 256 && l.moe == false) return run<false, 256, false>(l, p, tmap, x_rows, ldx, stream);
  return cudaErrorInvalidValue;
}

}  // namespace hq
