// wna16_int6.cu — instantiations and launcher of the WnA16 kernel for
// INT6 weights (kept in their own translation unit so the formats compile
// in parallel).
#include "gemm_wna16.cuh"
#include "hq_launch.h"

namespace hq {
namespace {

template <bool BF16, int CLS, bool MOE>
cudaError_t run(const Wna16Launch& l, const GemmParams& p, const Wna16Maps& maps, cudaStream_t stream) {
  auto k = wna16::wna16_kernel<1, BF16, CLS, MOE>;
  cudaError_t e = ensure_smem_optin(reinterpret_cast<const void*>(k));
  if (e != cudaSuccess) return e;
  return launch_pdl(reinterpret_cast<const void*>(k), l.grid, wna16::threads<CLS>(), l.smem, stream, p.cluster, p,
                    maps.x, maps.y);
}

template <bool BF16, bool MOE>
cudaError_t run_cls(const Wna16Launch& l, const GemmParams& p, const Wna16Maps& maps, cudaStream_t stream) {
  switch (l.cls) {
    case 0: return run<BF16, 0, MOE>(l, p, maps, stream);
    case 1: return run<BF16, 1, MOE>(l, p, maps, stream);
    case 2: return run<BF16, 2, MOE>(l, p, maps, stream);
    case 3: return run<BF16, 3, MOE>(l, p, maps, stream);
    case 4:  // dense only
      if constexpr (!MOE) return run<BF16, 4, false>(l, p, maps, stream);
      return cudaErrorInvalidValue;
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

cudaError_t launch_wna16_int6(const Wna16Launch& l, const GemmParams& p, const Wna16Maps& maps,
                              cudaStream_t stream) {
  if (l.moe) return l.bf16 ? run_cls<true, true>(l, p, maps, stream) : cudaErrorInvalidValue;
  return l.bf16 ? run_cls<true, false>(l, p, maps, stream)
                : run_cls<false, false>(l, p, maps, stream);
}

}  // namespace hq
