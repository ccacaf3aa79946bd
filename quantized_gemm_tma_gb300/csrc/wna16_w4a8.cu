// wna16_w4a8.cu — instantiations and launcher of the WnA16 kernel for
// W4A8-MXFP4: MXFP4 weights against MXFP8 activations, block-scaled MMA
// (dense and MoE grouped, every tile class; own translation unit so the
// formats compile in parallel).
#include "gemm_wna16.cuh"
#include "hq_launch.h"

namespace hq {
namespace {

constexpr int kFmt = static_cast<int>(WFmt::MXFP4_A8);

template <int CLS, bool MOE>
cudaError_t run(const Wna16Launch& l, const GemmParams& p, const Wna16Maps& maps, cudaStream_t stream) {
  auto k = wna16::wna16_kernel<kFmt, true, CLS, MOE>;
  cudaError_t e = ensure_smem_optin(reinterpret_cast<const void*>(k));
  if (e != cudaSuccess) return e;
  return launch_pdl(reinterpret_cast<const void*>(k), l.grid, wna16::threads<CLS>(), l.smem, stream, p.cluster, p,
                    maps.x, maps.y);
}

}  // namespace

cudaError_t launch_wna16_w4a8(const Wna16Launch& l, const GemmParams& p, const Wna16Maps& maps, cudaStream_t stream) {
  if (!l.bf16) return cudaErrorInvalidValue;
  switch (l.cls) {
    case 0: return l.moe ? run<0, true>(l, p, maps, stream) : run<0, false>(l, p, maps, stream);
    case 1: return l.moe ? run<1, true>(l, p, maps, stream) : run<1, false>(l, p, maps, stream);
    case 2: return l.moe ? run<2, true>(l, p, maps, stream) : run<2, false>(l, p, maps, stream);
    case 3: return l.moe ? run<3, true>(l, p, maps, stream) : run<3, false>(l, p, maps, stream);
    case 4: return l.moe ? cudaErrorInvalidValue : run<4, false>(l, p, maps, stream);  // dense only
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace hq

#if defined(HQ_ENABLE_TRACE) || defined(HQ_ENABLE_TRACE_CTA)
// Debug builds only: copy (and optionally clear) the W4A8 kernel's event trace.
extern "C" int hq_trace_read_w4a8(void* dst, size_t bytes, int clear) {
  if (cudaDeviceSynchronize() != cudaSuccess) return 1;
  if (bytes < sizeof(hq::dev::g_trace) + sizeof(hq::dev::g_trace_cta)) return 6;
  if (cudaMemcpyFromSymbol(dst, hq::dev::g_trace, sizeof(hq::dev::g_trace)) != cudaSuccess) return 2;
  if (cudaMemcpyFromSymbol(static_cast<char*>(dst) + sizeof(hq::dev::g_trace), hq::dev::g_trace_cta,
                           sizeof(hq::dev::g_trace_cta)) != cudaSuccess)
    return 5;
  if (clear) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, hq::dev::g_trace) != cudaSuccess) return 3;
    if (cudaMemset(p, 0, sizeof(hq::dev::g_trace)) != cudaSuccess) return 4;
    if (cudaGetSymbolAddress(&p, hq::dev::g_trace_cta) != cudaSuccess) return 3;
    if (cudaMemset(p, 0, sizeof(hq::dev::g_trace_cta)) != cudaSuccess) return 4;
  }
  return 0;
}
#endif
