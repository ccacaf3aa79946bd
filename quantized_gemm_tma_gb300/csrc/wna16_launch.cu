// wna16_launch.cu — format dispatch of the WnA16 kernel launches.
#include "gemm_wna16.cuh"
#include "hq_launch.h"

#include <mutex>

namespace hq {

cudaError_t launch_wna16_int4(const Wna16Launch&, const GemmParams&, const Wna16Maps&, cudaStream_t);
cudaError_t launch_wna16_int6(const Wna16Launch&, const GemmParams&, const Wna16Maps&, cudaStream_t);
cudaError_t launch_wna16_mxfp4(const Wna16Launch&, const GemmParams&, const Wna16Maps&, cudaStream_t);
cudaError_t launch_wna16_nvfp4(const Wna16Launch&, const GemmParams&, const Wna16Maps&, cudaStream_t);
cudaError_t launch_wna16_mxint4(const Wna16Launch&, const GemmParams&, const Wna16Maps&, cudaStream_t);
cudaError_t launch_wna16_w4a8(const Wna16Launch&, const GemmParams&, const Wna16Maps&, cudaStream_t);

cudaError_t launch_wna16(const Wna16Launch& l, const GemmParams& p, const Wna16Maps& maps, cudaStream_t stream) {
  switch (l.fmt) {
    case 0: return launch_wna16_int4(l, p, maps, stream);
    case 1: return launch_wna16_int6(l, p, maps, stream);
    case 2: return launch_wna16_mxfp4(l, p, maps, stream);
    case 3: return launch_wna16_nvfp4(l, p, maps, stream);
    case 4: return launch_wna16_mxint4(l, p, maps, stream);
    case 5: return launch_wna16_w4a8(l, p, maps, stream);
    default: return cudaErrorInvalidValue;
  }
}

uint32_t wna16_smem_bytes(int cls, int w_stages, int x_stages, uint32_t tile_bytes, int bn, int num_experts,
                          bool a8) {
  switch (cls) {
    case 0: return wna16::smem_bytes<0>(w_stages, x_stages, tile_bytes, bn, num_experts, a8);
    case 1: return wna16::smem_bytes<1>(w_stages, x_stages, tile_bytes, bn, num_experts, a8);
    case 2: return wna16::smem_bytes<2>(w_stages, x_stages, tile_bytes, bn, num_experts, a8);
    case 4: return wna16::smem_bytes<4>(w_stages, x_stages, tile_bytes, bn, num_experts, a8);
    default: return wna16::smem_bytes<3>(w_stages, x_stages, tile_bytes, bn, num_experts, a8);
  }
}

bool wna16_cluster_fits(int cls, int w_stages, int x_stages, uint32_t tile_bytes, int bn, bool a8) {
  if (cls == 0) return true;  // bn <= 16: rank 1's sums go to a dedicated buffer
  const uint32_t kps = static_cast<uint32_t>(wna16_kps(cls));
  const uint64_t rings = static_cast<uint64_t>(x_stages) * (a8 ? 1u : 2u) * kps * static_cast<uint32_t>(bn) * 128u +
                         static_cast<uint64_t>(w_stages) * ((kps * tile_bytes + 1023u) & ~1023u);
  const uint32_t need = cls == 1   ? wna16::xchg_bytes<1>()
                        : cls == 2 ? wna16::xchg_bytes<2>()
                        : cls == 4 ? wna16::xchg_bytes<4>()
                                   : wna16::xchg_bytes<3>();
  return need <= rings;
}

int wna16_stream_period(int cls, bool a8) {
  if (cls == 0 || cls == 1 || cls == 4) return 2;  // two K-blocks per stage
  return cls == 2 || (cls == 3 && a8) ? 4 : 1;      // one K-block per stage
}

int wna16_kps(int cls) {
  switch (cls) {
    case 0: return wna16::Cls<0>::kKps;
    case 1: return wna16::Cls<1>::kKps;
    case 2: return wna16::Cls<2>::kKps;
    case 4: return wna16::Cls<4>::kKps;
    default: return wna16::Cls<3>::kKps;
  }
}

cudaError_t ensure_smem_optin(const void* kernel) {
  constexpr int kSlots = 128;
  static const void* funcs[kSlots];
  static uint64_t done[kSlots];  // one bit per device
  static std::mutex mu;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = 1ull << (dev & 63);
  std::lock_guard<std::mutex> lk(mu);
  int i = 0;
  for (; i < kSlots && funcs[i]; ++i)
    if (funcs[i] == kernel) break;
  if (i < kSlots && funcs[i] == kernel && (done[i] & bit)) return cudaSuccess;
  int optin = 0;
  e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, optin);
  if (e != cudaSuccess) return e;
  if (i < kSlots) {
    funcs[i] = kernel;
    done[i] |= bit;
  }
  return cudaSuccess;
}

}  // namespace hq
