// noalloc.cu — hq_gemm_noalloc: the dense GEMM with the library's own fixed
// device scratch in place of a caller workspace.
//
// The scratch is one file-scope device array, zero at module load, so the
// split-K counters it holds start at zero; every call that completes leaves
// them at zero again.  Its address is looked up once per device (the first
// call made with that device current) and cached; after that a call does no
// set-up work and allocates nothing, neither host nor device memory.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "hq.h"

namespace {

constexpr size_t kScratchBytes = HQ_NOALLOC_SCRATCH_BYTES;

// status word (first 256 bytes), split-K counters, fp32 split-K partials
static __device__ __align__(256) unsigned char g_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
void* g_scratch_ptr[kMaxDevices];
std::mutex g_scratch_mu;

// Device address of g_scratch for the current device; the first call per
// device resolves it with cudaGetSymbolAddress.
hq_status scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return HQ_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_scratch_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_scratch) != cudaSuccess || !p) return HQ_ERR_CUDA;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return HQ_OK;
}

}  // namespace

extern "C" hq_status hq_gemm_noalloc(const hq_weight_desc* wdesc, const void* w_t, int32_t m, int32_t atype,
                                     const void* x, int64_t ldx, const float* x_scales, void* y, int64_t ldy,
                                     uint32_t flags, int32_t* device_status, hq_stream_t stream) {
  if (!wdesc || m < 0) return HQ_ERR_INVALID_ARG;
  // the size any sm_103 device could plan for this problem must fit the scratch
  size_t need = 0;
  hq_status st = hq_gemm_workspace_size(wdesc, m, atype, &need);
  if (st != HQ_OK) return st;
  if (need > kScratchBytes) return HQ_ERR_WORKSPACE_TOO_SMALL;
  if (m == 0) return hq_gemm(wdesc, w_t, 0, atype, x, ldx, x_scales, y, ldy, nullptr, 0, flags, stream);
  void* scratch = nullptr;
  st = scratch_address(&scratch);
  if (st != HQ_OK) return st;
  st = hq_gemm(wdesc, w_t, m, atype, x, ldx, x_scales, y, ldy, scratch, kScratchBytes, flags, stream);
  if (st != HQ_OK) return st;
  if (device_status) {
    // the status word is sticky: it is copied out, never cleared
    if (cudaMemcpyAsync(device_status, scratch, sizeof(int32_t), cudaMemcpyDeviceToDevice,
                        static_cast<cudaStream_t>(stream)) != cudaSuccess)
      return HQ_ERR_CUDA;
  }
  return HQ_OK;
}
