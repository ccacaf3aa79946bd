// noalloc.cu — hq_gemm_noalloc: the dense GEMM with the library's own fixed
// device scratch in place of a caller workspace.
//
// The scratch is one file-scope device array, zero at module load, so the
// split-K counters it holds start at zero; every call that completes leaves
// them at zero again.  Its device address is looked up with
// cudaGetSymbolAddress once per device and CUDA context (the first call made
// with that device current, and again after that device's context has been
// destroyed and recreated, since the module, and with it the array, may then
// sit elsewhere); after that a call does no set-up work and allocates
// nothing, neither host nor device memory.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "hq.h"
#include "hq_internal.h"

namespace {

constexpr size_t kScratchBytes = HQ_NOALLOC_SCRATCH_BYTES;
// status word and split-K / stream-K counters at the head of the scratch:
// what HQ_FLAG_NOALLOC_RESET clears
constexpr size_t kResetBytes = hq::kWsStatusBytes + hq::kWsCounterBytes;

// status word (first 256 bytes), split-K counters, fp32 split-K partials
static __device__ __align__(256) unsigned char g_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
struct ScratchSlot {
  void* ptr = nullptr;
  unsigned long long ctx_id = 0;  // unique id of the context the address belongs to
};
ScratchSlot g_slot[kMaxDevices];
std::mutex g_scratch_mu;

using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);
CtxGetCurrentFn g_ctx_current = nullptr;
CtxGetIdFn g_ctx_id = nullptr;
std::once_flag g_ctx_fns_once;

// Unique id of the context current on this thread (0 if there is none yet or
// the driver entry points are unavailable; the caller then re-resolves).
unsigned long long current_ctx_id() {
  std::call_once(g_ctx_fns_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &fn, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_ctx_current = reinterpret_cast<CtxGetCurrentFn>(fn);
    fn = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &fn, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_ctx_id = reinterpret_cast<CtxGetIdFn>(fn);
  });
  if (!g_ctx_current || !g_ctx_id) return 0;
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (g_ctx_current(&ctx) != CUDA_SUCCESS || !ctx) return 0;
  if (g_ctx_id(ctx, &id) != CUDA_SUCCESS) return 0;
  return id;
}

// Device address of g_scratch for the current device and context.
hq_status scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return HQ_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_scratch_mu);
  ScratchSlot& s = g_slot[dev];
  const unsigned long long id = current_ctx_id();
  if (!s.ptr || id == 0 || id != s.ctx_id) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_scratch) != cudaSuccess || !p) return HQ_ERR_CUDA;
    s.ptr = p;
    // the lookup has made the device's primary context current if it was not
    s.ctx_id = id != 0 ? id : current_ctx_id();
  }
  *out = s.ptr;
  return HQ_OK;
}

}  // namespace

extern "C" hq_status hq_gemm_noalloc(const hq_weight_desc* wdesc, const void* w_t, int32_t m, int32_t atype,
                                     const void* x, int64_t ldx, const void* x_scales, void* y, int64_t ldy,
                                     uint32_t flags, int32_t* device_status, hq_stream_t stream) {
  if (!wdesc || m < 0) return HQ_ERR_INVALID_ARG;
  const bool reset = (flags & HQ_FLAG_NOALLOC_RESET) != 0;
  flags &= ~HQ_FLAG_NOALLOC_RESET;
  // the size any sm_103 device could plan for this problem must fit the scratch
  size_t need = 0;
  hq_status st = hq_gemm_workspace_size(wdesc, m, atype, &need);
  if (st != HQ_OK) return st;
  if (need > kScratchBytes) return HQ_ERR_WORKSPACE_TOO_SMALL;
  if (m == 0) return hq_gemm(wdesc, w_t, 0, atype, x, ldx, x_scales, y, ldy, nullptr, 0, flags, stream);
  void* scratch = nullptr;
  st = scratch_address(&scratch);
  if (st != HQ_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (reset && cudaMemsetAsync(scratch, 0, kResetBytes, s) != cudaSuccess) return HQ_ERR_CUDA;
  st = hq_gemm(wdesc, w_t, m, atype, x, ldx, x_scales, y, ldy, scratch, kScratchBytes, flags, stream);
  if (st != HQ_OK) return st;
  if (device_status) {
    // the status word is sticky: it is copied out, cleared only by a reset
    if (cudaMemcpyAsync(device_status, scratch, sizeof(int32_t), cudaMemcpyDeviceToDevice, s) != cudaSuccess)
      return HQ_ERR_CUDA;
  }
  return HQ_OK;
}
