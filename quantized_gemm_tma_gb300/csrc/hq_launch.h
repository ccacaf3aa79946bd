// hq_launch.h — kernel launchers implemented in the .cu files, called by the
// host API (hq_api.cpp).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include "hq_internal.h"

namespace hq {

// Raise a kernel's dynamic shared memory limit to the device maximum, once per
// (kernel, device); later calls are a table lookup.
cudaError_t ensure_smem_optin(const void* kernel);

// Launch with programmatic stream serialization: the grid may begin its
// prologue while the previous grid on the stream finishes; the kernel itself
// waits (griddepcontrol.wait) before it touches global memory.
// `cluster` > 1 launches clusters of that many consecutive CTAs.
template <typename... Args>
cudaError_t launch_pdl(const void* kernel, int grid, int block, uint32_t smem, cudaStream_t stream, int cluster,
                       Args... args) {
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = static_cast<unsigned>(cluster > 1 ? cluster : 1);
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid));
  cfg.blockDim = dim3(static_cast<unsigned>(block));
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = cluster > 1 ? 2 : 1;
  void* argv[] = {static_cast<void*>(&args)...};
  return cudaLaunchKernelExC(&cfg, kernel, argv);
}

// transform.cu
cudaError_t launch_repack(const Layout& L, const hq_weight_desc& d, void* dst, cudaStream_t stream);
cudaError_t launch_unpack(const Layout& L, const void* src, void* codes, void* scales, void* zeros,
                          cudaStream_t stream);

// wna16_*.cu: fmt = WFmt; cls = tile-width class (0: bn <= 16, 1: <= 64,
// 2: <= 128, 3: <= 256, 4: dense <= 128 with one tile per CTA)
struct Wna16Launch {
  int fmt;
  bool bf16;
  int cls;
  bool moe;
  int grid;
  uint32_t smem;
};
// Tensor maps of one WnA16 launch: activations (loads) and Y (dense stores;
// unused when GemmParams::y_tma is 0).
struct Wna16Maps {
  CUtensorMap x, y;
};
cudaError_t launch_wna16(const Wna16Launch& l, const GemmParams& p, const Wna16Maps& maps, cudaStream_t stream);
uint32_t wna16_smem_bytes(int cls, int w_stages, int x_stages, uint32_t tile_bytes, int bn, int num_experts,
                          bool a8 = false);
int wna16_kps(int cls);  // K-blocks per shared-memory stage
// stages between two a dequantiser stream takes (1: no streams); the weight
// ring's depth is a multiple of it
int wna16_stream_period(int cls, bool a8);
// whether a 2-CTA cluster split of this class can pass rank 1's sums through
// rank 0's ring area
bool wna16_cluster_fits(int cls, int w_stages, int x_stages, uint32_t tile_bytes, int bn, bool a8 = false);

// gemm_fp8.cu
cudaError_t launch_fp8(const Fp8Params& p, const CUtensorMap& tmap, int bn_max, int grid, uint32_t smem,
                       cudaStream_t stream);
uint32_t fp8_smem_bytes(int stages, int bn);

// selftest.cu: one CTA whose bounded wait runs out and records HQ_ERR_DEVICE_TIMEOUT in *status
cudaError_t launch_wait_timeout(int* status, cudaStream_t stream);

// quant.cu: x bf16 [m][ldx] -> e4m3 codes [m][ldq] and UE8M0 exponents [m][lde] (k % 32 == 0)
cudaError_t launch_mxfp8_quantize(const void* x, int64_t ldx, int m, int k, void* q, int64_t ldq, void* e,
                                  int64_t lde, cudaStream_t stream);

// moe.cu
// Routing of more than kRouteSinglePairs pairs runs on up to kRouteMaxBlocks
// blocks of about kRoutePairsPerBlock pairs each, through an int32 table of
// per-block expert counts [blocks][E] in the workspace (`counts`).
constexpr int kRouteSinglePairs = 8192;
constexpr int kRouteMaxBlocks = 128;
constexpr int kRoutePairsPerBlock = 2048;
int moe_route_blocks(int pairs);
cudaError_t launch_moe_route(const int* topk_ids, int pairs, int num_experts, int bn, int* expert_offsets,
                             int* tile_offsets, int* perm, int* offsets_out, int* perm_out, int* counts, int* status,
                             cudaStream_t stream);
cudaError_t launch_moe_grouped_route(const int* rows_in, bool masked, int rows, int num_experts, int bn,
                                     int* expert_offsets, int* tile_offsets, int* perm, int* x_base, int* status,
                                     cudaStream_t stream);
// Xg[p][:k] = X[perm[p] / topk][:k] for p < *routed (a device count of at
// most `pairs`); bf16, k, ldx and ldg multiples of 8
cudaError_t launch_moe_permute(const void* x, int64_t ldx, int tokens, const int* perm, const int* routed,
                               int pairs, int topk, int k, void* xg, int64_t ldg, int sms, cudaStream_t stream);
// W4A8: the same gather quantised to MXFP8, Q[p][:k] e4m3 and Ex[p][:k/32]
// UE8M0 (k % 32 == 0; ldx, ldq multiples of 8)
cudaError_t launch_moe_permute_mxfp8(const void* x, int64_t ldx, int tokens, const int* perm, const int* routed,
                                     int pairs, int topk, int k, void* q, int64_t ldq, void* ex, int64_t lde,
                                     cudaStream_t stream);
cudaError_t launch_moe_act(const void* h, int64_t ldh, int pairs, int inter, void* a, int64_t lda,
                           cudaStream_t stream);
cudaError_t launch_moe_combine(const float* zbuf, const int* topk_ids, int tokens, int topk, int num_experts, int n,
                               int n_pad, void* y, int64_t ldy, bool bf16, cudaStream_t stream);

}  // namespace hq
