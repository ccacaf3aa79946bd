// hq_api.cpp — the C ABI declared in include/hq.h: argument validation, the
// tile layout, launch planning ("device-specific heuristics" that pick tile
// width and split-K from M, N, K and the SM count — Humming aiwiki article,
// "Device and workload selection"; launch article, tuning-controls paragraph)
// and kernel launches.  No memory is allocated here.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "hq.h"
#include "hq_internal.h"
#include "hq_launch.h"

namespace hq {
namespace {

constexpr size_t kAlign = 256;
constexpr int kMaxDim = 1 << 28;  // largest N and K (tile counts and offsets stay in 32 bits)
inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }
inline int cdiv(int a, int b) { return (a + b - 1) / b; }

thread_local hq_plan_info g_last_plan{};
thread_local int g_moe_x_stages = 0;  // activation stages of this thread's last grouped MoE launch

// ------------------------------------------------------------------ devices
struct DevInfo {
  bool init = false;
  int cc_major = 0, cc_minor = 0, sms = 0;
  size_t smem_optin = 0;
};
DevInfo g_dev[64];
std::mutex g_dev_mu;

hq_status device_info(DevInfo* out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return HQ_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_dev_mu);
  DevInfo& d = g_dev[dev];
  if (!d.init) {
    int v = 0;
    if (cudaDeviceGetAttribute(&d.cc_major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess) return HQ_ERR_CUDA;
    if (cudaDeviceGetAttribute(&d.cc_minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess) return HQ_ERR_CUDA;
    if (cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return HQ_ERR_CUDA;
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess) return HQ_ERR_CUDA;
    d.smem_optin = static_cast<size_t>(v);
    d.init = true;
  }
  *out = d;
  if (d.cc_major != 10 || d.cc_minor != 3) return HQ_ERR_ARCH;
  return HQ_OK;
}

// ------------------------------------------------------------------ tensor maps
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

// 2-D map {inner, outer} (row stride in elements) with box {box_inner,
// box_outer}; with slabs != 0 a 3-D map that views each row as slabs of
// `inner` columns: low 32 bits of `slabs` = slab count, high 32 bits = slabs
// per box (dims {inner, outer, slabs}, slab stride inner * elem bytes).
hq_status encode_uncached(CUtensorMap* map, CUtensorMapDataType dtype, uint32_t elem, const void* base,
                          uint64_t inner, uint64_t outer, uint64_t row_stride_elems, uint32_t box_inner,
                          uint32_t box_outer, uint64_t slabs, bool swizzle) {
  std::call_once(g_encode_once, [] {
    cudaDriverEntryPointQueryResult q;
    void* fn = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  if (!g_encode) return HQ_ERR_CUDA;
  CUresult r;
  if (slabs == 0) {
    cuuint64_t dims[2] = {inner, outer};
    cuuint64_t strides[1] = {row_stride_elems * elem};
    cuuint32_t box[2] = {box_inner, box_outer};
    cuuint32_t estr[2] = {1, 1};
    r = g_encode(map, dtype, 2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                 swizzle ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                 CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  } else {
    // slabs = (slabs per box << 32) | slab count: the matrix seen as
    // [slab][row][box_inner], slab z starting box_inner elements after slab
    // z - 1, so that one box holds several consecutive slabs of the same rows
    cuuint64_t dims[3] = {box_inner, outer, slabs & 0xffffffffull};
    cuuint64_t strides[2] = {row_stride_elems * elem, static_cast<cuuint64_t>(box_inner) * elem};
    cuuint32_t box[3] = {box_inner, box_outer, static_cast<cuuint32_t>(slabs >> 32)};
    cuuint32_t estr[3] = {1, 1, 1};
    r = g_encode(map, dtype, 3, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                 CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  }
  return r == CUDA_SUCCESS ? HQ_OK : HQ_ERR_CUDA;
}

// Tensor maps depend only on (address, shape, strides, box, type): keep the
// last few per host thread so repeated calls on the same buffers skip the
// driver encode.
struct MapKey {
  const void* base;
  uint64_t inner, outer, stride, slabs;
  uint32_t box_inner, box_outer, dtype, swizzle;
  bool operator==(const MapKey& o) const {
    return base == o.base && inner == o.inner && outer == o.outer && stride == o.stride && slabs == o.slabs &&
           box_inner == o.box_inner && box_outer == o.box_outer && dtype == o.dtype && swizzle == o.swizzle;
  }
};
struct MapCache {
  static constexpr int kSlots = 16;
  MapKey key[kSlots];
  CUtensorMap map[kSlots];
  int used = 0, next = 0;
};
thread_local MapCache g_maps;

// 128-byte swizzled boxes (operand loads) unless `swizzle` is false (plain
// row-major boxes, e.g. output stores staged in shared memory).
hq_status encode_2d(CUtensorMap* map, CUtensorMapDataType dtype, uint32_t elem, const void* base, uint64_t inner,
                    uint64_t outer, uint64_t row_stride_elems, uint32_t box_inner, uint32_t box_outer,
                    uint64_t slabs = 0, bool swizzle = true) {
  const MapKey k{base, inner, outer, row_stride_elems * elem, slabs, box_inner, box_outer, static_cast<uint32_t>(dtype),
                 swizzle ? 1u : 0u};
  MapCache& c = g_maps;
  for (int i = 0; i < c.used; ++i)
    if (c.key[i] == k) {
      *map = c.map[i];
      return HQ_OK;
    }
  hq_status st =
      encode_uncached(map, dtype, elem, base, inner, outer, row_stride_elems, box_inner, box_outer, slabs, swizzle);
  if (st != HQ_OK) return st;
  const int slot = c.used < MapCache::kSlots ? c.used++ : (c.next++ % MapCache::kSlots);
  c.key[slot] = k;
  c.map[slot] = *map;
  return HQ_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int env_int(const char* name, int dflt);

// Activation map of the WnA16 kernel: X [rows][k] in 128-byte slabs (box_inner
// elements) of bn rows.  When k fills whole slabs, one 3-D box carries the
// `per_stage` slabs of a stage (one tensor copy per stage; *x3d = 1); else one
// 2-D box per slab, which zero-fills the columns past k.
hq_status encode_x(CUtensorMap* map, CUtensorMapDataType dtype, uint32_t elem, const void* x, int64_t k,
                   int64_t rows, int64_t ldx, uint32_t box_inner, int bn, int per_stage, int* x3d) {
  *x3d = 0;
  if (k % box_inner == 0 && env_int("HQ_FORCE_X2D", 0) == 0) {
    const uint64_t slabs = (static_cast<uint64_t>(per_stage) << 32) | static_cast<uint64_t>(k / box_inner);
    if (encode_2d(map, dtype, elem, x, k, rows, ldx, box_inner, bn, slabs) == HQ_OK) {
      *x3d = 1;
      return HQ_OK;
    }
  }
  return encode_2d(map, dtype, elem, x, k, rows, ldx, box_inner, bn);
}

// Tiles are counted in 32-bit integers on the device.  `rows` rows in at most
// `groups` separately tiled runs (experts) need at most rows / 16 + groups + 1
// tiles of the narrowest width (16 tokens) per column of output tiles.
bool tiles_fit(int64_t rows, int64_t groups, int n_tiles) {
  return (rows / 16 + groups + 1) * static_cast<int64_t>(n_tiles) <= INT32_MAX;
}

// Tuning and trace switches from the environment, read on first use and
// again by hq_tuning_reload().
struct EnvKnobs {
  int force_bn = 0, force_splitk = 0, force_wstages = 0, force_xstages = 0, force_x2d = 0, trace = 0;
};
EnvKnobs read_env() {
  EnvKnobs e;
  auto get = [](const char* name) {
    const char* v = std::getenv(name);
    return v ? std::atoi(v) : 0;
  };
  e.force_bn = get("HQ_FORCE_BN");
  e.force_splitk = get("HQ_FORCE_SPLITK");
  e.force_wstages = get("HQ_FORCE_WSTAGES");
  e.force_xstages = get("HQ_FORCE_XSTAGES");
  e.force_x2d = get("HQ_FORCE_X2D");
  e.trace = get("HQ_TRACE");
  return e;
}
EnvKnobs g_knobs;
std::once_flag g_knobs_once;
const EnvKnobs& env() {
  std::call_once(g_knobs_once, [] { g_knobs = read_env(); });
  return g_knobs;
}

int env_int(const char* name, int dflt) {
  int v = 0;
  if (!std::strcmp(name, "HQ_FORCE_BN")) v = env().force_bn;
  else if (!std::strcmp(name, "HQ_FORCE_SPLITK")) v = env().force_splitk;
  else if (!std::strcmp(name, "HQ_FORCE_WSTAGES")) v = env().force_wstages;
  else if (!std::strcmp(name, "HQ_FORCE_XSTAGES")) v = env().force_xstages;
  else if (!std::strcmp(name, "HQ_FORCE_X2D")) v = env().force_x2d;
  else if (!std::strcmp(name, "HQ_TRACE")) v = env().trace;
  return v ? v : dflt;
}

}  // namespace

// ------------------------------------------------------------------ layout
hq_status make_layout(const hq_weight_desc& d, Layout* L) {
  if (d.n <= 0 || d.k <= 0 || d.num_experts <= 0) return HQ_ERR_INVALID_ARG;
  if (d.n > kMaxDim || d.k > kMaxDim) return HQ_ERR_UNSUPPORTED;
  if (d.wtype < HQ_W_INT4 || d.wtype > HQ_W_MXINT4) return HQ_ERR_INVALID_ARG;
  if (d.stype < HQ_S_BF16 || d.stype > HQ_S_E4M3) return HQ_ERR_INVALID_ARG;
  std::memset(L, 0, sizeof(*L));
  L->wtype = d.wtype; L->stype = d.stype; L->n = d.n; L->k = d.k; L->num_experts = d.num_experts;
  L->group_k = d.group_k; L->signed_codes = (d.signed_codes || d.wtype == HQ_W_MXINT4) ? 1 : 0;
  L->has_zeros = d.has_zeros ? 1 : 0;
  L->n_tiles = cdiv(d.n, kTileN); L->k_tiles = cdiv(d.k, kTileK);
  L->n_pad = L->n_tiles * kTileN; L->k_pad = L->k_tiles * kTileK;
  const bool is_int = d.wtype == HQ_W_INT4 || d.wtype == HQ_W_INT6;
  if (is_int) {
    if (d.stype != HQ_S_BF16 && d.stype != HQ_S_FP16) return HQ_ERR_INVALID_ARG;
    if (d.group_n != 1 && d.group_n != 0) return HQ_ERR_INVALID_ARG;
    const int g = d.group_k;
    if (g < 0) return HQ_ERR_INVALID_ARG;
    if (g != 0) {
      if (!(g == 32 || g == 64 || g % 128 == 0)) return HQ_ERR_INVALID_ARG;
      if (d.k % g != 0) return HQ_ERR_INVALID_ARG;
    }
    if (d.wtype == HQ_W_INT6 && d.k % 4 != 0) return HQ_ERR_INVALID_ARG;
    L->channel = g == 0;
    L->groups = g == 0 ? 1 : d.k / g;
    L->g_kb = g == 0 ? 0 : (g < 128 ? 128 / g : 1);
  } else if (d.wtype == HQ_W_MXFP4 || d.wtype == HQ_W_MXINT4) {
    if (d.stype != HQ_S_UE8M0 || d.group_k != 32 || d.k % 32 != 0 || d.has_zeros) return HQ_ERR_INVALID_ARG;
    if (d.group_n != 1 && d.group_n != 0) return HQ_ERR_INVALID_ARG;
  } else if (d.wtype == HQ_W_NVFP4) {
    if (d.stype != HQ_S_E4M3 || d.group_k != 16 || d.k % 16 != 0 || d.has_zeros) return HQ_ERR_INVALID_ARG;
    if (d.group_n != 1 && d.group_n != 0) return HQ_ERR_INVALID_ARG;
  } else {
    if (d.stype != HQ_S_FP32 || d.group_k != 128 || d.group_n != 128 || d.has_zeros) return HQ_ERR_INVALID_ARG;
  }
  uint32_t codes = 0, hi = 0, sc = 0, zr = 0;
  switch (d.wtype) {
    case HQ_W_INT4: codes = 8192; break;
    case HQ_W_INT6: codes = 8192; hi = 4096; break;
    case HQ_W_MXFP4:
    case HQ_W_MXINT4: codes = 8192; sc = 512; break;
    case HQ_W_NVFP4: codes = 8192; sc = 1024; break;
    default: codes = 16384; break;
  }
  if (is_int && !L->channel) {
    sc = 256u * L->g_kb;
    if (L->has_zeros) zr = 128u * L->g_kb;
  }
  L->codes_bytes = codes;
  L->hi_off = codes;
  L->scale_off = codes + hi;
  L->scale_bytes = sc;
  L->zero_off = L->scale_off + sc;
  L->zero_bytes = zr;
  L->tile_bytes = L->zero_off + zr;
  L->tiles_off = kHeaderBytes;
  L->expert_stride = static_cast<uint64_t>(L->n_tiles) * L->k_tiles * L->tile_bytes;
  uint64_t off = align_up(L->tiles_off + L->expert_stride * d.num_experts, kAlign);
  if (is_int && L->channel) {
    L->row_off = off;
    off = align_up(off + 4ull * d.num_experts * L->n_pad, kAlign);
    if (L->has_zeros) {
      L->row_zero_off = off;
      off = align_up(off + 1ull * d.num_experts * L->n_pad, kAlign);
    }
  }
  if (d.wtype == HQ_W_FP8_E4M3) {
    L->blk_off = off;
    off = align_up(off + 4ull * d.num_experts * L->n_tiles * L->k_tiles, kAlign);
  }
  if (d.wtype == HQ_W_NVFP4) {
    L->ts_off = off;
    off = align_up(off + 4ull * d.num_experts, kAlign);
  }
  L->total = off;
  return HQ_OK;
}

}  // namespace hq

using namespace hq;

// ====================================================================== C ABI
extern "C" {

int32_t hq_version(void) { return 200; }

const char* hq_status_string(int32_t s) {
  switch (s) {
    case HQ_OK: return "ok";
    case HQ_ERR_INVALID_ARG: return "invalid argument";
    case HQ_ERR_UNSUPPORTED: return "unsupported combination";
    case HQ_ERR_ALIGNMENT: return "pointer or stride not 16-byte aligned";
    case HQ_ERR_WORKSPACE_TOO_SMALL: return "buffer or workspace too small";
    case HQ_ERR_CUDA: return "CUDA runtime error";
    case HQ_ERR_DEVICE_TIMEOUT: return "device-side wait timed out";
    case HQ_ERR_ARCH: return "device is not sm_103";
    case HQ_ERR_INVALID_VALUE: return "invalid value found on the device";
    default: return "unknown status";
  }
}

hq_status hq_transform_size(const hq_weight_desc* desc, size_t* bytes) {
  if (!desc || !bytes) return HQ_ERR_INVALID_ARG;
  Layout L;
  hq_status st = make_layout(*desc, &L);
  if (st != HQ_OK) return st;
  *bytes = L.total;
  return HQ_OK;
}

hq_status hq_transform(const hq_weight_desc* desc, void* dst, size_t dst_bytes, hq_stream_t stream) {
  if (!desc || !dst) return HQ_ERR_INVALID_ARG;
  Layout L;
  hq_status st = make_layout(*desc, &L);
  if (st != HQ_OK) return st;
  if (!desc->codes || !desc->scales || (L.has_zeros && !desc->zeros)) return HQ_ERR_INVALID_ARG;
  if (desc->wtype == HQ_W_NVFP4 && !desc->tensor_scales) return HQ_ERR_INVALID_ARG;
  if (desc->wtype == HQ_W_NVFP4 && (reinterpret_cast<uintptr_t>(desc->tensor_scales) & 3u)) return HQ_ERR_ALIGNMENT;
  if (dst_bytes < L.total) return HQ_ERR_WORKSPACE_TOO_SMALL;
  if ((reinterpret_cast<uintptr_t>(dst) & 255u) != 0) return HQ_ERR_ALIGNMENT;
  if (desc->wtype == HQ_W_FP8_E4M3 && (reinterpret_cast<uintptr_t>(desc->scales) & 3u)) return HQ_ERR_ALIGNMENT;
  if ((desc->wtype == HQ_W_INT4 || desc->wtype == HQ_W_INT6) && (reinterpret_cast<uintptr_t>(desc->scales) & 1u))
    return HQ_ERR_ALIGNMENT;
  DevInfo di;
  st = device_info(&di);
  if (st != HQ_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (launch_repack(L, *desc, dst, s) != cudaSuccess) return HQ_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return HQ_ERR_CUDA;
  TileHeader h;
  if (cudaMemcpy(&h, dst, sizeof(h), cudaMemcpyDeviceToHost) != cudaSuccess) return HQ_ERR_CUDA;
  if (h.magic != kMagic) return HQ_ERR_CUDA;
  return h.invalid_count ? HQ_ERR_INVALID_VALUE : HQ_OK;
}

hq_status hq_untransform(const hq_weight_desc* desc, const void* src, void* codes, void* scales, void* zeros,
                         hq_stream_t stream) {
  if (!desc || !src || !codes || !scales) return HQ_ERR_INVALID_ARG;
  Layout L;
  hq_status st = make_layout(*desc, &L);
  if (st != HQ_OK) return st;
  if ((L.has_zeros || L.wtype == HQ_W_NVFP4) && !zeros) return HQ_ERR_INVALID_ARG;
  DevInfo di;
  st = device_info(&di);
  if (st != HQ_OK) return st;
  if (launch_unpack(L, src, codes, scales, zeros, static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return HQ_ERR_CUDA;
  return HQ_OK;
}

hq_status hq_workspace_init(void* workspace, size_t bytes, hq_stream_t stream) {
  if (!workspace || bytes < kHeaderBytes) return HQ_ERR_INVALID_ARG;
  return cudaMemsetAsync(workspace, 0, bytes, static_cast<cudaStream_t>(stream)) == cudaSuccess ? HQ_OK
                                                                                               : HQ_ERR_CUDA;
}

hq_status hq_status_read(void* workspace, int32_t clear, hq_stream_t stream, int32_t* device_status) {
  if (!workspace || !device_status) return HQ_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(s) != cudaSuccess) return HQ_ERR_CUDA;
  int32_t v = 0;
  if (cudaMemcpy(&v, workspace, sizeof(v), cudaMemcpyDeviceToHost) != cudaSuccess) return HQ_ERR_CUDA;
  *device_status = v;
  if (clear && v != 0) {
    if (cudaMemset(workspace, 0, sizeof(int32_t)) != cudaSuccess) return HQ_ERR_CUDA;
  }
  return HQ_OK;
}

void hq_tuning_reload(void) {
  env();  // the first read has happened, so this one is not overwritten by it
  g_knobs = read_env();
}

hq_status hq_last_plan(hq_plan_info* info) {
  if (!info) return HQ_ERR_INVALID_ARG;
  *info = g_last_plan;
  return HQ_OK;
}

}  // extern "C"

// ====================================================================== GEMM planning
namespace hq {
namespace {

constexpr int kMaxSplits = 64;
constexpr int kPlanSmsBound = 192;  // >= the SM count of any sm_103 part (workspace sizing)
// split-K runs only on problems of at most kMaxSplitTiles output tiles
constexpr size_t kCounterBytes = kWsCounterBytes;
static_assert(kAlign == kWsStatusBytes, "the status region is one alignment unit");

// Tokens per tile of every batch-invariant WnA16 plan (FP8: weight rows).
constexpr int kInvariantBn = 64;
constexpr int kInvariantFp8Bn = 128;

struct DensePlan {
  int cls, bn, m_tiles, tiles, stages, x_stages, groups, grid, stream_k, cluster;
  long long iters;
  uint32_t smem;
};

// FP8: 128 tokens per tile (MMA M), 128 or 256 weight rows (MMA N), split-K
// until the work items fill the SMs.
struct Fp8Plan {
  int bn, m_tiles, n_groups, splits, kb_per_split, stages, grid;
  uint32_t smem;
};

Fp8Plan plan_fp8(const Layout& L, int m, int sms, size_t smem_optin, uint32_t flags) {
  Fp8Plan p{};
  p.m_tiles = cdiv(m, 128);
  const bool inv = (flags & HQ_FLAG_BATCH_INVARIANT) != 0;
  p.bn = inv ? kInvariantFp8Bn : (L.n_tiles >= 2 && p.m_tiles * cdiv(L.n_tiles, 2) >= sms / 2) ? 256 : 128;
  const int forced_bn = env_int("HQ_FORCE_BN", 0);
  if (!inv && (forced_bn == 128 || forced_bn == 256)) p.bn = forced_bn;
  p.n_groups = cdiv(L.n_tiles, p.bn / 128);
  const int tiles = p.m_tiles * p.n_groups;
  int splits = 1;
  if (!(flags & HQ_FLAG_BATCH_INVARIANT) && tiles < sms)
    splits = std::min(std::max(1, sms / tiles), std::max(1, L.k_tiles / 4));
  const int forced = env_int("HQ_FORCE_SPLITK", 0);
  if (forced > 0 && !(flags & HQ_FLAG_BATCH_INVARIANT)) splits = std::min(forced, L.k_tiles);
  splits = std::min(splits, kMaxSplits);
  if (tiles > kMaxSplitTiles) splits = 1;
  p.kb_per_split = cdiv(L.k_tiles, splits);
  p.splits = cdiv(L.k_tiles, p.kb_per_split);
  const size_t budget = std::min<size_t>(smem_optin, 232448) - 4096;
  const uint32_t per_stage = 16384u * (p.bn / 128) + 16384u;
  p.stages = std::max(2, static_cast<int>(std::min<size_t>(6, budget / per_stage)));
  p.smem = fp8_smem_bytes(p.stages, p.bn);
  p.grid = std::min(tiles * p.splits, sms);
  return p;
}

// Split-K scratch: a counter region of fixed size right after the status word
// (8 counters per split tile, at most kMaxSplitTiles tiles), then the fp32
// partials.  The fixed offset keeps one problem's partials off another
// problem's counters when a workspace is reused across shapes.
// Stream-K scratch: the counter region, then a head and a tail partial
// [bn][128] fp32 per CTA.
size_t streamk_bytes(int grid, int bn) {
  return kCounterBytes + align_up(sizeof(float) * 2ull * grid * bn * kTileN, kAlign);
}

size_t splitk_bytes(int splits, int m, int n_pad) {
  if (splits <= 1) return 0;
  return kCounterBytes + align_up(sizeof(float) * static_cast<size_t>(splits) * m * n_pad, kAlign);
}

// Shared-memory rings for a tile-width class: a few activation stages (the
// MMA holds them), then as many weight stages as fit, up to 8.  Tiles of 256
// tokens take three activation stages (192 KB for bf16) and leave the
// weights two: one 128 x 256 x 128 MMA block (about 0.65 us on one SM) does
// not cover the L2 latency of the next 64 KB stage behind a single one.
void plan_stages(int cls, const Layout& L, int bn, int num_experts, size_t smem_optin, int* w_stages,
                 int* x_stages, int* groups, bool a8 = false) {
  const size_t cap = std::min<size_t>(smem_optin, 232448);
  static const int kXWant[5] = {6, 3, 3, 3, 2};
  // sweep overrides (clamped to [2, 12] and to what fits)
  const int fx = env_int("HQ_FORCE_XSTAGES", 0), fw = env_int("HQ_FORCE_WSTAGES", 0);
  int sx = fx >= 2 ? std::min(fx, 12) : kXWant[cls], sw = 0;
  const int sw_max = fw >= 2 ? std::min(fw, 12) : 8;
  // A dequantiser stream waits only on the stages it takes (every second with
  // two K-blocks per stage, every fourth for 128-token tiles with one K-block
  // per stage and W4A8 256-token tiles), so every
  // slot of the weight ring must always hold stages of one residue, i.e. a
  // ring depth that is a multiple of that period.  Otherwise a slot cycles
  // through residues and a stream's parity wait on it could pass one phase
  // early, while another stream's copy is still landing.
  const int sw_step = wna16_stream_period(cls, a8);
  // W4A8 256-token tiles refill an activation slot on the A-slot release of
  // the stream that read it, and their streams wait for the stage's
  // activations themselves: parity waits that need a ring of exactly four
  // stages
  const bool x4 = cls == 3 && a8;
  if (x4) sx = 4;
  const int sx_min = x4 ? 4 : 2;
  const int sw_top = std::max(sw_step, sw_max - sw_max % sw_step);
  for (; sx >= sx_min; --sx) {
    for (sw = sw_top; sw >= 2; sw -= sw_step)
      if (wna16_smem_bytes(cls, sw, sx, L.tile_bytes, bn, num_experts, a8) <= cap) break;
    if (sw >= 2) break;
  }
  *w_stages = sw >= 2 && sx >= 2 ? sw : 0;
  *x_stages = sx;
  *groups = wna16_kps(cls);
}

int wna16_class(int bn) { return bn <= 16 ? 0 : (bn <= 64 ? 1 : (bn <= 128 ? 2 : 3)); }

// WFmt of a weight type handled by the WnA16 kernel
int wna16_fmt(int wtype) {
  switch (wtype) {
    case HQ_W_INT4: return static_cast<int>(WFmt::INT4);
    case HQ_W_INT6: return static_cast<int>(WFmt::INT6);
    case HQ_W_NVFP4: return static_cast<int>(WFmt::NVFP4);
    case HQ_W_MXINT4: return static_cast<int>(WFmt::MXINT4);
    default: return static_cast<int>(WFmt::MXFP4);
  }
}

// Heuristic for one GB300: tokens per tile from M; problems with fewer than
// four tiles per SM are split stream-K so every SM streams the same number
// of weight K-blocks.
DensePlan plan_wna16(const Layout& L, int m, int sms, size_t smem_optin, uint32_t flags, bool a8 = false) {
  DensePlan p{};
  // Batch invariance: one configuration for every M (64-token tiles of the
  // two-K-block class, whose two issuers accumulate even and odd K-blocks
  // and are summed in that order; group scales folded into the operand; no
  // K split), so a row's result does not depend on the other rows.
  const bool inv = (flags & HQ_FLAG_BATCH_INVARIANT) != 0;
  p.bn = inv ? kInvariantBn : m <= 64 ? std::max(16, cdiv(m, 16) * 16) : (m <= 128 ? 128 : (m <= 192 ? 192 : 256));
  const int forced_bn = env_int("HQ_FORCE_BN", 0);
  if (!inv && forced_bn >= 16 && forced_bn % 16 == 0 && forced_bn <= 256) p.bn = forced_bn;
  p.cls = wna16_class(p.bn);
  p.m_tiles = cdiv(m, p.bn);
  p.tiles = p.m_tiles * L.n_tiles;
  p.iters = static_cast<long long>(p.tiles) * L.k_tiles;
  p.stream_k = !(flags & HQ_FLAG_BATCH_INVARIANT) && p.tiles < 4 * sms && p.tiles <= kMaxSplitTiles && L.k_tiles > 1;
  // Wide tiles (bn >= 128): once there are half as many tiles as SMs, whole
  // tiles beat stream-K, whose fp32 partial reduction of 64-128 KB per tile
  // costs more than the wave quantisation it removes (N = K = 8192 on GB300:
  // M = 512 56 vs 102 us, M = 1024 119 vs 135 us, M = 2048 228 vs 231 us).
  if (p.cls >= 2 && 2 * p.tiles >= sms) p.stream_k = 0;
  const int forced_sk = env_int("HQ_FORCE_SPLITK", 0);  // 1: stream-K on, 2: off
  if (forced_sk == 1 && !(flags & HQ_FLAG_BATCH_INVARIANT) && p.tiles <= kMaxSplitTiles) p.stream_k = 1;
  if (forced_sk == 2) p.stream_k = 0;
  plan_stages(p.cls, L, p.bn, 0, smem_optin, &p.stages, &p.x_stages, &p.groups, a8);
  // A tile per 2-CTA cluster, K split in halves and combined through
  // distributed shared memory, when that fills most SMs: no cross-CTA global
  // reduction at all.
  p.cluster = 1;
  if (!(flags & HQ_FLAG_BATCH_INVARIANT) && L.k_tiles >= 2 && 2 * p.tiles <= sms && 8 * p.tiles >= 3 * sms &&
      env_int("HQ_FORCE_SPLITK", 0) == 0 && wna16_cluster_fits(p.cls, p.stages, p.x_stages, L.tile_bytes, p.bn, a8)) {
    p.cluster = 2;
    p.stream_k = 0;
  }
  // 128-token tiles with one tile per CTA: the stream class with two K-blocks
  // per stage (class 4) for 16-bit activations; W4A8 keeps class 2, whose
  // streams take one K-block per stage (N = K = 8192, M = 128: 23.1 against
  // 23.9 us; bf16 25.4 against 24.8 us)
  if (p.cls == 2 && !a8 && (p.cluster == 2 || (!p.stream_k && p.tiles <= sms))) {
    int st4 = 0, sx4 = 0, g4 = 0;
    plan_stages(4, L, p.bn, 0, smem_optin, &st4, &sx4, &g4, a8);
    if (st4 >= 2 && (p.cluster != 2 || wna16_cluster_fits(4, st4, sx4, L.tile_bytes, p.bn, a8))) {
      p.cls = 4;
      p.stages = st4;
      p.x_stages = sx4;
      p.groups = g4;
    }
  }
  p.smem = wna16_smem_bytes(p.cls, p.stages, p.x_stages, L.tile_bytes, p.bn, 0, a8);
  // stream-K: at least 8 K-blocks per CTA, so that partial tiles stay few
  p.grid = p.cluster == 2 ? 2 * p.tiles
           : p.stream_k ? static_cast<int>(std::min<long long>(sms, std::max<long long>(1, (p.iters + 7) / 8)))
                        : std::min(sms, p.tiles);
  return p;
}

// Tokens per expert tile, from the mean routed rows per expert: 16 (the
// decode class) up to a mean of 1 row, 32 up to 8, 64 up to 64, else 128.
// Measured on GB300 (E = 128, N = 1536, K = 2048, top-8, µs per call for
// tiles of 16 / 32 / 64 / 128 / 256 tokens): T = 16 48.1 / 47.4 / 48.8 /
// 61.2 / 99.7, T = 256 121.8 / 89.5 / 86.2 / 106.2 / 190.6, T = 4096
// 1166 / 647 / 428 / 375 / 521.
int moe_tile_bn(double mean_rows) {
  int bn = mean_rows <= 1 ? 16 : mean_rows <= 8 ? 32 : mean_rows <= 64 ? 64 : 128;
  const int forced_bn = env_int("HQ_FORCE_BN", 0);
  if (forced_bn >= 16 && forced_bn % 16 == 0 && forced_bn <= 256) bn = forced_bn;
  return bn;
}

// The gated feed-forward output's gate buffer: one [128 tokens][128 rows]
// fp32 block per CTA (tiles of at most 128 tokens), for any sm_103 SM count.
constexpr int kGateBufBn = 128;
constexpr size_t kGateBufBytes = sizeof(float) * kPlanSmsBound * kGateBufBn * kTileN;

// The grouped WnA16 GEMM over routed rows whose offsets, m-tile prefix, row
// map and X row bases are already in the workspace.  The routed rows of expert
// e stand together in X from row x_base[e] on (the permuted activations of the
// indexed form, the caller's rows of the grouped forms); each unit loads whole
// tiles of them.  Routed position p of expert e's group writes, by `out`: the
// weighted fp32 row zbuf[perm[p]] (indexed form, combined afterwards), the
// 16-bit Y row perm[p] (grouped forms), or the 16-bit Y row p (routed order).
hq_status launch_moe_grouped(const Layout& L, const uint8_t* wt, int bn, const void* x, int64_t ldx, int x_rows,
                             const int* x_base, int out, const float* topk_w, void* y, int64_t ldy,
                             const int* exp_off, const int* tile_off, const int* perm, float* zbuf, int* status,
                             const DevInfo& di, cudaStream_t s, int* stages, int* groups,
                             float* gate_buf = nullptr, const uint8_t* x_mx = nullptr, int64_t ld_mx = 0) {
  // W4A8: x holds MXFP8 codes [x_rows][ldx bytes] and x_mx their UE8M0
  // exponents [x_rows][ld_mx]
  const bool a8 = x_mx != nullptr;
  if (a8 && (L.wtype != HQ_W_MXFP4 || L.k % kTileK != 0 || ld_mx % 4 != 0 || out == kMoeOutGated))
    return HQ_ERR_UNSUPPORTED;
  const int cls = wna16_class(bn);
  GemmParams p{};
  p.tiles = wt + L.tiles_off;
  p.expert_stride = L.expert_stride;
  p.tile_bytes = L.tile_bytes; p.hi_off = L.hi_off; p.scale_off = L.scale_off; p.zero_off = L.zero_off;
  p.g_kb = L.g_kb; p.group_k = L.group_k; p.has_zeros = L.has_zeros; p.channel = L.channel;
  p.zero_sym = (L.has_zeros || !L.signed_codes) ? 0 : (L.wtype == HQ_W_INT4 ? 8 : 32);
  p.row_scale = L.channel ? reinterpret_cast<const float*>(wt + L.row_off) : nullptr;
  p.row_zero = (L.channel && L.has_zeros) ? wt + L.row_zero_off : nullptr;
  p.tensor_scale = L.wtype == HQ_W_NVFP4 ? reinterpret_cast<const float*>(wt + L.ts_off) : nullptr;
  p.n = L.n; p.n_pad = L.n_pad; p.k = L.k; p.k_tiles = L.k_tiles; p.n_tiles = L.n_tiles; p.m = x_rows;
  // m_tiles: whether an expert's weights are, on average, read by more than one
  // tile row (their copies are then kept in L2 for the next row)
  p.bn = bn; p.num_tiles = 0; p.stream_k = 0; p.iters = 0; p.cluster = 1;
  p.m_tiles = static_cast<int64_t>(x_rows) > static_cast<int64_t>(L.num_experts) * bn ? 2 : 1;
  p.idesc = a8 ? idesc_mx_e4m3(128, bn) : idesc_f16(true, 128, bn);
  p.x_mx = x_mx;
  p.ld_mx = static_cast<int>(ld_mx);
  p.y = y; p.ldy = ldy; p.moe_out = out;
  p.status = status;
  p.num_experts = L.num_experts; p.topk = 1;
  p.tile_offsets = tile_off; p.expert_offsets = exp_off; p.perm = perm; p.topk_w = topk_w; p.zbuf = zbuf;
  p.x_base = x_base;
  p.gate_buf = gate_buf;
  if (out == kMoeOutGated && (!gate_buf || di.sms > kPlanSmsBound || bn > kGateBufBn)) return HQ_ERR_UNSUPPORTED;
  plan_stages(cls, L, bn, L.num_experts, di.smem_optin, &p.stages, &p.x_stages, &p.groups, a8);
  if (p.stages < 2) return HQ_ERR_UNSUPPORTED;
  Wna16Launch l{};
  l.fmt = a8 ? static_cast<int>(WFmt::MXFP4_A8) : wna16_fmt(L.wtype);
  l.bf16 = true;
  l.cls = cls;
  l.moe = true;
  l.grid = di.sms;
  l.smem = wna16_smem_bytes(cls, p.stages, p.x_stages, L.tile_bytes, bn, L.num_experts, a8);
  // X [x_rows][K]: slabs of 128 bytes (64 bf16 or 128 e4m3 columns, swizzled) of bn rows
  Wna16Maps maps;
  hq_status st = a8 ? encode_x(&maps.x, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, x, L.k, x_rows, ldx, 128, bn,
                               wna16_kps(cls), &p.x3d)
                    : encode_x(&maps.x, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, x, L.k, x_rows, ldx, 64, bn,
                               2 * wna16_kps(cls), &p.x3d);
  if (st != HQ_OK) return st;
  maps.y = maps.x;  // MoE output rows use plain stores
  if (launch_wna16(l, p, maps, s) != cudaSuccess) return HQ_ERR_CUDA;
  *stages = p.stages;
  *groups = p.groups;
  g_moe_x_stages = p.x_stages;
  return HQ_OK;
}

// Row pitch (elements) of the permuted activations: K rounded up to 8 bf16
// (16 bytes, the tensor-map stride rule).
inline int64_t permuted_ld(int k) { return (static_cast<int64_t>(k) + 7) / 8 * 8; }

}  // namespace
}  // namespace hq

extern "C" {

hq_status hq_gemm_workspace_size(const hq_weight_desc* desc, int32_t m, int32_t atype, size_t* bytes) {
  if (!desc || !bytes || m < 0) return HQ_ERR_INVALID_ARG;
  if (atype < HQ_A_BF16 || atype > HQ_A_MXFP8_E4M3) return HQ_ERR_INVALID_ARG;
  Layout L;
  hq_status st = make_layout(*desc, &L);
  if (st != HQ_OK) return st;
  if (m > (1 << 30) || !tiles_fit(m, 0, L.n_tiles)) return HQ_ERR_UNSUPPORTED;
  size_t ws = kAlign;  // status word
  if (m > 0) {
    // split-K scratch of the largest plan any sm_103 device would choose
    size_t best = 0;
    for (int sms = 1; sms <= kPlanSmsBound; sms = sms < 64 ? sms * 2 : sms + 8) {
      if (desc->wtype == HQ_W_FP8_E4M3) {
        const Fp8Plan p = plan_fp8(L, m, sms, 232448, 0);
        best = std::max(best, splitk_bytes(p.splits, m, L.n_pad));
      } else {
        const DensePlan p = plan_wna16(L, m, sms, 232448, 0, atype == HQ_A_MXFP8_E4M3);
        if (p.stream_k) best = std::max(best, streamk_bytes(p.grid, p.bn));
      }
    }
    ws += best;
  }
  *bytes = ws;
  return HQ_OK;
}

hq_status hq_gemm(const hq_weight_desc* wdesc, const void* w_t, int32_t m, int32_t atype, const void* x,
                  int64_t ldx, const void* x_scales, void* y, int64_t ldy, void* workspace, size_t ws_bytes,
                  uint32_t flags, hq_stream_t stream) {
  if (!wdesc || m < 0) return HQ_ERR_INVALID_ARG;
  Layout L;
  hq_status st = make_layout(*wdesc, &L);
  if (st != HQ_OK) return st;
  if (L.num_experts != 1) return HQ_ERR_INVALID_ARG;
  if (atype < HQ_A_BF16 || atype > HQ_A_MXFP8_E4M3) return HQ_ERR_INVALID_ARG;
  if (m == 0) return HQ_OK;
  if (m > (1 << 30) || !tiles_fit(m, 0, L.n_tiles)) return HQ_ERR_UNSUPPORTED;
  if (!w_t || !x || !y || !workspace) return HQ_ERR_INVALID_ARG;
  if (ldx < L.k || ldy < L.n) return HQ_ERR_INVALID_ARG;
  const bool fp8 = L.wtype == HQ_W_FP8_E4M3;
  const bool a8 = atype == HQ_A_MXFP8_E4M3;  // W4A8-MXFP4
  if (fp8 != (atype == HQ_A_FP8_E4M3)) return HQ_ERR_UNSUPPORTED;
  if (a8 && L.wtype != HQ_W_MXFP4) return HQ_ERR_UNSUPPORTED;
  if (a8 && L.k % kTileK != 0) return HQ_ERR_INVALID_ARG;
  if ((fp8 || a8) && !x_scales) return HQ_ERR_INVALID_ARG;
  if ((L.wtype == HQ_W_INT4 || L.wtype == HQ_W_INT6) && !L.channel) {
    if ((L.stype == HQ_S_BF16) != (atype == HQ_A_BF16)) return HQ_ERR_UNSUPPORTED;
  }
  if ((L.wtype == HQ_W_INT4 || L.wtype == HQ_W_INT6) && a8) return HQ_ERR_UNSUPPORTED;
  if ((L.wtype == HQ_W_NVFP4 || L.wtype == HQ_W_MXINT4) && atype != HQ_A_BF16) return HQ_ERR_UNSUPPORTED;
  if (L.wtype == HQ_W_MXFP4 && atype != HQ_A_BF16 && !a8) return HQ_ERR_UNSUPPORTED;
  const uint32_t xelem = (fp8 || a8) ? 1 : 2;
  if (!aligned16(x) || !aligned16(y) || !aligned16(workspace) || (reinterpret_cast<uintptr_t>(w_t) & 255u))
    return HQ_ERR_ALIGNMENT;
  if ((ldx * xelem) % 16 != 0 || (ldy * 2) % 4 != 0) return HQ_ERR_ALIGNMENT;
  if (fp8 && !aligned16(x_scales)) return HQ_ERR_ALIGNMENT;
  if (a8 && (reinterpret_cast<uintptr_t>(x_scales) & 3u)) return HQ_ERR_ALIGNMENT;
  if (ws_bytes < kAlign) return HQ_ERR_WORKSPACE_TOO_SMALL;
  DevInfo di;
  st = device_info(&di);
  if (st != HQ_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  const uint8_t* wt = static_cast<const uint8_t*>(w_t);

  if (fp8) {
    const Fp8Plan pl = plan_fp8(L, m, di.sms, di.smem_optin, flags);
    // the plan this device runs needs at most what hq_gemm_workspace_size reports
    if (ws_bytes < kAlign + splitk_bytes(pl.splits, m, L.n_pad))
      return HQ_ERR_WORKSPACE_TOO_SMALL;
    Fp8Params p{};
    p.tiles = wt + L.tiles_off;
    p.expert_stride = L.expert_stride;
    p.tile_bytes = L.tile_bytes;
    p.blk_scale = reinterpret_cast<const float*>(wt + L.blk_off);
    p.x_scale = static_cast<const float*>(x_scales);
    p.n = L.n; p.n_pad = L.n_pad; p.k_tiles = L.k_tiles; p.n_tiles = L.n_tiles; p.m = m;
    p.bn = pl.bn; p.m_tiles = pl.m_tiles; p.stages = pl.stages;
    p.splits = pl.splits; p.kb_per_split = pl.kb_per_split;
    p.idesc = idesc_e4m3(128, pl.bn);
    p.y = y; p.ldy = ldy;
    p.status = reinterpret_cast<int*>(ws);
    p.counters = reinterpret_cast<int*>(ws + kAlign);
    p.partials = reinterpret_cast<float*>(ws + kAlign + kCounterBytes);
    CUtensorMap tm;
    st = encode_2d(&tm, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, x, L.k, m, ldx, 128, 128);
    if (st != HQ_OK) return st;
    g_last_plan = hq_plan_info{pl.bn, pl.splits, pl.grid, 1, pl.stages, 0, 0, 0};
    if (env_int("HQ_TRACE", 0))
      std::fprintf(stderr, "hq_gemm fp8: m=%d n=%d k=%d bn=%d splits=%d grid=%d stages=%d smem=%u\n", m, L.n, L.k,
                   pl.bn, pl.splits, pl.grid, pl.stages, pl.smem);
    return launch_fp8(p, tm, pl.bn, pl.grid, pl.smem, s) == cudaSuccess ? HQ_OK : HQ_ERR_CUDA;
  }

  const DensePlan pl = plan_wna16(L, m, di.sms, di.smem_optin, flags, a8);
  if (pl.stages < 2) return HQ_ERR_UNSUPPORTED;
  if (ws_bytes < kAlign + (pl.stream_k ? streamk_bytes(pl.grid, pl.bn) : 0)) return HQ_ERR_WORKSPACE_TOO_SMALL;
  GemmParams p{};
  p.tiles = wt + L.tiles_off;
  p.expert_stride = L.expert_stride;
  p.tile_bytes = L.tile_bytes; p.hi_off = L.hi_off; p.scale_off = L.scale_off; p.zero_off = L.zero_off;
  p.g_kb = L.g_kb; p.group_k = L.group_k; p.has_zeros = L.has_zeros; p.channel = L.channel;
  p.zero_sym = (L.has_zeros || !L.signed_codes) ? 0 : (L.wtype == HQ_W_INT4 ? 8 : 32);
  p.row_scale = L.channel ? reinterpret_cast<const float*>(wt + L.row_off) : nullptr;
  p.row_zero = (L.channel && L.has_zeros) ? wt + L.row_zero_off : nullptr;
  p.tensor_scale = L.wtype == HQ_W_NVFP4 ? reinterpret_cast<const float*>(wt + L.ts_off) : nullptr;
  p.n = L.n; p.n_pad = L.n_pad; p.k = L.k; p.k_tiles = L.k_tiles; p.n_tiles = L.n_tiles; p.m = m;
  p.bn = pl.bn; p.m_tiles = pl.m_tiles; p.num_tiles = pl.tiles;
  p.stages = pl.stages; p.x_stages = pl.x_stages; p.groups = pl.groups;
  p.stream_k = pl.stream_k; p.iters = pl.iters; p.cluster = pl.cluster;
  p.idesc = a8 ? idesc_mx_e4m3(128, pl.bn) : idesc_f16(atype == HQ_A_BF16, 128, pl.bn);
  p.x_mx = a8 ? static_cast<const uint8_t*>(x_scales) : nullptr;
  p.ld_mx = L.k / 32;
  p.y = y; p.ldy = ldy;
  p.status = reinterpret_cast<int*>(ws);
  p.counters = reinterpret_cast<int*>(ws + kAlign);
  p.partials = reinterpret_cast<float*>(ws + kAlign + kCounterBytes);
  p.num_experts = 1;
  // X [M][K]: one box = 128 bytes (64 bf16/fp16 or 128 e4m3 columns, swizzled) of bn rows
  const CUtensorMapDataType t16 = atype == HQ_A_FP16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  Wna16Maps maps;
  st = a8 ? encode_x(&maps.x, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, x, L.k, m, ldx, 128, pl.bn, wna16_kps(pl.cls),
                     &p.x3d)
          : encode_x(&maps.x, t16, 2, x, L.k, m, ldx, 64, pl.bn, 2 * wna16_kps(pl.cls), &p.x3d);
  if (st != HQ_OK) return st;
  // Y [M][N]: tensor stores of 16 tokens x 32 output rows when its row pitch
  // is a multiple of 16 bytes (the tensor-map stride rule); plain stores else
  p.y_tma = (ldy * 2) % 16 == 0 ? 1 : 0;
  maps.y = maps.x;
  if (p.y_tma) {
    st = encode_2d(&maps.y, a8 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : t16, 2, y, L.n, m, ldy, 32, 16, 0, false);
    if (st != HQ_OK) return st;
  }
  Wna16Launch l{};
  l.fmt = wna16_fmt(L.wtype);
  l.bf16 = atype != HQ_A_FP16;
  if (a8) l.fmt = static_cast<int>(WFmt::MXFP4_A8);
  l.cls = pl.cls;
  l.moe = false;
  l.grid = pl.grid;
  l.smem = pl.smem;
  g_last_plan = hq_plan_info{pl.bn, pl.cluster == 2 ? 2 : (pl.stream_k ? 0 : 1), pl.grid, 1, pl.stages, pl.cls,
                             pl.groups, pl.x_stages};
  if (env_int("HQ_TRACE", 0))
    std::fprintf(stderr, "hq_gemm: m=%d n=%d k=%d bn=%d cls=%d stream_k=%d grid=%d stages=%d groups=%d smem=%u x3d=%d\n",
                 m, L.n, L.k, pl.bn, pl.cls, pl.stream_k, pl.grid, pl.stages, pl.groups, pl.smem, p.x3d);
  return launch_wna16(l, p, maps, s) == cudaSuccess ? HQ_OK : HQ_ERR_CUDA;
}

hq_status hq_plan_query(const hq_weight_desc* wdesc, int32_t m, int32_t atype, int32_t sms, int64_t smem_optin,
                        uint32_t flags, hq_plan_info* info) {
  if (!wdesc || !info || m < 0 || sms <= 0 || sms > kPlanSmsBound || smem_optin <= 0) return HQ_ERR_INVALID_ARG;
  Layout L;
  hq_status st = make_layout(*wdesc, &L);
  if (st != HQ_OK) return st;
  if (L.num_experts != 1) return HQ_ERR_INVALID_ARG;
  if (atype < HQ_A_BF16 || atype > HQ_A_MXFP8_E4M3) return HQ_ERR_INVALID_ARG;
  if (m > (1 << 30) || !tiles_fit(m, 0, L.n_tiles)) return HQ_ERR_UNSUPPORTED;
  const bool fp8 = L.wtype == HQ_W_FP8_E4M3;
  if (fp8 != (atype == HQ_A_FP8_E4M3)) return HQ_ERR_UNSUPPORTED;
  const bool a8 = atype == HQ_A_MXFP8_E4M3;
  if (a8 && (L.wtype != HQ_W_MXFP4 || L.k % kTileK != 0)) return HQ_ERR_UNSUPPORTED;
  if ((L.wtype == HQ_W_INT4 || L.wtype == HQ_W_INT6) && !L.channel && (L.stype == HQ_S_BF16) != (atype == HQ_A_BF16))
    return HQ_ERR_UNSUPPORTED;
  if ((L.wtype == HQ_W_NVFP4 || L.wtype == HQ_W_MXINT4) && atype != HQ_A_BF16) return HQ_ERR_UNSUPPORTED;
  if (L.wtype == HQ_W_MXFP4 && atype != HQ_A_BF16 && !a8) return HQ_ERR_UNSUPPORTED;
  *info = hq_plan_info{};
  if (m == 0) return HQ_OK;
  const size_t optin = static_cast<size_t>(smem_optin);
  if (fp8) {
    const Fp8Plan pl = plan_fp8(L, m, sms, optin, flags);
    *info = hq_plan_info{pl.bn, pl.splits, pl.grid, 1, pl.stages, 0, 0, 0};
    return HQ_OK;
  }
  const DensePlan pl = plan_wna16(L, m, sms, optin, flags, a8);
  if (pl.stages < 2) return HQ_ERR_UNSUPPORTED;
  *info = hq_plan_info{pl.bn, pl.cluster == 2 ? 2 : (pl.stream_k ? 0 : 1), pl.grid, 1, pl.stages, pl.cls, pl.groups,
                       pl.x_stages};
  return HQ_OK;
}

hq_status hq_selftest_wait_timeout(void* workspace, hq_stream_t stream) {
  if (!workspace) return HQ_ERR_INVALID_ARG;
  if (!aligned16(workspace)) return HQ_ERR_ALIGNMENT;
  DevInfo di;
  hq_status st = device_info(&di);
  if (st != HQ_OK) return st;
  return launch_wait_timeout(static_cast<int*>(workspace), static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? HQ_OK
             : HQ_ERR_CUDA;
}

hq_status hq_moe_plan_query(const hq_weight_desc* wdesc, int32_t tokens, int32_t topk, int32_t sms,
                            int64_t smem_optin, hq_plan_info* info) {
  if (!wdesc || !info || tokens < 0 || topk <= 0 || sms <= 0 || sms > kPlanSmsBound || smem_optin <= 0)
    return HQ_ERR_INVALID_ARG;
  Layout L;
  hq_status st = make_layout(*wdesc, &L);
  if (st != HQ_OK) return st;
  if (L.num_experts > 1024 || L.wtype == HQ_W_FP8_E4M3) return HQ_ERR_UNSUPPORTED;
  const int64_t pairs = static_cast<int64_t>(tokens) * topk;
  if (pairs > (1 << 24) || !tiles_fit(pairs, L.num_experts, L.n_tiles)) return HQ_ERR_UNSUPPORTED;
  *info = hq_plan_info{};
  if (tokens == 0) return HQ_OK;
  const int bn = moe_tile_bn(static_cast<double>(pairs) / L.num_experts);
  const int cls = wna16_class(bn);
  int stages = 0, x_stages = 0, groups = 0;
  plan_stages(cls, L, bn, L.num_experts, static_cast<size_t>(smem_optin), &stages, &x_stages, &groups);
  if (stages < 2) return HQ_ERR_UNSUPPORTED;
  *info = hq_plan_info{bn, 1, sms, 4, stages, cls, groups, x_stages};
  return HQ_OK;
}

hq_status hq_mxfp8_quantize(int32_t m, int32_t k, const void* x, int64_t ldx, void* q, int64_t ldq, void* e,
                            int64_t lde, hq_stream_t stream) {
  if (m < 0 || k <= 0 || k % 32 != 0 || k > kMaxDim) return HQ_ERR_INVALID_ARG;
  if (m == 0) return HQ_OK;
  if (m > (1 << 30)) return HQ_ERR_UNSUPPORTED;
  if (!x || !q || !e || ldx < k || ldq < k || lde < k / 32) return HQ_ERR_INVALID_ARG;
  if (!aligned16(x) || ldx % 8 != 0 || (reinterpret_cast<uintptr_t>(q) & 7u) || ldq % 8 != 0) return HQ_ERR_ALIGNMENT;
  DevInfo di;
  hq_status st = device_info(&di);
  if (st != HQ_OK) return st;
  return launch_mxfp8_quantize(x, ldx, m, k, q, ldq, e, lde, static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? HQ_OK
             : HQ_ERR_CUDA;
}

// ------------------------------------------------------------------ MoE
hq_status hq_moe_workspace_size(const hq_weight_desc* desc, int32_t tokens, int32_t topk, int32_t atype,
                                size_t* bytes) {
  if (!desc || !bytes || tokens < 0 || topk <= 0) return HQ_ERR_INVALID_ARG;
  if (atype < HQ_A_BF16 || atype > HQ_A_MXFP8_E4M3) return HQ_ERR_INVALID_ARG;
  Layout L;
  hq_status st = make_layout(*desc, &L);
  if (st != HQ_OK) return st;
  const size_t pairs = static_cast<size_t>(tokens) * topk;
  size_t ws = kAlign;
  ws += 2 * align_up(sizeof(int) * (L.num_experts + 1), kAlign);
  ws += align_up(sizeof(int) * std::max<size_t>(pairs, 1), kAlign);
  ws += align_up(sizeof(float) * pairs * L.n_pad, kAlign);
  ws += align_up(2 * pairs * static_cast<size_t>(permuted_ld(L.k)), kAlign);  // permuted activations, bf16
  ws += align_up(sizeof(int) * kRouteMaxBlocks * L.num_experts, kAlign);  // routing: per-block expert counts
  *bytes = ws;
  return HQ_OK;
}

hq_status hq_moe_gemm(const hq_weight_desc* wdesc, const void* w_t, int32_t tokens, int32_t topk,
                      const int32_t* topk_ids, const float* topk_w, int32_t atype, const void* x, int64_t ldx,
                      void* y, int64_t ldy, int32_t* expert_offsets_out, int32_t* perm_out, void* workspace,
                      size_t ws_bytes, uint32_t flags, hq_stream_t stream) {
  (void)flags;
  if (!wdesc || tokens < 0 || topk <= 0) return HQ_ERR_INVALID_ARG;
  Layout L;
  hq_status st = make_layout(*wdesc, &L);
  if (st != HQ_OK) return st;
  if (atype < HQ_A_BF16 || atype > HQ_A_MXFP8_E4M3) return HQ_ERR_INVALID_ARG;
  if (L.num_experts > 1024) return HQ_ERR_UNSUPPORTED;
  if (tokens == 0) return HQ_OK;
  if (!w_t || !topk_ids || !topk_w || !x || !y || !workspace) return HQ_ERR_INVALID_ARG;
  if (ldx < L.k || ldy < L.n) return HQ_ERR_INVALID_ARG;
  // W4A8-MXFP4: bf16 activations quantised to MXFP8 as they are gathered
  const bool a8 = atype == HQ_A_MXFP8_E4M3;
  if (atype != HQ_A_BF16 && !a8) return HQ_ERR_UNSUPPORTED;
  if (a8 && (L.wtype != HQ_W_MXFP4 || L.k % kTileK != 0)) return HQ_ERR_UNSUPPORTED;
  if (L.wtype == HQ_W_FP8_E4M3) return HQ_ERR_UNSUPPORTED;
  if ((L.wtype == HQ_W_INT4 || L.wtype == HQ_W_INT6) && !L.channel && L.stype != HQ_S_BF16) return HQ_ERR_UNSUPPORTED;
  if (!aligned16(x) || !aligned16(y) || !aligned16(workspace) || (reinterpret_cast<uintptr_t>(w_t) & 255u))
    return HQ_ERR_ALIGNMENT;
  if ((ldx * 2) % 16 != 0 || (ldy * 2) % 16 != 0 || L.k % 8 != 0) return HQ_ERR_ALIGNMENT;
  const int64_t pairs = static_cast<int64_t>(tokens) * topk;
  if (pairs > (1 << 24) || !tiles_fit(pairs, L.num_experts, L.n_tiles)) return HQ_ERR_UNSUPPORTED;
  size_t need = 0;
  hq_moe_workspace_size(wdesc, tokens, topk, atype, &need);
  if (ws_bytes < need) return HQ_ERR_WORKSPACE_TOO_SMALL;
  DevInfo di;
  st = device_info(&di);
  if (st != HQ_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  const uint8_t* wt = static_cast<const uint8_t*>(w_t);
  size_t off = kAlign;
  int* exp_off = reinterpret_cast<int*>(ws + off);
  off += align_up(sizeof(int) * (L.num_experts + 1), kAlign);
  int* tile_off = reinterpret_cast<int*>(ws + off);
  off += align_up(sizeof(int) * (L.num_experts + 1), kAlign);
  int* perm = reinterpret_cast<int*>(ws + off);
  off += align_up(sizeof(int) * std::max<int64_t>(pairs, 1), kAlign);
  float* zbuf = reinterpret_cast<float*>(ws + off);
  off += align_up(sizeof(float) * static_cast<size_t>(pairs) * L.n_pad, kAlign);
  void* xg = ws + off;  // the routed activation rows in expert order
  const int64_t ldg = permuted_ld(L.k);
  // W4A8: e4m3 rows [pairs][k] then their exponents [pairs][k/32] in the same
  // region (k + k/32 bytes a row, within the 2k of a bf16 row)
  uint8_t* xq = static_cast<uint8_t*>(xg);
  uint8_t* xe = xq + static_cast<size_t>(pairs) * L.k;
  off += align_up(2 * static_cast<size_t>(pairs) * static_cast<size_t>(ldg), kAlign);
  int* counts = reinterpret_cast<int*>(ws + off);

  const int bn = moe_tile_bn(static_cast<double>(pairs) / L.num_experts);
  if (launch_moe_route(topk_ids, static_cast<int>(pairs), L.num_experts, bn, exp_off, tile_off, perm,
                       expert_offsets_out, perm_out, counts, reinterpret_cast<int*>(ws), s) != cudaSuccess)
    return HQ_ERR_CUDA;
  const cudaError_t pe =
      a8 ? launch_moe_permute_mxfp8(x, ldx, tokens, perm, exp_off + L.num_experts, static_cast<int>(pairs), topk, L.k,
                                    xq, L.k, xe, L.k / 32, s)
         : launch_moe_permute(x, ldx, tokens, perm, exp_off + L.num_experts, static_cast<int>(pairs), topk, L.k, xg,
                              ldg, di.sms, s);
  if (pe != cudaSuccess) return HQ_ERR_CUDA;
  int stages = 0, groups = 0;
  st = a8 ? launch_moe_grouped(L, wt, bn, xq, L.k, static_cast<int>(pairs), exp_off, kMoeOutZ, topk_w, y, ldy, exp_off,
                               tile_off, perm, zbuf, reinterpret_cast<int*>(ws), di, s, &stages, &groups, nullptr, xe,
                               L.k / 32)
          : launch_moe_grouped(L, wt, bn, xg, ldg, static_cast<int>(pairs), exp_off, kMoeOutZ, topk_w, y, ldy, exp_off,
                               tile_off, perm, zbuf, reinterpret_cast<int*>(ws), di, s, &stages, &groups);
  if (st != HQ_OK) return st;
  if (launch_moe_combine(zbuf, topk_ids, tokens, topk, L.num_experts, L.n, L.n_pad, y, ldy, true, s) != cudaSuccess)
    return HQ_ERR_CUDA;
  g_last_plan = hq_plan_info{bn, 1, di.sms, 4, stages, wna16_class(bn), groups, g_moe_x_stages};
  return HQ_OK;
}

// MoE feed-forward: layouts of the two expert weights and the sizes they imply.
static hq_status ffn_layouts(const hq_weight_desc* w13, const hq_weight_desc* w2, hq::Layout* L13, hq::Layout* L2,
                             int* inter) {
  using namespace hq;
  if (!w13 || !w2) return HQ_ERR_INVALID_ARG;
  hq_status st = make_layout(*w13, L13);
  if (st != HQ_OK) return st;
  st = make_layout(*w2, L2);
  if (st != HQ_OK) return st;
  if (L13->num_experts != L2->num_experts || L13->n % 2 != 0) return HQ_ERR_INVALID_ARG;
  *inter = L13->n / 2;
  if (L2->k != *inter) return HQ_ERR_INVALID_ARG;
  if (*inter % 8 != 0) return HQ_ERR_ALIGNMENT;
  return HQ_OK;
}

hq_status hq_moe_ffn_workspace_size(const hq_weight_desc* w13, const hq_weight_desc* w2, int32_t tokens,
                                    int32_t topk, size_t* bytes) {
  if (!bytes || tokens < 0 || topk <= 0) return HQ_ERR_INVALID_ARG;
  Layout L13, L2;
  int inter = 0;
  hq_status st = ffn_layouts(w13, w2, &L13, &L2, &inter);
  if (st != HQ_OK) return st;
  const size_t pairs = static_cast<size_t>(tokens) * topk;
  const size_t ldh = align_up(2 * static_cast<size_t>(inter), 8), lda = align_up(static_cast<size_t>(inter), 8);
  size_t ws = kAlign;
  ws += 2 * align_up(sizeof(int) * (L13.num_experts + 1), kAlign);
  ws += align_up(sizeof(int) * std::max<size_t>(pairs, 1), kAlign);
  ws += align_up(2 * pairs * ldh, kAlign);             // H: gate and up, bf16
  ws += align_up(2 * pairs * lda, kAlign);             // A: silu(gate) * up, bf16
  ws += align_up(sizeof(float) * pairs * L2.n_pad, kAlign);  // weighted down-projection rows
  ws += align_up(2 * pairs * static_cast<size_t>(permuted_ld(L13.k)), kAlign);  // permuted activations, bf16
  ws += kGateBufBytes;  // per-CTA gate sums of the fused silu(gate) * up
  ws += align_up(sizeof(int) * kRouteMaxBlocks * L13.num_experts, kAlign);  // routing: per-block expert counts
  *bytes = ws;
  return HQ_OK;
}

hq_status hq_moe_ffn(const hq_weight_desc* w13, const void* w13_t, const hq_weight_desc* w2, const void* w2_t,
                     int32_t tokens, int32_t topk, const int32_t* topk_ids, const float* topk_w, int32_t atype,
                     const void* x, int64_t ldx, void* y, int64_t ldy, void* workspace, size_t ws_bytes,
                     uint32_t flags, hq_stream_t stream) {
  (void)flags;
  if (tokens < 0 || topk <= 0) return HQ_ERR_INVALID_ARG;
  Layout L13, L2;
  int inter = 0;
  hq_status st = ffn_layouts(w13, w2, &L13, &L2, &inter);
  if (st != HQ_OK) return st;
  if (atype < HQ_A_BF16 || atype > HQ_A_MXFP8_E4M3) return HQ_ERR_INVALID_ARG;
  if (L13.num_experts > 1024) return HQ_ERR_UNSUPPORTED;
  if (tokens == 0) return HQ_OK;
  if (!w13_t || !w2_t || !topk_ids || !topk_w || !x || !y || !workspace) return HQ_ERR_INVALID_ARG;
  if (ldx < L13.k || ldy < L2.n) return HQ_ERR_INVALID_ARG;
  if (atype != HQ_A_BF16) return HQ_ERR_UNSUPPORTED;
  for (const Layout* L : {&L13, &L2}) {
    if (L->wtype == HQ_W_FP8_E4M3) return HQ_ERR_UNSUPPORTED;
    if ((L->wtype == HQ_W_INT4 || L->wtype == HQ_W_INT6) && !L->channel && L->stype != HQ_S_BF16)
      return HQ_ERR_UNSUPPORTED;
  }
  if (!aligned16(x) || !aligned16(y) || !aligned16(workspace) || (reinterpret_cast<uintptr_t>(w13_t) & 255u) ||
      (reinterpret_cast<uintptr_t>(w2_t) & 255u))
    return HQ_ERR_ALIGNMENT;
  if ((ldx * 2) % 16 != 0 || (ldy * 2) % 16 != 0 || L13.k % 8 != 0) return HQ_ERR_ALIGNMENT;
  const int64_t pairs = static_cast<int64_t>(tokens) * topk;
  if (pairs > (1 << 24) || !tiles_fit(pairs, L13.num_experts, std::max(L13.n_tiles, L2.n_tiles)))
    return HQ_ERR_UNSUPPORTED;
  size_t need = 0;
  hq_moe_ffn_workspace_size(w13, w2, tokens, topk, &need);
  if (ws_bytes < need) return HQ_ERR_WORKSPACE_TOO_SMALL;
  DevInfo di;
  st = device_info(&di);
  if (st != HQ_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  const int64_t ldh = static_cast<int64_t>(align_up(2 * static_cast<size_t>(inter), 8));
  const int64_t lda = static_cast<int64_t>(align_up(static_cast<size_t>(inter), 8));
  size_t off = kAlign;
  int* exp_off = reinterpret_cast<int*>(ws + off);
  off += align_up(sizeof(int) * (L13.num_experts + 1), kAlign);
  int* tile_off = reinterpret_cast<int*>(ws + off);
  off += align_up(sizeof(int) * (L13.num_experts + 1), kAlign);
  int* perm = reinterpret_cast<int*>(ws + off);
  off += align_up(sizeof(int) * static_cast<size_t>(pairs), kAlign);
  void* hbuf = ws + off;
  off += align_up(2 * static_cast<size_t>(pairs) * ldh, kAlign);
  void* abuf = ws + off;
  off += align_up(2 * static_cast<size_t>(pairs) * lda, kAlign);
  float* zbuf = reinterpret_cast<float*>(ws + off);
  off += align_up(sizeof(float) * static_cast<size_t>(pairs) * L2.n_pad, kAlign);
  void* xg = ws + off;  // the routed activation rows in expert order
  const int64_t ldg = permuted_ld(L13.k);
  off += align_up(2 * static_cast<size_t>(pairs) * static_cast<size_t>(ldg), kAlign);
  float* gate_buf = reinterpret_cast<float*>(ws + off);
  off += kGateBufBytes;
  int* counts = reinterpret_cast<int*>(ws + off);
  const int bn = moe_tile_bn(static_cast<double>(pairs) / L13.num_experts);
  if (launch_moe_route(topk_ids, static_cast<int>(pairs), L13.num_experts, bn, exp_off, tile_off, perm, nullptr,
                       nullptr, counts, reinterpret_cast<int*>(ws), s) != cudaSuccess)
    return HQ_ERR_CUDA;
  if (launch_moe_permute(x, ldx, tokens, perm, exp_off + L13.num_experts, static_cast<int>(pairs), topk, L13.k, xg,
                         ldg, di.sms, s) != cudaSuccess)
    return HQ_ERR_CUDA;
  int stages = 0, groups = 0;
  // gate+up with silu(gate) * up in its epilogue when the up rows start on a
  // tile boundary (I a multiple of 128) and the tiles have two accumulator
  // buffers (at most 128 tokens): A[p] straight from the two accumulators.
  // Otherwise H[p] = Xg[p] . W13_e^T in routed order, then an elementwise
  // kernel.
  const bool fused = inter % kTileN == 0 && bn <= kGateBufBn && di.sms <= kPlanSmsBound;
  if (fused) {
    st = launch_moe_grouped(L13, static_cast<const uint8_t*>(w13_t), bn, xg, ldg, static_cast<int>(pairs), exp_off,
                            kMoeOutGated, nullptr, abuf, lda, exp_off, tile_off, perm, nullptr,
                            reinterpret_cast<int*>(ws), di, s, &stages, &groups, gate_buf);
    if (st != HQ_OK) return st;
  } else {
    st = launch_moe_grouped(L13, static_cast<const uint8_t*>(w13_t), bn, xg, ldg, static_cast<int>(pairs), exp_off,
                            kMoeOutRouted, nullptr, hbuf, ldh, exp_off, tile_off, perm, nullptr,
                            reinterpret_cast<int*>(ws), di, s, &stages, &groups);
    if (st != HQ_OK) return st;
    if (launch_moe_act(hbuf, ldh, static_cast<int>(pairs), inter, abuf, lda, s) != cudaSuccess) return HQ_ERR_CUDA;
  }
  // down: Z[perm[p]] = topk_w[perm[p]] * A[p] . W2_e^T (A in routed order)
  st = launch_moe_grouped(L2, static_cast<const uint8_t*>(w2_t), bn, abuf, lda, static_cast<int>(pairs), exp_off,
                          kMoeOutZ, topk_w, y, ldy, exp_off, tile_off, perm, zbuf, reinterpret_cast<int*>(ws), di, s,
                          &stages, &groups);
  if (st != HQ_OK) return st;
  if (launch_moe_combine(zbuf, topk_ids, tokens, topk, L2.num_experts, L2.n, L2.n_pad, y, ldy, true, s) !=
      cudaSuccess)
    return HQ_ERR_CUDA;
  g_last_plan = hq_plan_info{bn, 1, di.sms, fused ? 5 : 6, stages, wna16_class(bn), groups, g_moe_x_stages};
  return HQ_OK;
}

hq_status hq_moe_grouped_workspace_size(const hq_weight_desc* desc, int32_t form, int32_t rows, size_t* bytes) {
  if (!desc || !bytes || rows < 0 || (form != HQ_MOE_GROUPED_CONTIGUOUS && form != HQ_MOE_GROUPED_MASKED))
    return HQ_ERR_INVALID_ARG;
  Layout L;
  hq_status st = make_layout(*desc, &L);
  if (st != HQ_OK) return st;
  const int64_t x_rows = form == HQ_MOE_GROUPED_MASKED ? static_cast<int64_t>(rows) * L.num_experts : rows;
  size_t ws = kAlign;
  ws += 3 * align_up(sizeof(int) * (L.num_experts + 1), kAlign);
  ws += align_up(sizeof(int) * std::max<int64_t>(x_rows, 1), kAlign);
  *bytes = ws;
  return HQ_OK;
}

hq_status hq_moe_grouped_gemm(const hq_weight_desc* wdesc, const void* w_t, int32_t form, int32_t rows,
                              const int32_t* expert_rows, int32_t expected_rows, int32_t atype, const void* x,
                              int64_t ldx, void* y, int64_t ldy, void* workspace, size_t ws_bytes, uint32_t flags,
                              hq_stream_t stream) {
  (void)flags;
  if (!wdesc || rows < 0 || (form != HQ_MOE_GROUPED_CONTIGUOUS && form != HQ_MOE_GROUPED_MASKED))
    return HQ_ERR_INVALID_ARG;
  Layout L;
  hq_status st = make_layout(*wdesc, &L);
  if (st != HQ_OK) return st;
  if (atype < HQ_A_BF16 || atype > HQ_A_MXFP8_E4M3) return HQ_ERR_INVALID_ARG;
  if (L.num_experts > 1024) return HQ_ERR_UNSUPPORTED;
  if (rows == 0) return HQ_OK;
  if (!w_t || !expert_rows || !x || !y || !workspace) return HQ_ERR_INVALID_ARG;
  if (ldx < L.k || ldy < L.n) return HQ_ERR_INVALID_ARG;
  if (atype != HQ_A_BF16) return HQ_ERR_UNSUPPORTED;
  if (L.wtype == HQ_W_FP8_E4M3) return HQ_ERR_UNSUPPORTED;
  if ((L.wtype == HQ_W_INT4 || L.wtype == HQ_W_INT6) && !L.channel && L.stype != HQ_S_BF16) return HQ_ERR_UNSUPPORTED;
  if (!aligned16(x) || !aligned16(y) || !aligned16(workspace) || (reinterpret_cast<uintptr_t>(w_t) & 255u))
    return HQ_ERR_ALIGNMENT;
  if ((ldx * 2) % 16 != 0 || (ldy * 2) % 16 != 0 || L.k % 8 != 0) return HQ_ERR_ALIGNMENT;
  const bool masked = form == HQ_MOE_GROUPED_MASKED;
  const int64_t x_rows = masked ? static_cast<int64_t>(rows) * L.num_experts : rows;
  if (x_rows > (1 << 24) || !tiles_fit(x_rows, L.num_experts, L.n_tiles)) return HQ_ERR_UNSUPPORTED;
  size_t need = 0;
  hq_moe_grouped_workspace_size(wdesc, form, rows, &need);
  if (ws_bytes < need) return HQ_ERR_WORKSPACE_TOO_SMALL;
  DevInfo di;
  st = device_info(&di);
  if (st != HQ_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  const uint8_t* wt = static_cast<const uint8_t*>(w_t);
  size_t off = kAlign;
  int* exp_off = reinterpret_cast<int*>(ws + off);
  off += align_up(sizeof(int) * (L.num_experts + 1), kAlign);
  int* tile_off = reinterpret_cast<int*>(ws + off);
  off += align_up(sizeof(int) * (L.num_experts + 1), kAlign);
  int* x_base = reinterpret_cast<int*>(ws + off);
  off += align_up(sizeof(int) * (L.num_experts + 1), kAlign);
  int* perm = reinterpret_cast<int*>(ws + off);
  // tile width from the caller's expected rows per expert (the counts stay on
  // the device), else from the mean that fills the given rows
  const double mean_rows = expected_rows > 0 ? expected_rows
                           : masked          ? static_cast<double>(rows)
                                             : static_cast<double>(rows) / L.num_experts;
  const int bn = moe_tile_bn(mean_rows);
  if (launch_moe_grouped_route(expert_rows, masked, rows, L.num_experts, bn, exp_off, tile_off, perm, x_base,
                               reinterpret_cast<int*>(ws), s) != cudaSuccess)
    return HQ_ERR_CUDA;
  int stages = 0, groups = 0;
  st = launch_moe_grouped(L, wt, bn, x, ldx, static_cast<int>(x_rows), x_base, kMoeOutRowMap, nullptr, y, ldy,
                          exp_off, tile_off, perm, nullptr, reinterpret_cast<int*>(ws), di, s, &stages, &groups);
  if (st != HQ_OK) return st;
  g_last_plan = hq_plan_info{bn, 1, di.sms, 2, stages, wna16_class(bn), groups, g_moe_x_stages};
  return HQ_OK;
}

}  // extern "C"
