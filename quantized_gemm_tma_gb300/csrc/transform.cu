// transform.cu — hq_transform / hq_untransform device code: repack a
// standard-format quantized weight into the sm_103 tile layout described in
// hq_internal.h and back, bit-exactly ("Preprocessing then validates
// parameters, pads dimensions, and repacks these tensors into layouts suited
// to the target kernel" — Humming launch article, standard-format paragraph).
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "hq_internal.h"

namespace hq {
namespace {

struct TArgs {
  Layout L;
  const uint8_t* codes;
  const uint8_t* scales;
  const uint8_t* zeros;
  const float* tensor_scales;  // NVFP4: [E]
  uint8_t* dst;  // transformed buffer (header first)
};

__device__ __forceinline__ int std_code_bytes_per_row(const Layout& L) {
  switch (L.wtype) {
    case HQ_W_INT4:
    case HQ_W_MXFP4:
    case HQ_W_NVFP4:
    case HQ_W_MXINT4: return (L.k + 1) / 2;
    case HQ_W_INT6: return 3 * L.k / 4;
    default: return L.k;
  }
}

__device__ __forceinline__ int std_zero_bytes_per_row(const Layout& L) {
  return L.wtype == HQ_W_INT4 ? (L.groups + 1) / 2 : 3 * ((L.groups + 3) / 4);
}

// unsigned code k of a standard-format row
__device__ __forceinline__ uint32_t read_code(const Layout& L, const uint8_t* row, int k) {
  if (L.wtype == HQ_W_INT6) {
    const int bit = 6 * k;
    const int b = bit >> 3, sh = bit & 7;
    uint32_t v = row[b];
    if (sh > 2) v |= static_cast<uint32_t>(row[b + 1]) << 8;
    return (v >> sh) & 0x3Fu;
  }
  if (L.wtype == HQ_W_FP8_E4M3) return row[k];
  return (row[k >> 1] >> (4 * (k & 1))) & 0xFu;
}

// the zero point of group g (packed like the codes)
__device__ __forceinline__ uint32_t read_zero(const Layout& L, const uint8_t* zrow, int g) {
  if (L.wtype == HQ_W_INT6) {
    const int bit = 6 * g;
    const int b = bit >> 3, sh = bit & 7;
    uint32_t v = zrow[b];
    if (sh > 2) v |= static_cast<uint32_t>(zrow[b + 1]) << 8;
    return (v >> sh) & 0x3Fu;
  }
  return (zrow[g >> 1] >> (4 * (g & 1))) & 0xFu;
}

// offset-binary code stored in the tile for a standard code
__device__ __forceinline__ uint32_t to_tile_code(const Layout& L, uint32_t c) {
  if (L.wtype == HQ_W_MXFP4 || L.wtype == HQ_W_NVFP4 || L.wtype == HQ_W_FP8_E4M3) return c;  // float codes as they are
  if (L.wtype == HQ_W_MXINT4) return c ^ 0x8u;  // always two's complement: q + 8
  if (L.has_zeros || !L.signed_codes) return c;
  return L.wtype == HQ_W_INT4 ? (c ^ 0x8u) : (c ^ 0x20u);  // q + 2^(b-1)
}

__device__ __forceinline__ uint32_t from_tile_code(const Layout& L, uint32_t u) { return to_tile_code(L, u); }

__device__ __forceinline__ uint32_t pad_code(const Layout& L) {
  if ((L.wtype == HQ_W_INT4 && !L.has_zeros && L.signed_codes) || L.wtype == HQ_W_MXINT4) return 8u;
  if (L.wtype == HQ_W_INT6 && !L.has_zeros && L.signed_codes) return 32u;
  return 0u;
}

// Standard-format group index of tile-local scale slot g of tile kt (or -1 for padding).
__device__ __forceinline__ int std_group(const Layout& L, int kt, int g) {
  if (L.g_kb > 1) {
    const int grp = kt * L.g_kb + g;
    return grp < L.groups ? grp : -1;
  }
  const int grp = (kt * kTileK) / L.group_k;
  return grp < L.groups ? grp : -1;
}

__device__ __forceinline__ float f16bits_to_f32(uint16_t b, int stype) {
  if (stype == HQ_S_BF16) return __uint_as_float(static_cast<uint32_t>(b) << 16);
  return __half2float(__ushort_as_half(b));
}

__device__ __forceinline__ uint32_t f32_to_f16bits(float f, int stype) {
  if (stype == HQ_S_BF16) return __float_as_uint(f) >> 16;  // exact: the value came from bf16
  return __half_as_ushort(__float2half_rn(f));                // exact: the value came from fp16
}

// ------------------------------------------------------------------ repack
// grid (k_tiles, n_tiles, E), block 128: thread r handles row r of one tile.
__global__ void __launch_bounds__(128) repack_kernel(const TArgs a) {
  const Layout& L = a.L;
  const int kt = blockIdx.x, nt = blockIdx.y, e = blockIdx.z;
  const int r = threadIdx.x;
  const int n = nt * kTileN + r;
  const bool row_ok = n < L.n;
  TileHeader* hdr = reinterpret_cast<TileHeader*>(a.dst);
  uint8_t* tile = a.dst + L.tiles_off + static_cast<uint64_t>(e) * L.expert_stride +
                  (static_cast<uint64_t>(nt) * L.k_tiles + kt) * L.tile_bytes;
  const size_t rowsN = static_cast<size_t>(e) * L.n + n;
  const uint8_t* crow = a.codes + rowsN * std_code_bytes_per_row(L);
  uint32_t invalid = 0;

  if (kt == 0 && nt == 0 && e == 0 && r == 0) {
    hdr->magic = kMagic;
    hdr->version = kLayoutVersion;
    hdr->wtype = L.wtype; hdr->stype = L.stype; hdr->n = L.n; hdr->k = L.k;
    hdr->num_experts = L.num_experts; hdr->group_k = L.group_k;
    hdr->signed_codes = L.signed_codes; hdr->has_zeros = L.has_zeros;
  }

  if (L.wtype == HQ_W_FP8_E4M3) {
    // swizzled 128-byte rows: chunk j of row r stored at chunk j ^ (r % 8)
    for (int j = 0; j < 8; ++j) {
      uint32_t w[4];
      for (int q = 0; q < 4; ++q) {
        uint32_t word = 0;
        for (int b = 0; b < 4; ++b) {
          const int k = kt * kTileK + 16 * j + 4 * q + b;
          uint32_t c = 0;
          if (row_ok && k < L.k) {
            c = crow[k];
            if ((c & 0x7Fu) == 0x7Fu) ++invalid;
          }
          word |= c << (8 * b);
        }
        w[q] = word;
      }
      *reinterpret_cast<uint4*>(tile + r * 128 + 16 * (j ^ (r & 7))) = make_uint4(w[0], w[1], w[2], w[3]);
    }
    if (r == 0) {
      const float* s = reinterpret_cast<const float*>(a.scales);
      float* blk = reinterpret_cast<float*>(a.dst + L.blk_off);
      const size_t idx = (static_cast<size_t>(e) * L.n_tiles + nt) * L.k_tiles + kt;
      blk[idx] = s[idx];
    }
    if (invalid) atomicAdd(&hdr->invalid_count, invalid);
    return;
  }

  // 4-bit low nibbles (INT4, MXFP4, and the low part of INT6)
  const uint32_t pad = pad_code(L);
  for (int c = 0; c < 4; ++c) {
    uint32_t lo[4] = {0, 0, 0, 0};
    uint32_t hi[2] = {0, 0};
    for (int j = 0; j < 4; ++j) {
      for (int el = 0; el < 8; ++el) {
        const int k = kt * kTileK + 32 * c + 8 * j + el;
        uint32_t u = pad;
        if (row_ok && k < L.k) u = to_tile_code(L, read_code(L, crow, k));
        const int p = el / 2 + 4 * (el % 2);
        lo[j] |= (u & 0xFu) << (4 * p);
        if (L.wtype == HQ_W_INT6) {
          const int pos = (4 + 16 * (el % 2) + 4 * (el / 2) + 2 * (j % 2)) & 31;
          hi[j / 2] |= ((u >> 4) & 0x3u) << pos;
        }
      }
    }
    *reinterpret_cast<uint4*>(tile + (c * kTileN + r) * 16) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
    if (L.wtype == HQ_W_INT6)
      *reinterpret_cast<uint2*>(tile + L.hi_off + (c * kTileN + r) * 8) = make_uint2(hi[0], hi[1]);
  }

  if (L.wtype == HQ_W_NVFP4) {
    // e4m3 block scales [row][8]; a NaN scale or tensor scale is invalid
    uint32_t sc[2] = {0, 0};
    for (int j = 0; j < 8; ++j) {
      const int kk = kt * kTileK + 16 * j;
      uint32_t b = 0;
      if (row_ok && kk < L.k) {
        b = a.scales[rowsN * (L.k / 16) + kk / 16];
        if ((b & 0x7Fu) == 0x7Fu) ++invalid;
      }
      sc[j / 4] |= b << (8 * (j % 4));
    }
    *reinterpret_cast<uint2*>(tile + L.scale_off + r * 8) = make_uint2(sc[0], sc[1]);
    if (kt == 0 && nt == 0 && r == 0) {
      const float g = a.tensor_scales[e];
      if (g != g) ++invalid;
      reinterpret_cast<float*>(a.dst + L.ts_off)[e] = g;
    }
    if (invalid) atomicAdd(&hdr->invalid_count, invalid);
    return;
  }
  if (L.wtype == HQ_W_MXFP4 || L.wtype == HQ_W_MXINT4) {
    uint32_t sc = 0;
    for (int c = 0; c < 4; ++c) {
      const int kk = kt * kTileK + 32 * c;
      uint32_t E = 127;
      if (row_ok && kk < L.k) {
        E = a.scales[rowsN * (L.k / 32) + kk / 32];
        if (E == 255u) ++invalid;
      }
      sc |= E << (8 * c);
    }
    *reinterpret_cast<uint32_t*>(tile + L.scale_off + r * 4) = sc;
    if (invalid) atomicAdd(&hdr->invalid_count, invalid);
    return;
  }

  // INT scales / zeros
  const uint16_t* srow = reinterpret_cast<const uint16_t*>(a.scales) + rowsN * L.groups;
  const uint8_t* zrow = L.has_zeros ? a.zeros + rowsN * std_zero_bytes_per_row(L) : nullptr;
  if (L.channel) {
    if (kt == 0) {
      float* rs = reinterpret_cast<float*>(a.dst + L.row_off);
      rs[static_cast<size_t>(e) * L.n_pad + n] = row_ok ? f16bits_to_f32(srow[0], L.stype) : 0.f;
      if (L.has_zeros) a.dst[L.row_zero_off + static_cast<size_t>(e) * L.n_pad + n] =
          static_cast<uint8_t>(row_ok ? read_zero(L, zrow, 0) : 0u);
    }
    return;
  }
  for (int g = 0; g < L.g_kb; ++g) {
    const int grp = std_group(L, kt, g);
    const bool ok = row_ok && grp >= 0;
    reinterpret_cast<uint16_t*>(tile + L.scale_off)[r * L.g_kb + g] = ok ? srow[grp] : static_cast<uint16_t>(0);
    if (L.has_zeros) tile[L.zero_off + r * L.g_kb + g] = static_cast<uint8_t>(ok ? read_zero(L, zrow, grp) : 0u);
  }
}

// ------------------------------------------------------------------ unpack codes
// grid (k_tiles, n_tiles, E), block 128: thread r rebuilds its row's codes of one tile.
__global__ void __launch_bounds__(128) unpack_codes_kernel(const TArgs a, uint8_t* codes_out) {
  const Layout& L = a.L;
  const int kt = blockIdx.x, nt = blockIdx.y, e = blockIdx.z;
  const int r = threadIdx.x;
  const int n = nt * kTileN + r;
  if (n >= L.n) return;
  const uint8_t* tile = a.dst + L.tiles_off + static_cast<uint64_t>(e) * L.expert_stride +
                        (static_cast<uint64_t>(nt) * L.k_tiles + kt) * L.tile_bytes;
  const size_t rowsN = static_cast<size_t>(e) * L.n + n;
  uint8_t* crow = codes_out + rowsN * std_code_bytes_per_row(L);
  const int k0 = kt * kTileK;
  const int kend = min(L.k, k0 + kTileK);

  if (L.wtype == HQ_W_FP8_E4M3) {
    for (int k = k0; k < kend; ++k) {
      const int kk = k - k0, j = kk / 16;
      crow[k] = tile[r * 128 + 16 * (j ^ (r & 7)) + (kk & 15)];
    }
    return;
  }
  auto tile_code = [&](int kk) -> uint32_t {
    const int c = kk / 32, j = (kk % 32) / 8, el = kk % 8;
    const uint32_t word = reinterpret_cast<const uint32_t*>(tile + (c * kTileN + r) * 16)[j];
    uint32_t u = (word >> (4 * (el / 2 + 4 * (el % 2)))) & 0xFu;
    if (L.wtype == HQ_W_INT6) {
      const uint32_t h = reinterpret_cast<const uint32_t*>(tile + L.hi_off + (c * kTileN + r) * 8)[j / 2];
      const int pos = (4 + 16 * (el % 2) + 4 * (el / 2) + 2 * (j % 2)) & 31;
      u |= ((h >> pos) & 0x3u) << 4;
    }
    return from_tile_code(L, u);
  };
  if (L.wtype == HQ_W_INT6) {
    // groups of 4 codes -> 3 bytes; tile boundaries are multiples of 4 codes
    for (int k = k0; k < kend; k += 4) {
      uint32_t v = 0;
      for (int q = 0; q < 4; ++q) v |= tile_code(k - k0 + q) << (6 * q);
      const int b = 3 * k / 4;
      crow[b] = v & 0xFF; crow[b + 1] = (v >> 8) & 0xFF; crow[b + 2] = (v >> 16) & 0xFF;
    }
    return;
  }
  for (int k = k0; k < kend; k += 2) {
    uint32_t v = tile_code(k - k0);
    if (k + 1 < kend) v |= tile_code(k - k0 + 1) << 4;
    crow[k >> 1] = static_cast<uint8_t>(v);
  }
}

// ------------------------------------------------------------------ unpack scales / zeros
// grid ceil(E*N/128), block 128: one thread per weight row rebuilds scales and zeros.
__global__ void __launch_bounds__(128) unpack_meta_kernel(const TArgs a, uint8_t* scales_out, uint8_t* zeros_out) {
  const Layout& L = a.L;
  const size_t row = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (row >= static_cast<size_t>(L.num_experts) * L.n) return;
  const int e = static_cast<int>(row / L.n), n = static_cast<int>(row % L.n);
  const int nt = n / kTileN, r = n % kTileN;
  auto tile_at = [&](int kt) {
    return a.dst + L.tiles_off + static_cast<uint64_t>(e) * L.expert_stride +
           (static_cast<uint64_t>(nt) * L.k_tiles + kt) * L.tile_bytes;
  };
  if (L.wtype == HQ_W_FP8_E4M3) {
    if (r == 0) {
      const float* blk = reinterpret_cast<const float*>(a.dst + L.blk_off);
      float* s = reinterpret_cast<float*>(scales_out);
      for (int kt = 0; kt < L.k_tiles; ++kt) {
        const size_t idx = (static_cast<size_t>(e) * L.n_tiles + nt) * L.k_tiles + kt;
        s[idx] = blk[idx];
      }
    }
    return;
  }
  if (L.wtype == HQ_W_NVFP4) {
    for (int g = 0; g < L.k / 16; ++g) {
      const int kt = g / 8, j = g % 8;
      scales_out[row * (L.k / 16) + g] = tile_at(kt)[L.scale_off + r * 8 + j];
    }
    // the tensor scales go to the zeros argument (NVFP4 has no zero points)
    if (n == 0) reinterpret_cast<float*>(zeros_out)[e] = reinterpret_cast<const float*>(a.dst + L.ts_off)[e];
    return;
  }
  if (L.wtype == HQ_W_MXFP4 || L.wtype == HQ_W_MXINT4) {
    for (int g = 0; g < L.k / 32; ++g) {
      const int kt = g / 4, c = g % 4;
      scales_out[row * (L.k / 32) + g] = tile_at(kt)[L.scale_off + r * 4 + c];
    }
    return;
  }
  uint16_t* srow = reinterpret_cast<uint16_t*>(scales_out) + row * L.groups;
  auto zero_of = [&](int g) -> uint32_t {
    if (L.channel) return a.dst[L.row_zero_off + static_cast<size_t>(e) * L.n_pad + n];
    if (L.g_kb > 1) return tile_at(g / L.g_kb)[L.zero_off + r * L.g_kb + g % L.g_kb];
    return tile_at(g * L.group_k / kTileK)[L.zero_off + r];
  };
  for (int g = 0; g < L.groups; ++g) {
    uint16_t s;
    if (L.channel) {
      const float* rs = reinterpret_cast<const float*>(a.dst + L.row_off);
      s = static_cast<uint16_t>(f32_to_f16bits(rs[static_cast<size_t>(e) * L.n_pad + n], L.stype));
    } else if (L.g_kb > 1) {
      s = reinterpret_cast<const uint16_t*>(tile_at(g / L.g_kb) + L.scale_off)[r * L.g_kb + g % L.g_kb];
    } else {
      s = reinterpret_cast<const uint16_t*>(tile_at(g * L.group_k / kTileK) + L.scale_off)[r];
    }
    srow[g] = s;
  }
  if (!L.has_zeros) return;
  if (L.wtype == HQ_W_INT4) {
    uint8_t* zrow = zeros_out + row * ((L.groups + 1) / 2);
    for (int g = 0; g < L.groups; g += 2) {
      uint32_t v = zero_of(g);
      if (g + 1 < L.groups) v |= zero_of(g + 1) << 4;
      zrow[g >> 1] = static_cast<uint8_t>(v);
    }
  } else {
    const int gp = (L.groups + 3) / 4;
    uint8_t* zrow = zeros_out + row * (3 * gp);
    for (int q4 = 0; q4 < gp; ++q4) {
      uint32_t v = 0;
      for (int q = 0; q < 4; ++q) {
        const int g = 4 * q4 + q;
        if (g < L.groups) v |= zero_of(g) << (6 * q);
      }
      zrow[3 * q4] = v & 0xFF; zrow[3 * q4 + 1] = (v >> 8) & 0xFF; zrow[3 * q4 + 2] = (v >> 16) & 0xFF;
    }
  }
}

}  // namespace

cudaError_t launch_repack(const Layout& L, const hq_weight_desc& d, void* dst, cudaStream_t stream) {
  TArgs a{L, static_cast<const uint8_t*>(d.codes), static_cast<const uint8_t*>(d.scales),
          static_cast<const uint8_t*>(d.zeros), static_cast<const float*>(d.tensor_scales),
          static_cast<uint8_t*>(dst)};
  cudaError_t err = cudaMemsetAsync(dst, 0, L.total, stream);
  if (err != cudaSuccess) return err;
  dim3 grid(L.k_tiles, L.n_tiles, L.num_experts);
  repack_kernel<<<grid, 128, 0, stream>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_unpack(const Layout& L, const void* src, void* codes, void* scales, void* zeros,
                          cudaStream_t stream) {
  TArgs a{L, nullptr, nullptr, nullptr, nullptr, const_cast<uint8_t*>(static_cast<const uint8_t*>(src))};
  dim3 grid(L.k_tiles, L.n_tiles, L.num_experts);
  unpack_codes_kernel<<<grid, 128, 0, stream>>>(a, static_cast<uint8_t*>(codes));
  cudaError_t err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  const size_t rows = static_cast<size_t>(L.num_experts) * L.n;
  unpack_meta_kernel<<<static_cast<unsigned>((rows + 127) / 128), 128, 0, stream>>>(
      a, static_cast<uint8_t*>(scales), static_cast<uint8_t*>(zeros));
  return cudaGetLastError();
}

}  // namespace hq
