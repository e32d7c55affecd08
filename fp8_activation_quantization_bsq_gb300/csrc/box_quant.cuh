// Quantization of one row of a 64-column box (the per-lane step of the dense
// and grouped kernels): 8 x 16-byte chunks of BF16 -> NVFP4 (4 blocks of 16)
// or MX (2 blocks of 32) codes, stored to the packed output, and the box's
// scale bytes returned to the caller.
#pragma once

#include "device_common.cuh"

namespace bsq {

// NVFP4 element-scale source: a 256-entry table indexed by the scale byte,
// or (null) the division tensor_sf / ds itself.
struct NvScale {
  float tsf;
  const float* factor_tab;  // 256 entries, or nullptr
  const float* div6_tab;    // 128 entries: fl32((128 + f) / 192)
};

__device__ __forceinline__ BlockScale nvfp4_block_scale(float amax, const NvScale& ns) {
  const uint32_t b = f32_to_e4m3(__fmul_rn(amax_div6(amax, ns.div6_tab), ns.tsf));
  if (ns.factor_tab) return {b, ns.factor_tab[b]};
  const float ds = e4m3_to_f32(b);
  return {b, ds == 0.0f ? 0.0f : __fdiv_rn(ns.tsf, ds)};
}

// Quantize one row of a 64-column box held in registers (8 x 16-byte chunks
// of BF16).  valid_cols: 64 or 32 columns hold data (chunks 4..7 are ignored
// and treated as zeros when 32).  dst: packed output of the box's first
// column (nullptr: compute the scales only).  vec32: dst allows 32-byte
// stores.  Returns the box's scale bytes (block i in byte i).
template <int FMT>
__device__ __forceinline__ uint32_t quant_box_regs(uint4 (&v)[8], int valid_cols, uint8_t* dst,
                                                   bool vec32, const NvScale& ns) {
  const bool full = valid_cols == 64;
  if (!full) {
#pragma unroll
    for (int c = 4; c < 8; ++c) v[c] = make_uint4(0u, 0u, 0u, 0u);
  }
  uint32_t scale_bytes = 0;

  if constexpr (FMT == kNVFP4) {
    uint32_t o[8];
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      uint32_t acc = 0;
      acc = absmax2(acc, v[2 * b].x); acc = absmax2(acc, v[2 * b].y);
      acc = absmax2(acc, v[2 * b].z); acc = absmax2(acc, v[2 * b].w);
      acc = absmax2(acc, v[2 * b + 1].x); acc = absmax2(acc, v[2 * b + 1].y);
      acc = absmax2(acc, v[2 * b + 1].z); acc = absmax2(acc, v[2 * b + 1].w);
      const BlockScale sc = nvfp4_block_scale(absmax_final(acc), ns);
      o[2 * b] = quant8_e2m1(v[2 * b], sc.factor);
      o[2 * b + 1] = quant8_e2m1(v[2 * b + 1], sc.factor);
      scale_bytes |= sc.byte << (8 * b);
    }
    if (dst) {
      if (full && vec32) {
        st_global_v8(dst, o);
      } else {
        st_global_v4(dst, o[0], o[1], o[2], o[3]);
        if (full) st_global_v4(dst + 16, o[4], o[5], o[6], o[7]);
      }
    }
  } else {
    constexpr int QMAX = FMT == kMXFP4 ? 6 : 448;
#pragma unroll
    for (int b = 0; b < 2; ++b) {
      uint32_t acc = 0;
#pragma unroll
      for (int c = 4 * b; c < 4 * b + 4; ++c) {
        acc = absmax2(acc, v[c].x); acc = absmax2(acc, v[c].y);
        acc = absmax2(acc, v[c].z); acc = absmax2(acc, v[c].w);
      }
      const MxScale sc = mx_scale<QMAX>(absmax_final(acc));
      scale_bytes |= sc.byte << (8 * b);
      if constexpr (FMT == kMXFP4) {
        const uint32_t o0 = quant8_e2m1_pow2(v[4 * b], sc.pow2), o1 = quant8_e2m1_pow2(v[4 * b + 1], sc.pow2);
        const uint32_t o2 = quant8_e2m1_pow2(v[4 * b + 2], sc.pow2), o3 = quant8_e2m1_pow2(v[4 * b + 3], sc.pow2);
        if (dst && (b == 0 || full)) st_global_v4(dst + 16 * b, o0, o1, o2, o3);
      } else {
        uint32_t o[8];
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const uint2 q = quant8_e4m3_pow2(v[4 * b + c], sc.pow2);
          o[2 * c] = q.x;
          o[2 * c + 1] = q.y;
        }
        if (dst && (b == 0 || full)) {
          if (vec32) {
            st_global_v8(dst + 32 * b, o);
          } else {
            st_global_v4(dst + 32 * b, o[0], o[1], o[2], o[3]);
            st_global_v4(dst + 32 * b + 16, o[4], o[5], o[6], o[7]);
          }
        }
      }
    }
  }
  return scale_bytes;
}

// The same for a row held in shared memory at rowp (SWIZZLED: chunk c sits
// at c ^ (row % 8), the TMA 128-byte swizzle; else at c).
template <int FMT, bool SWIZZLED>
__device__ __forceinline__ uint32_t quant_box_row(const uint8_t* rowp, int row, int valid_cols,
                                                   uint8_t* dst, bool vec32, const NvScale& ns) {
  uint4 v[8];
#pragma unroll
  for (int c = 0; c < 8; ++c)
    v[c] = *reinterpret_cast<const uint4*>(rowp + ((SWIZZLED ? (c ^ (row & 7)) : c) << 4));
  return quant_box_regs<FMT>(v, valid_cols, dst, vec32, ns);
}

}  // namespace bsq
