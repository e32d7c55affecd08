// Grouped per-expert block-scaled quantization (MoE activations).
//
// The 5D scale buffer is cut into 128-row tiles; the groups' scale rows are
// padded to whole tiles (scales_offsets are multiples of 128), so every tile
// belongs to exactly one group.  Thread block (tile, chunk) handles one tile
// and KT consecutive 5D atom columns (k_tiles_per_block): warp 0 finds the
// group with a warp-parallel search over scales_offsets (256 probes per
// round, one round of loads for up to 256 groups, row_offsets / expert_ids
// read in the same round) and broadcasts it through shared memory; batching KT column
// tiles per block amortizes that search and shrinks the grid, which dominates
// at decode where a tile holds a few routed rows.
//
// Work inside a block: one thread per scale block (16 or 32 elements of one
// row), consecutive threads on consecutive blocks of a row, so a warp reads
// and writes contiguous runs (256-bit loads of the gathered source row).
// Each thread reduces its block's amax in registers, derives the scale
// (NVFP4 through the division-free amax/6 and the per-block element-scale
// table; MX from the exponent bits), encodes and stores its elements; the
// four scale bytes of a row's atom are OR-reduced over 4 lanes and written as
// one word.  Blocks of the last atom that lie beyond K are zero, giving scale
// byte 0x00.
#pragma once

#include "device_common.cuh"

namespace bsq {

constexpr int kGroupedThreads = 128;

struct GroupedArgs {
  const uint16_t* in;
  int64_t ld_in;        // elements
  int64_t in_rows;
  int K;
  const uint32_t* row_offsets;
  const uint32_t* scales_offsets;
  const int32_t* expert_ids;
  const float* sf;
  int num_experts;
  const int32_t* row_indices;  // may be null
  int G;
  int64_t total_rows;
  int64_t total_scale_rows;
  uint8_t* out;
  int64_t out_ld;       // packed row bytes
  uint8_t* scales;
  int kt_atoms;         // atoms per 128-row band
  int in_vec32;         // input rows allow 32-byte loads
  int out_vec32;        // packed rows allow 32-byte stores
};

// Pick entry j (0..255, warp-uniform) of a 256-entry array held as 8
// registers per lane (entry j in register j/32 of lane j%32).
template <typename T>
__device__ __forceinline__ T warp_pick(const T (&reg)[8], int j) {
  T v = reg[0];
#pragma unroll
  for (int i = 1; i < 8; ++i)
    if ((j >> 5) == i) v = reg[i];
  return __shfl_sync(0xFFFFFFFFu, v, j & 31);
}

struct GroupHit {
  int64_t so_g, so_n, r_beg, r_end;
  int e;
};

// Locate the group of padded scale row `row0`: g = max{g : so[g] <= row0}
// for non-decreasing scales_offsets with so[0] <= row0 < so[G].  Runs on one
// full warp.  Rounds of 256 evenly spaced probes (8 loads per lane, issued
// together, counted with ballots) narrow the range 256-fold; the final round
// (step 1) also loads row_offsets and expert_ids at the probe positions, so
// the group's bounds and expert come out of registers by shuffles: for up to
// 256 groups the whole search is one round of loads.
__device__ __forceinline__ GroupHit warp_group_search(const GroupedArgs& a, int64_t row0) {
  const uint32_t* so = a.scales_offsets;
  const int lane = threadIdx.x & 31;
  int lo = 0, hi = a.G;
  while (hi - lo > 256) {
    const int step = (hi - lo + 255) >> 8;
    bool le[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int64_t pos = lo + static_cast<int64_t>(step) * (1 + lane + 32 * i);
      le[i] = pos < hi && static_cast<int64_t>(__ldg(so + pos)) <= row0;
    }
    int cnt = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) cnt += __popc(__ballot_sync(0xFFFFFFFFu, le[i]));
    const int nlo = lo + cnt * step;
    hi = min(hi, nlo + step);
    lo = nlo;
  }
  // final round: positions lo+1 .. lo+256 (so / ro up to G, expert ids below G)
  uint32_t so_p[8], ro_p[8];
  int32_t e_p[8];
  bool le[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int pos = lo + 1 + lane + 32 * i;
    so_p[i] = pos <= a.G ? __ldg(so + pos) : 0xFFFFFFFFu;
    ro_p[i] = pos <= a.G ? __ldg(a.row_offsets + pos) : 0u;
    e_p[i] = pos < a.G ? __ldg(a.expert_ids + pos) : -1;
    le[i] = pos < hi && static_cast<int64_t>(so_p[i]) <= row0;
  }
  const uint32_t so_lo = __ldg(so + lo), ro_lo = __ldg(a.row_offsets + lo);
  const int32_t e_lo = __ldg(a.expert_ids + lo);
  int cnt = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i) cnt += __popc(__ballot_sync(0xFFFFFFFFu, le[i]));
  // g = lo + cnt; entry g sits at probe index cnt-1, entry g+1 at index cnt
  GroupHit h;
  h.so_g = cnt == 0 ? so_lo : warp_pick(so_p, cnt - 1);
  h.r_beg = cnt == 0 ? ro_lo : warp_pick(ro_p, cnt - 1);
  h.e = cnt == 0 ? e_lo : warp_pick(e_p, cnt - 1);
  h.so_n = warp_pick(so_p, cnt);
  h.r_end = warp_pick(ro_p, cnt);
  return h;
}

struct GroupMeta {
  int64_t dst0;   // first destination row of this tile
  int n;          // valid rows in the tile (0: nothing to do)
  int e;          // expert id
};

template <int FMT, int KT>
__global__ void __launch_bounds__(kGroupedThreads) grouped_quant_kernel(const GroupedArgs a) {
  constexpr int SF = Fmt<FMT>::SF;
  constexpr int BPR = 4 * KT;                      // scale blocks per row in a chunk
  constexpr int LOG_BPR = KT == 1 ? 2 : KT == 2 ? 3 : KT == 4 ? 4 : 5;
  constexpr int U = FMT == kMXFP8 ? 2 : 4;         // blocks in flight per thread

  __shared__ GroupMeta meta;
  __shared__ float factor_tab[FMT == kNVFP4 ? 256 : 1];
  __shared__ float div6_tab[FMT == kNVFP4 ? 128 : 1];

  const int64_t row0 = static_cast<int64_t>(blockIdx.x) * 128;
  if (threadIdx.x < 32) {
    // ---- warp 0: locate the group
    GroupMeta m{0, 0, -1};
    const GroupHit h = warp_group_search(a, row0);
    const int64_t so0 = __ldg(a.scales_offsets), so_end = __ldg(a.scales_offsets + a.G);
    const int64_t ro_end = __ldg(a.row_offsets + a.G);
    if (blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0 &&
        (so0 != 0 || so_end > a.total_scale_rows || ro_end > a.total_rows))
      record_error(kErrValue);
    if (so0 == 0 && row0 < so_end) {
      const int64_t m_g = h.r_end - h.r_beg;
      const int64_t i0 = row0 - h.so_g;
      if (m_g < 0 || m_g > h.so_n - h.so_g || h.r_end > a.total_rows) {
        if (threadIdx.x == 0) record_error(kErrValue);
      } else if (i0 < m_g && h.e >= 0) {
        if (FMT == kNVFP4 && h.e >= a.num_experts) {
          if (threadIdx.x == 0) record_error(kErrValue);
        } else {
          m.dst0 = h.r_beg + i0;
          m.n = static_cast<int>(m_g - i0 < 128 ? m_g - i0 : 128);
          m.e = h.e;
        }
      }
    }
    if (threadIdx.x == 0) meta = m;
  } else if (FMT == kNVFP4) {
    fill_div6_table(div6_tab, threadIdx.x - 32, kGroupedThreads - 32);
  }
  __syncthreads();
  const GroupMeta m = meta;
  if (m.n == 0) return;

  const int atom0 = blockIdx.y * KT;
  const int col_base = atom0 * 4 * SF;
  const int total = m.n << LOG_BPR;
  uint8_t* band = a.scales + static_cast<int64_t>(blockIdx.x) * a.kt_atoms * 512;
  float tsf = 1.0f;

  for (int base = 0; base < total; base += kGroupedThreads * U) {
    uint4 v[U][SF / 8];
    bool ok[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int q = base + u * kGroupedThreads + threadIdx.x;
      const int r = q >> LOG_BPR;
      const int col = col_base + (q & (BPR - 1)) * SF;
#pragma unroll
      for (int c = 0; c < SF / 8; ++c) v[u][c] = make_uint4(0u, 0u, 0u, 0u);
      ok[u] = false;
      if (q < total && col < a.K) {
        const int64_t d = m.dst0 + r;
        const int64_t src = a.row_indices ? static_cast<int64_t>(__ldg(a.row_indices + d)) : d;
        if (src >= 0 && src < a.in_rows) {
          const uint16_t* p = a.in + src * a.ld_in + col;
          if (a.in_vec32) {
#pragma unroll
            for (int c = 0; c < SF / 8; c += 2) ld_global_nc_v8(p + 8 * c, v[u][c], v[u][c + 1]);
          } else {
#pragma unroll
            for (int c = 0; c < SF / 8; ++c) v[u][c] = ld_global_nc_v4(p + 8 * c);
          }
          ok[u] = true;
        } else {
          record_error(kErrValue);
        }
      }
    }
    if constexpr (FMT == kNVFP4) {
      if (base == 0) {
        // the expert's tensor_sf and element-scale table, while the first
        // round of gathered loads is in flight
        tsf = __ldg(a.sf + m.e);
        fill_nvfp4_factor_table(factor_tab, tsf, threadIdx.x, kGroupedThreads);
        __syncthreads();
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int q = base + u * kGroupedThreads + threadIdx.x;
      const int r = q >> LOG_BPR;
      const int b = q & (BPR - 1);
      const int col = col_base + b * SF;

      uint32_t acc = 0;
#pragma unroll
      for (int c = 0; c < SF / 8; ++c) {
        acc = absmax2(acc, v[u][c].x); acc = absmax2(acc, v[u][c].y);
        acc = absmax2(acc, v[u][c].z); acc = absmax2(acc, v[u][c].w);
      }
      const float amax = absmax_final(acc);
      uint32_t sbyte;
      const int64_t d = m.dst0 + r;
      uint8_t* dst = a.out + d * a.out_ld + (Fmt<FMT>::OUT_BITS == 4 ? col >> 1 : col);
      if constexpr (FMT == kNVFP4) {
        const BlockScale sc = nvfp4_scale_tab(amax, tsf, factor_tab, div6_tab);
        sbyte = sc.byte;
        const uint32_t o0 = quant8_e2m1(v[u][0], sc.factor), o1 = quant8_e2m1(v[u][1], sc.factor);
        if (ok[u]) *reinterpret_cast<uint2*>(dst) = make_uint2(o0, o1);
      } else if constexpr (FMT == kMXFP4) {
        const MxScale sc = mx_scale<6>(amax);
        sbyte = sc.byte;
        const uint32_t o0 = quant8_e2m1_pow2(v[u][0], sc.pow2), o1 = quant8_e2m1_pow2(v[u][1], sc.pow2);
        const uint32_t o2 = quant8_e2m1_pow2(v[u][2], sc.pow2), o3 = quant8_e2m1_pow2(v[u][3], sc.pow2);
        if (ok[u]) st_global_v4(dst, o0, o1, o2, o3);
      } else {
        const MxScale sc = mx_scale<448>(amax);
        sbyte = sc.byte;
        uint32_t o[8];
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const uint2 qq = quant8_e4m3_pow2(v[u][c], sc.pow2);
          o[2 * c] = qq.x;
          o[2 * c + 1] = qq.y;
        }
        if (ok[u]) {
          if (a.out_vec32) {
            st_global_v8(dst, o);
          } else {
            st_global_v4(dst, o[0], o[1], o[2], o[3]);
            st_global_v4(dst + 16, o[4], o[5], o[6], o[7]);
          }
        }
      }

      // scale word of (row r, atom b/4): byte of block b%4 at bits 8*(b%4)
      uint32_t word = sbyte << (8 * (b & 3));
      word |= __shfl_xor_sync(0xFFFFFFFFu, word, 1);
      word |= __shfl_xor_sync(0xFFFFFFFFu, word, 2);
      if (ok[u] && (b & 3) == 0) {
        const int atom = atom0 + (b >> 2);
        *reinterpret_cast<uint32_t*>(band + atom * 512 + (r & 31) * 16 + (r >> 5) * 4) = word;
      }
    }
  }
}

}  // namespace bsq
