// Grouped per-expert block-scaled quantization (MoE activations).
//
// The 5D scale buffer is cut into 128-row tiles; the groups' scale rows are
// padded to whole tiles (scales_offsets are multiples of 128), so every tile
// belongs to exactly one group.  Thread block (tile, chunk) handles one tile
// and KT consecutive 5D atom columns (k_tiles_per_block): a warp-parallel
// search over scales_offsets finds the group, row_offsets give its rows,
// expert_ids / sf_tensor its scale, row_indices the gathered source rows.
// Batching KT column tiles per block amortizes the search and shrinks the
// grid, which dominates at decode where a tile holds a few routed rows.
//
// Inside a block the (rows x columns) region is flattened into 8-element
// segments, consecutive segments of a row on consecutive lanes: each lane
// loads 16 bytes of BF16, a block's amax is reduced over its 2 (NVFP4) or 4
// (MX) lanes with shuffles, every lane encodes its 8 elements and a warp
// stores whole contiguous runs of packed bytes.  The scale bytes of one row's
// atom (4 blocks) are OR-reduced onto the atom's first lane, which writes the
// 4-byte word at its 5D position.  Padding columns inside the last atom are
// zero segments, whose blocks get scale byte 0x00.
#pragma once

#include "device_common.cuh"

namespace bsq {

constexpr int kGroupedThreads = 128;
constexpr int kGroupedUnroll = 8;

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
};

// g = max{ g in [0, G) : so[g] <= row0 } for non-decreasing so with
// so[0] <= row0 < so[G].  Each round probes 32 evenly spaced entries with one
// ballot and narrows the range 32-fold.
__device__ __forceinline__ int warp_group_search(const uint32_t* so, int G, int64_t row0) {
  const int lane = threadIdx.x & 31;
  int lo = 0, hi = G;
  while (hi - lo > 1) {
    const int step = (hi - lo + 31) >> 5;
    const int64_t pos = lo + static_cast<int64_t>(step) * (lane + 1);
    const bool le = pos < hi && static_cast<int64_t>(__ldg(so + pos)) <= row0;
    const int cnt = __popc(__ballot_sync(0xFFFFFFFFu, le));
    const int nlo = lo + cnt * step;
    hi = min(hi, nlo + step);
    lo = nlo;
  }
  return lo;
}

template <int FMT, int KT>
__global__ void __launch_bounds__(kGroupedThreads) grouped_quant_kernel(const GroupedArgs a) {
  constexpr int SF = Fmt<FMT>::SF;
  constexpr int AC = Fmt<FMT>::ATOM_COLS;
  constexpr int SEG_PER_BLOCK = SF / 8;
  constexpr int SEG_PER_ATOM = AC / 8;

  const int64_t row0 = static_cast<int64_t>(blockIdx.x) * 128;
  const int64_t so_end = __ldg(a.scales_offsets + a.G);

  if (blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0) {
    if (__ldg(a.scales_offsets) != 0u || so_end > a.total_scale_rows ||
        static_cast<int64_t>(__ldg(a.row_offsets + a.G)) > a.total_rows)
      record_error(kErrValue);
  }
  if (row0 >= so_end || __ldg(a.scales_offsets) != 0u) return;

  const int g = warp_group_search(a.scales_offsets, a.G, row0);
  const int64_t so_g = __ldg(a.scales_offsets + g), so_n = __ldg(a.scales_offsets + g + 1);
  const int64_t r_beg = __ldg(a.row_offsets + g), r_end = __ldg(a.row_offsets + g + 1);
  const int64_t m_g = r_end - r_beg;
  if (m_g < 0 || m_g > so_n - so_g || r_end > a.total_rows) {
    if (threadIdx.x == 0) record_error(kErrValue);
    return;
  }
  const int64_t i0 = row0 - so_g;
  if (i0 >= m_g) return;  // a padding tile of this group
  const int n = static_cast<int>(m_g - i0 < 128 ? m_g - i0 : 128);
  const int e = __ldg(a.expert_ids + g);
  if (e < 0) return;
  float tsf = 1.0f;
  if constexpr (FMT == kNVFP4) {
    if (e >= a.num_experts) {
      if (threadIdx.x == 0) record_error(kErrValue);
      return;
    }
    tsf = __ldg(a.sf + e);
  }

  const int atom0 = blockIdx.y * KT;
  const int natoms = min(KT, a.kt_atoms - atom0);
  const int segs_row = natoms * SEG_PER_ATOM;
  const int total = n * segs_row;
  const int col_base = atom0 * AC;
  const int64_t dst0 = r_beg + i0;
  uint8_t* band = a.scales + static_cast<int64_t>(blockIdx.x) * a.kt_atoms * 512;

  for (int base = 0; base < total; base += kGroupedThreads * kGroupedUnroll) {
    uint4 v[kGroupedUnroll];
    bool ok[kGroupedUnroll];
#pragma unroll
    for (int u = 0; u < kGroupedUnroll; ++u) {
      const int q = base + u * kGroupedThreads + threadIdx.x;
      const int r = q / segs_row;
      const int col = col_base + (q - r * segs_row) * 8;
      v[u] = make_uint4(0u, 0u, 0u, 0u);
      ok[u] = false;
      if (q < total && col < a.K) {
        const int64_t d = dst0 + r;
        const int64_t src = a.row_indices ? static_cast<int64_t>(__ldg(a.row_indices + d)) : d;
        if (src >= 0 && src < a.in_rows) {
          v[u] = ld_global_nc_v4(a.in + src * a.ld_in + col);
          ok[u] = true;
        } else {
          record_error(kErrValue);
        }
      }
    }
#pragma unroll
    for (int u = 0; u < kGroupedUnroll; ++u) {
      const int q = base + u * kGroupedThreads + threadIdx.x;
      const int r = q / segs_row;
      const int sg = q - r * segs_row;
      const int col = col_base + sg * 8;

      uint32_t acc = 0;
      acc = absmax2(acc, v[u].x); acc = absmax2(acc, v[u].y);
      acc = absmax2(acc, v[u].z); acc = absmax2(acc, v[u].w);
#pragma unroll
      for (int x = 1; x < SEG_PER_BLOCK; x <<= 1) acc = absmax2(acc, __shfl_xor_sync(0xFFFFFFFFu, acc, x));
      const float amax = absmax_final(acc);

      BlockScale sc;
      if constexpr (FMT == kNVFP4) sc = nvfp4_scale(amax, tsf);
      else sc = mx_scale<FMT == kMXFP4 ? 6 : 448>(amax);

      const int64_t d = dst0 + r;
      if constexpr (Fmt<FMT>::OUT_BITS == 4) {
        const uint32_t o = quant8_e2m1(v[u], sc.factor);
        if (ok[u]) *reinterpret_cast<uint32_t*>(a.out + d * a.out_ld + (col >> 1)) = o;
      } else {
        const uint2 o = quant8_e4m3(v[u], sc.factor);
        if (ok[u]) *reinterpret_cast<uint2*>(a.out + d * a.out_ld + col) = o;
      }

      // scale word of (row r, atom): byte of block j at bits 8j
      const int blk_in_atom = (sg / SEG_PER_BLOCK) & 3;
      uint32_t word = sc.byte << (8 * blk_in_atom);
#pragma unroll
      for (int x = SEG_PER_BLOCK; x < SEG_PER_ATOM; x <<= 1) word |= __shfl_xor_sync(0xFFFFFFFFu, word, x);
      if (ok[u] && (sg % SEG_PER_ATOM) == 0) {
        const int atom = atom0 + sg / SEG_PER_ATOM;
        *reinterpret_cast<uint32_t*>(band + atom * 512 + (r & 31) * 16 + (r >> 5) * 4) = word;
      }
    }
  }
}

}  // namespace bsq
