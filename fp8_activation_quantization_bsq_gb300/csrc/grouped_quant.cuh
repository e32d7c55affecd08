// Grouped per-expert block-scaled quantization (MoE activations).
//
// Each destination row d belongs to the group g with row_offsets[g] <= d <
// row_offsets[g+1]; its scales go to 5D row scales_offsets[g] + (d -
// row_offsets[g]) (groups padded to whole 128-row tiles), its NVFP4 tensor
// scale is sf_tensor[expert_ids[g]], and it reads source row row_indices[d]
// (or d).  Three kernels, one per regime, give identical bytes:
//
//  * grouped_band_kernel (groups of many rows, prefill).  A thread block
//    owns 32 consecutive destination rows, whichever groups they belong to,
//    and a run of scale blocks.  Warp 0 finds the first row's group by
//    searching row_offsets with all 32 lanes (rounds of 256 probes), each lane
//    steps on to its own row's group, and the distinct expert scales of the
//    32 rows get shared element-scale tables.  Then each warp walks its rows
//    one at a time with its 32 lanes on 32 consecutive 32-element chunks of
//    the row (two NVFP4 scale blocks or one MX block per lane): gathered
//    loads and packed stores are contiguous per instruction (whole L1
//    lines, not one sector per lane), with one (NVFP4) or two (MX) steps of
//    loads in flight, and the lanes of one atom OR their scale bytes into
//    its word.
//
//  * grouped_rows_kernel (groups of a few rows, decode).  A warp owns R
//    consecutive destination rows and one run of k_tiles_per_block atom
//    columns, whatever the group sizes.  Lane r resolves row d0 + r by a
//    binary search over row_offsets (the group tables staged in shared
//    memory by one coalesced pass when G <= 1024), then the rows' scale
//    blocks are spread over the lanes, consecutive blocks on consecutive
//    lanes, each lane quantizing whole blocks; the scale bytes of a row's
//    atom are OR-reduced over 4 lanes into one word.
//
//  * grouped_token_kernel (grouped_token.cuh; a row_indices gather that
//    reuses source rows, top-k routing).  Token-major: each source row is
//    read once and quantized into all of its destination rows.
//
// Batching column tiles per unit (k_tiles_per_block) amortizes the lookups
// and makes the grid smaller; at decode, where each unit holds only a few
// routed rows, the grid size is what the time depends on.  Blocks of the
// last atom beyond K are zero (scale 0x00).
#pragma once

#include "box_quant.cuh"
#include "device_common.cuh"

namespace bsq {

struct GroupedArgs {
  const uint16_t* in;
  int64_t ld_in;        // elements
  int64_t in_rows;
  int K;
  const uint32_t* row_offsets;
  const uint32_t* scales_offsets;
  const int32_t* expert_ids;
  const float* sf;      // null for MX formats
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
  int ktc;              // 32-element chunks per thread block (band kernel)
  uint8_t* scale_ws;    // token kernel: scale rows staged row-major here (null: straight to 5D),
                        // then one int32 per 128-row band: its rows written (ws_band_rows)
};

// Rows of 5D band b (scale rows 128 b ..) that the grouped quantize writes:
// with g the last group with scales_offsets[g] <= 128 b, the band's rows
// that are destination rows of g below min(row_offsets[G], total_rows); 0
// when g is skipped (expert id < 0 or, NVFP4, >= num_experts) or no group
// starts at or below the band.  ro / so / e: the group metadata (any
// memory space).
__device__ __forceinline__ int band_rows_written(const GroupedArgs& a, const uint32_t* ro, const uint32_t* so,
                                                 const int32_t* e, int64_t b) {
  const int64_t s0 = b * 128;
  int lo = 0, hi = a.G;  // g = max{g : so[g] <= s0}
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (static_cast<int64_t>(so[mid]) <= s0) lo = mid;
    else hi = mid - 1;
  }
  if (lo >= a.G || static_cast<int64_t>(so[lo]) > s0) return 0;
  const int ex = e[lo];
  if (ex < 0 || (a.sf != nullptr && ex >= a.num_experts)) return 0;
  const int64_t ro_end = ro[a.G];
  const int64_t rows = ro_end < a.total_rows ? ro_end : a.total_rows;
  const int64_t r_end = ro[lo + 1];
  const int64_t first = static_cast<int64_t>(ro[lo]) + (s0 - so[lo]);
  int64_t n = (r_end < rows ? r_end : rows) - first;
  return static_cast<int>(n < 0 ? 0 : (n > 128 ? 128 : n));
}
__device__ __forceinline__ int32_t* ws_band_rows(const GroupedArgs& a) {
  return reinterpret_cast<int32_t*>(a.scale_ws + a.total_scale_rows * static_cast<int64_t>(a.kt_atoms) * 4);
}

// Checks of the offsets' first and last entries (one thread reports).
__device__ __forceinline__ void check_offsets(const GroupedArgs& a) {
  if (__ldg(a.row_offsets) != 0u || __ldg(a.scales_offsets) != 0u ||
      static_cast<int64_t>(__ldg(a.row_offsets + a.G)) > a.total_rows ||
      static_cast<int64_t>(__ldg(a.scales_offsets + a.G)) > a.total_scale_rows)
    record_error(kErrValue);
}

// ------------------------------------------------------ grouped_band_kernel --

// Warps per block: 4 (with 63-70 registers per thread, blocks of 4 warps
// keep 6-7 blocks resident per SM).
template <int FMT>
__host__ __device__ constexpr int band_warps() { return 4; }
constexpr int kBdRows = 32;        // destination rows per block
constexpr int kBdTables = 2;       // distinct tensor scales of the band with a shared element-scale table

struct BdRow {
  int64_t src;       // source row
  int64_t dst;       // destination row
  int64_t band;      // byte offset of the row's 128-row band in the 5D scales
  int atom_off;      // the row's word inside an atom
  int tab;           // factor table slot, -1: divide
  float tsf;
  int ok;            // quantize this row
};

// g = max{g : row_offsets[g] <= d} for a warp-uniform d: rounds of 256
// probes (8 per lane) narrow [lo, hi) until it holds one group.
__device__ __forceinline__ int band_group_of(const GroupedArgs& a, int64_t d) {
  const int lane = threadIdx.x & 31;
  int lo = 0, hi = a.G;  // ro[lo] <= d < ro[hi] (ro[G] > d is guaranteed by the caller)
  while (hi - lo > 1) {
    const int step = (hi - lo + 255) >> 8;
    int cnt = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int64_t pos = lo + static_cast<int64_t>(step) * (1 + lane + 32 * i);
      cnt += __popc(__ballot_sync(0xFFFFFFFFu, pos < hi && static_cast<int64_t>(__ldg(a.row_offsets + pos)) <= d));
    }
    const int nlo = lo + cnt * step;
    hi = min(hi, nlo + step);
    lo = nlo;
  }
  return lo;
}

// Quantize one MX scale block held in registers (32 elements) to dst;
// returns the block's scale byte.
template <int FMT>
__device__ __forceinline__ uint32_t band_block(const uint4 (&v)[4], uint8_t* dst, bool out_vec32,
                                               const NvScale& ns) {
  uint32_t acc = 0;
#pragma unroll
  for (int c = 0; c < Fmt<FMT>::SF / 8; ++c) {
    acc = absmax2(acc, v[c].x); acc = absmax2(acc, v[c].y);
    acc = absmax2(acc, v[c].z); acc = absmax2(acc, v[c].w);
  }
  const float amax = absmax_final(acc);
  if constexpr (FMT == kNVFP4) {
    const BlockScale sc = nvfp4_block_scale(amax, ns);
    *reinterpret_cast<uint2*>(dst) = make_uint2(quant8_e2m1(v[0], sc.factor), quant8_e2m1(v[1], sc.factor));
    return sc.byte;
  } else if constexpr (FMT == kMXFP4) {
    const MxScale sc = mx_scale<6>(amax);
    st_global_v4(dst, quant8_e2m1_pow2(v[0], sc.pow2), quant8_e2m1_pow2(v[1], sc.pow2),
                 quant8_e2m1_pow2(v[2], sc.pow2), quant8_e2m1_pow2(v[3], sc.pow2));
    return sc.byte;
  } else {
    const MxScale sc = mx_scale<448>(amax);
    uint32_t o[8];
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const uint2 q = quant8_e4m3_pow2(v[c], sc.pow2);
      o[2 * c] = q.x;
      o[2 * c + 1] = q.y;
    }
    if (out_vec32) {
      st_global_v8(dst, o);
    } else {
      st_global_v4(dst, o[0], o[1], o[2], o[3]);
      st_global_v4(dst + 16, o[4], o[5], o[6], o[7]);
    }
    return sc.byte;
  }
}

// One 32-element chunk of a row from global memory (64 bytes).
__device__ __forceinline__ void band_load(uint4 (&v)[4], const uint16_t* p, bool vec32) {
  if (vec32) {
    ld_global_nc_v8(p, v[0], v[1]);
    ld_global_nc_v8(p + 16, v[2], v[3]);
  } else {
#pragma unroll
    for (int c = 0; c < 4; ++c) v[c] = ld_global_nc_v4(p + 8 * c);
  }
}

// Quantize one 32-element chunk of a row held in registers (two NVFP4
// blocks or one MX block) to dst; returns its scale bytes (NVFP4: block 0 in
// bits 0-7, block 1 in bits 8-15).
template <int FMT>
__device__ __forceinline__ uint32_t band_chunk(const uint4 (&v)[4], uint8_t* dst, bool out_vec32, const NvScale& ns) {
  if constexpr (FMT == kNVFP4) {
    uint32_t o[4], bytes = 0;
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      uint32_t acc = 0;
#pragma unroll
      for (int c = 2 * j; c < 2 * j + 2; ++c) {
        acc = absmax2(acc, v[c].x); acc = absmax2(acc, v[c].y);
        acc = absmax2(acc, v[c].z); acc = absmax2(acc, v[c].w);
      }
      const BlockScale sc = nvfp4_block_scale(absmax_final(acc), ns);
      o[2 * j] = quant8_e2m1(v[2 * j], sc.factor);
      o[2 * j + 1] = quant8_e2m1(v[2 * j + 1], sc.factor);
      bytes |= sc.byte << (8 * j);
    }
    st_global_v4(dst, o[0], o[1], o[2], o[3]);
    return bytes;
  } else {
    return band_block<FMT>(v, dst, out_vec32, ns);
  }
}

// One chunk step of a band row: lane chunk ch (< c_end), data in v; the
// lanes of one atom OR their scale bytes into its word.
template <int FMT>
__device__ __forceinline__ void band_chunk_step(const uint4 (&v)[4], int ch, int n_chunks, int c_end,
                                                uint8_t* out_row, uint8_t* scale_row, bool out_vec32,
                                                const NvScale& ns) {
  constexpr int BPL = 32 / Fmt<FMT>::SF;  // scale blocks per chunk
  constexpr int CPA = 4 / BPL;            // chunks per atom
  const int lane = threadIdx.x & 31;
  uint32_t bytes = 0;  // padding blocks of the last atom stay 0x00
  if (ch < n_chunks && ch < c_end)
    bytes = band_chunk<FMT>(v, out_row + (Fmt<FMT>::OUT_BITS == 4 ? 16 * ch : 32 * ch), out_vec32, ns);
  uint32_t word = bytes << (8 * BPL * (lane % CPA));
#pragma unroll
  for (int m = 1; m < CPA; m <<= 1) word |= __shfl_xor_sync(0xFFFFFFFFu, word, m);
  // (the atom's 32-byte sectors fill from rows of 4 blocks: kept in L2 until
  // complete by an evict_last hint; the next ordinary read returns them to
  // normal priority)
  if (lane % CPA == 0 && ch < c_end) {
    const uint64_t keep = l2_policy_evict_last();
    asm volatile("st.global.L2::cache_hint.b32 [%0], %1, %2;" ::"l"(scale_row + (ch / CPA) * 512), "r"(word),
                 "l"(keep)
                 : "memory");
  }
}

// A block owns kBdRows consecutive destination rows (across group boundaries)
// and a run of a.ktc 32-element chunks (a multiple of 32).  Warp 0 resolves the
// rows: one warp-wide search for the first row's group, then each lane steps
// forward to its own row's group; the first kBdTables distinct tensor scales
// among the rows get a 256-entry element-scale table (NVFP4).  Warp w then
// takes rows w, w + kBdWarps, ...: for each, the 32 lanes hold 32 consecutive
// 32-element chunks of the row (two NVFP4 or one MX scale block each: 2 KB
// of contiguous loads and 512 B / 1 KB of contiguous stores per step), and
// the lanes of one atom OR their scale bytes into its word.
template <int FMT>
__global__ void __launch_bounds__(32 * band_warps<FMT>()) grouped_band_kernel(const GroupedArgs a) {
  constexpr int SF = Fmt<FMT>::SF;
  constexpr int kBdWarps = band_warps<FMT>();
  constexpr int kBdThreads = 32 * kBdWarps;
  __shared__ BdRow rows[kBdRows];
  __shared__ float factor_tab[kBdTables][256];
  __shared__ float div6_tab[128];
  __shared__ float tab_tsf[kBdTables];
  __shared__ int n_tabs;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int64_t d0 = static_cast<int64_t>(blockIdx.x) * kBdRows;
  if constexpr (FMT == kNVFP4) fill_div6_table(div6_tab, threadIdx.x, kBdThreads);
  pdl_wait();
  if (blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0) check_offsets(a);

  // ---- rows of the band (warp 0)
  if (warp == 0) {
    const int64_t d = d0 + lane;
    BdRow st{0, d, 0, 0, -1, 1.0f, 0};
    const int64_t ro_end = static_cast<int64_t>(__ldg(a.row_offsets + a.G));
    const int64_t d_lim = ro_end < a.total_rows ? ro_end : a.total_rows;  // rows inside groups
    if (d0 < d_lim) {
      int g = band_group_of(a, d0);
      if (d < d_lim) {
        // step forward to this row's group (consecutive rows: a few groups at most)
        while (g + 1 < a.G && static_cast<int64_t>(__ldg(a.row_offsets + g + 1)) <= d) ++g;
        const int64_t r_beg = __ldg(a.row_offsets + g), r_end = __ldg(a.row_offsets + g + 1);
        const int64_t so_g = __ldg(a.scales_offsets + g), so_n = __ldg(a.scales_offsets + g + 1);
        const int e = __ldg(a.expert_ids + g);
        const int64_t srow = so_g + (d - r_beg);
        if (r_end - r_beg < 0 || r_end - r_beg > so_n - so_g || r_end > a.total_rows ||
            srow >= a.total_scale_rows || d < r_beg || d >= r_end ||
            (a.sf != nullptr && e >= a.num_experts)) {
          record_error(kErrValue);
        } else if (e >= 0) {
          const int64_t src = a.row_indices ? static_cast<int64_t>(__ldg(a.row_indices + d)) : d;
          if (src < 0 || src >= a.in_rows) {
            record_error(kErrValue);
          } else {
            st.src = src;
            st.band = (srow >> 7) * static_cast<int64_t>(a.kt_atoms) * 512;
            st.atom_off = static_cast<int>((srow & 31) * 16 + ((srow & 127) >> 5) * 4);
            st.ok = 1;
            if (a.sf != nullptr) st.tsf = __ldg(a.sf + e);
          }
        }
      }
    }
    if constexpr (FMT == kNVFP4) {
      // table slots: the lowest lane of each distinct tensor scale leads its
      // lanes; leaders in lane order take the first kBdTables slots
      const uint32_t key = st.ok ? __float_as_uint(st.tsf) : 0xFFFFFFFFu;
      const uint32_t same = __match_any_sync(0xFFFFFFFFu, key);
      const int leader = __ffs(same) - 1;
      const uint32_t leaders = __ballot_sync(0xFFFFFFFFu, st.ok && leader == lane);
      const int rank = __popc(leaders & ((1u << leader) - 1u));
      st.tab = st.ok && rank < kBdTables ? rank : -1;
      if (st.ok && leader == lane && rank < kBdTables) tab_tsf[rank] = st.tsf;
      if (lane == 0) n_tabs = min(__popc(leaders), kBdTables);
    }
    rows[lane] = st;
  }
  __syncthreads();
  if constexpr (FMT == kNVFP4) {
    for (int t = 0; t < n_tabs; ++t) fill_nvfp4_factor_table(factor_tab[t], tab_tsf[t], threadIdx.x, kBdThreads);
    __syncthreads();
  }

  // ---- quantize: warp -> rows, lane -> 32-element chunks
  constexpr int CPA = 4 / (32 / SF);            // chunks per 5D atom
  const int n_chunks = a.K / 32;                // chunks per row
  const int c_pad = a.kt_atoms * CPA;           // with the last atom's padding
  const int c_beg = blockIdx.y * a.ktc;
  const int c_end = min(c_pad, c_beg + a.ktc);
  const int lim = min(n_chunks, c_end);         // chunks with data
  const bool in_vec32 = a.in_vec32 != 0, out_vec32 = a.out_vec32 != 0;
  for (int r = warp; r < kBdRows; r += kBdWarps) {
    const BdRow row = rows[r];
    if (!row.ok) continue;  // warp-uniform
    const uint16_t* in_row = a.in + row.src * a.ld_in;
    uint8_t* out_row = a.out + row.dst * a.out_ld;
    uint8_t* scale_row = a.scales + row.band + row.atom_off;
    const NvScale ns{row.tsf, row.tab >= 0 ? factor_tab[row.tab] : nullptr, div6_tab};
    int ch = c_beg + lane;  // this lane's chunks: ch, ch + 32, ...
    if constexpr (FMT == kNVFP4) {
      // two alternating buffers, one step of loads ahead (fewer registers,
      // more resident warps: the better trade for the NVFP4 arithmetic)
      uint4 va[4], vb[4];
      if (ch < lim) band_load(va, in_row + 32 * ch, in_vec32);
#pragma unroll 1
      for (int c0 = c_beg; c0 < c_end; c0 += 64, ch += 64) {
        if (ch + 32 < lim) band_load(vb, in_row + 32 * (ch + 32), in_vec32);
        band_chunk_step<FMT>(va, ch, n_chunks, c_end, out_row, scale_row, out_vec32, ns);
        if (c0 + 32 >= c_end) break;
        if (ch + 64 < lim) band_load(va, in_row + 32 * (ch + 64), in_vec32);
        band_chunk_step<FMT>(vb, ch + 32, n_chunks, c_end, out_row, scale_row, out_vec32, ns);
      }
    } else {
      // two steps of loads ahead
      uint4 v0[4], v1[4];
      if (ch < lim) band_load(v0, in_row + 32 * ch, in_vec32);
      if (ch + 32 < lim) band_load(v1, in_row + 32 * (ch + 32), in_vec32);
#pragma unroll 1
      for (int c0 = c_beg; c0 < c_end; c0 += 32, ch += 32) {
        uint4 v[4];
#pragma unroll
        for (int c = 0; c < 4; ++c) { v[c] = v0[c]; v0[c] = v1[c]; }
        if (ch + 64 < lim) band_load(v1, in_row + 32 * (ch + 64), in_vec32);
        band_chunk_step<FMT>(v, ch, n_chunks, c_end, out_row, scale_row, out_vec32, ns);
      }
    }
  }
}

// ------------------------------------------------------ grouped_rows_kernel --

constexpr int kGrWarps = 4;
constexpr int kGrThreads = 32 * kGrWarps;
constexpr int kGrStageGroups = 1024;  // group tables staged in shared memory up to this many groups / experts

// Per-row state of a warp's rows, in shared memory so that any lane can read
// the row of the block it holds.
struct alignas(16) RowState {
  int64_t src;     // source row (input)
  int64_t dst;     // destination row (packed output)
  int64_t band;    // byte offset of the 5D row band of the scale row
  int atom_off;    // (srow % 32) * 16 + ((srow % 128) / 32) * 4
  int ok;          // quantize this row
  float tsf;
};

template <int FMT, int KT, int R>
__global__ void __launch_bounds__(kGrThreads) grouped_rows_kernel(const GroupedArgs a) {
  static_assert(R <= 32, "one lane per row");
  constexpr int SF = Fmt<FMT>::SF;
  constexpr int BPR = 4 * KT;                       // scale blocks per row in a run
  constexpr int LOG_BPR = KT == 1 ? 2 : KT == 2 ? 3 : KT == 4 ? 4 : 5;
  constexpr int SLOTS = (R * BPR + 31) / 32;        // blocks per lane
  constexpr int U = FMT != kNVFP4 ? (SLOTS < 4 ? SLOTS : 4) : (SLOTS < 8 ? SLOTS : 8);

  __shared__ RowState rs_all[kGrWarps][R];
  __shared__ float div6_tab[128];
  __shared__ uint32_t ro_s[kGrStageGroups + 1], so_s[kGrStageGroups + 1];
  __shared__ int32_t e_s[kGrStageGroups];
  __shared__ float sf_s[kGrStageGroups];
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  if constexpr (FMT == kNVFP4) fill_div6_table(div6_tab, threadIdx.x, kGrThreads);
  pdl_wait();

  const int64_t d0_blk = static_cast<int64_t>(blockIdx.x) * kGrWarps * R;
  if (d0_blk >= a.total_rows) return;  // block-uniform
  const int64_t d0 = d0_blk + static_cast<int64_t>(warp) * R;
  RowState* rs = rs_all[warp];
  if (blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0) check_offsets(a);
  // the row's source index does not depend on its group: in flight first
  const int64_t dl = d0 + lane;
  const int64_t src_pre =
      (lane < R && dl < a.total_rows && a.row_indices) ? static_cast<int64_t>(__ldg(a.row_indices + dl)) : dl;
  // the group tables in shared memory (one coalesced pass) when they fit, so
  // that resolving a row costs no chain of dependent global loads
  const bool staged = a.G <= kGrStageGroups && (a.sf == nullptr || a.num_experts <= kGrStageGroups);
  if (staged) {
    for (int i = threadIdx.x; i <= a.G; i += kGrThreads) {
      ro_s[i] = __ldg(a.row_offsets + i);
      so_s[i] = __ldg(a.scales_offsets + i);
      if (i < a.G) e_s[i] = __ldg(a.expert_ids + i);
    }
    if (a.sf != nullptr)
      for (int i = threadIdx.x; i < a.num_experts; i += kGrThreads) sf_s[i] = __ldg(a.sf + i);
  }
  __syncthreads();
  if (d0 >= a.total_rows) return;

  // ---- lane r resolves row d0 + r
  if (lane < R) {
    const int64_t d = dl;
    RowState st{d, d, 0, 0, 0, 1.0f};
    const int64_t ro_end =
        d < a.total_rows ? static_cast<int64_t>(staged ? ro_s[a.G] : __ldg(a.row_offsets + a.G)) : 0;
    if (d < ro_end) {
      // g = max{g : ro[g] <= d}: binary search for the first ro[g+1] > d
      int lo = 0, hi = a.G - 1;
      while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if (static_cast<int64_t>(staged ? ro_s[mid + 1] : __ldg(a.row_offsets + mid + 1)) <= d) lo = mid + 1;
        else hi = mid;
      }
      const int64_t r_beg = staged ? ro_s[lo] : __ldg(a.row_offsets + lo);
      const int64_t r_end = staged ? ro_s[lo + 1] : __ldg(a.row_offsets + lo + 1);
      const int64_t so_g = staged ? so_s[lo] : __ldg(a.scales_offsets + lo);
      const int64_t so_n = staged ? so_s[lo + 1] : __ldg(a.scales_offsets + lo + 1);
      const int e = staged ? e_s[lo] : __ldg(a.expert_ids + lo);
      const int64_t srow = so_g + (d - r_beg);
      if (r_end - r_beg < 0 || r_end - r_beg > so_n - so_g || r_end > a.total_rows ||
          srow >= a.total_scale_rows || d < r_beg || (a.sf != nullptr && e >= a.num_experts)) {
        record_error(kErrValue);
      } else if (e >= 0) {
        const int64_t src = src_pre;
        if (src < 0 || src >= a.in_rows) {
          record_error(kErrValue);
        } else {
          st.src = src;
          st.band = (srow >> 7) * static_cast<int64_t>(a.kt_atoms) * 512;
          st.atom_off = static_cast<int>((srow & 31) * 16 + ((srow & 127) >> 5) * 4);
          st.ok = 1;
          if (a.sf != nullptr) st.tsf = staged ? sf_s[e] : __ldg(a.sf + e);
        }
      }
    }
    rs[lane] = st;
  }
  __syncwarp();

  // ---- quantize the warp's (row, block) slots
  const int atom0 = blockIdx.y * KT;
  const int col_base = atom0 * 4 * SF;
#pragma unroll
  for (int j0 = 0; j0 < SLOTS; j0 += U) {
    uint4 v[U][SF / 8];
    bool ok[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int q = (j0 + u) * 32 + lane;
      const int r = q >> LOG_BPR;
      const int col = col_base + (q & (BPR - 1)) * SF;
#pragma unroll
      for (int c = 0; c < SF / 8; ++c) v[u][c] = make_uint4(0u, 0u, 0u, 0u);
      ok[u] = r < R && col < a.K && rs[r < R ? r : 0].ok;
      if (ok[u]) {
        const uint16_t* p = a.in + rs[r].src * a.ld_in + col;
        if (a.in_vec32) {
#pragma unroll
          for (int c = 0; c < SF / 8; c += 2) ld_global_nc_v8(p + 8 * c, v[u][c], v[u][c + 1]);
        } else {
#pragma unroll
          for (int c = 0; c < SF / 8; ++c) v[u][c] = ld_global_nc_v4(p + 8 * c);
        }
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int q = (j0 + u) * 32 + lane;
      const int r = (q >> LOG_BPR) < R ? (q >> LOG_BPR) : 0;
      const int b = q & (BPR - 1);
      const int col = col_base + b * SF;
      uint32_t acc = 0;
#pragma unroll
      for (int c = 0; c < SF / 8; ++c) {
        acc = absmax2(acc, v[u][c].x); acc = absmax2(acc, v[u][c].y);
        acc = absmax2(acc, v[u][c].z); acc = absmax2(acc, v[u][c].w);
      }
      const float amax = absmax_final(acc);
      uint8_t* dst = a.out + rs[r].dst * a.out_ld + (Fmt<FMT>::OUT_BITS == 4 ? col >> 1 : col);
      uint32_t sbyte;
      if constexpr (FMT == kNVFP4) {
        const NvScale ns{rs[r].tsf, nullptr, div6_tab};
        const BlockScale sc = nvfp4_block_scale(amax, ns);
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
        *reinterpret_cast<uint32_t*>(a.scales + rs[r].band + atom * 512 + rs[r].atom_off) = word;
      }
    }
  }
}

// ------------------------------------------------------ NVFP4 factor table --

// NVFP4 element scale tsf / ds for one destination row without a division.
// A positive E4M3 scale byte b decodes to ds = m * 2^-(shift) with m a small
// integer: b = E.f (4 exponent, 3 fraction bits), m = 8 + f and
// shift = 10 - E when E > 0, m = f and shift = 9 when E = 0.  So
// tsf / ds = (tsf / m) * 2^shift, and fl(tsf / ds) = fl(tsf / m) * 2^shift
// exactly whenever both sides are normal FP32 numbers, which holds for every
// reachable (m, shift) when 2^-117 <= tsf <= 2^118.  tab[m] = fl(tsf / m)
// (tab[0] = 0: ds = 0 gives factor 0); other tsf use the division.
__device__ __forceinline__ bool tk_factor_table_ok(float tsf) {
  return tsf >= 0x1p-117f && tsf <= 0x1p118f;
}
__device__ __forceinline__ float tk_factor(const float* tab, uint32_t b) {
  const uint32_t E = b >> 3;
  const uint32_t m = (b & 7u) | (E != 0u ? 8u : 0u);
  const uint32_t e_eff = E != 0u ? E : 1u;
  return __fmul_rn(tab[m], __uint_as_float((137u - e_eff) << 23));  // * 2^(10 - e_eff)
}

}  // namespace bsq
