// Token-major grouped quantize for row_indices gathers that reuse source rows
// (top-k MoE routing: every token row feeds k destination rows).
//
// Persistent: one 1024-thread block per SM, each owning an equal share of
// the source rows (tokens), so every SM gets the same work when tokens carry
// the same number of destination rows.  A block
//   (1) issues each warp's first token-row loads and the group metadata
//       loads (held in registers), then scans all of row_indices itself
//       (staged by bulk copies; the 128 KB of a 32768-row prefill stay in L2
//       for the other blocks) and files every destination row whose source
//       row it owns into a per-token bucket in shared memory;
//   (2) builds, per token, the list of its destination rows (group, 5D scale
//       row, expert scale: the same checks as the other grouped kernels);
//   (3) streams the token row once, 32 lanes on 32 consecutive scale blocks
//       per step, computing each block's maximum and widening its elements
//       to FP32 once, then for every destination row only the per-row scale,
//       the products and the conversions (MX: the codes do not depend on the
//       row and are encoded once, then stored per row).
// Warp w takes tokens w, w + 32, ...; a block with at most kTqUnitTokens
// tokens (fewer than its warps) instead lets its warps claim (token, step)
// units from a shared-memory counter, so that every warp works.
// A token with more destination rows than a bucket holds is left to a
// re-scan after the others (rare: never with top-k routing to distinct
// experts); its rows are then quantized one at a time.
//
// Scale bytes go to their 5D positions, or, with a caller workspace, to a
// row-major staging row per 5D scale row (scale_ws): one destination row's
// 32 scale bytes of a step then fill one 32-byte sector instead of landing
// in 8 atoms 512 bytes apart (8 partial sectors per store instruction), and
// grouped_scale_ws_kernel moves the staged rows to the 5D layout afterwards
// with whole-atom stores, writing only the rows the quantize wrote.
//
// NVFP4 element scale tsf / ds without a division: per expert a table of
// fl32(tsf / m), m = 1..15, and tk_factor's power-of-two step (exact for
// 2^-117 <= tsf <= 2^118; other scales divide).
#pragma once

#include "grouped_quant.cuh"
#include "interleave.cuh"

namespace bsq {

constexpr int kTqWarps = 32;
constexpr int kTqThreads = 32 * kTqWarps;
constexpr int kTqBucket = 16;        // destination rows kept per token (more: the re-scan path)
constexpr int kTqMaxTokens = 512;    // tokens per block at most (more: more blocks)
constexpr int kTqMaxGroups = 1024;   // group metadata held in shared memory
constexpr int kTqTabExperts = 1024;  // NVFP4: experts with a factor table in shared memory
constexpr int kTqStageInts = 16384;  // row_indices entries per staging buffer at most (64 KB)
constexpr int kTqScanVec = 1;      // staged row_indices vectors tested per thread at a time
constexpr int kTqUnitTokens = 16;    // tokens per block at most for claimed (token, step) units
constexpr int kTqBadList = 64;       // out-of-range source rows block 0 keeps for the check (more: a re-scan)
static_assert(kTqMaxGroups + 1 <= 2 * kTqThreads && kTqTabExperts <= kTqThreads,
              "the token kernel's threads hold the metadata in registers during the scan");

// One destination row of the token a warp is quantizing.
struct alignas(16) TqDesc {
  uint8_t* out;    // its packed row
  uint8_t* scale;  // its byte in the first 5D atom of its scale row
  float tsf;       // NVFP4 tensor scale of its expert
  int tab;         // NVFP4: offset of the expert's factor table (floats), -1: divide
};

struct TqShared {
  uint32_t ro[kTqMaxGroups + 1];
  uint32_t so[kTqMaxGroups + 1];
  int32_t e[kTqMaxGroups];
  TqDesc desc[kTqWarps][kTqBucket];
  float div6_tab[128];
  uint64_t stage_bar[2];  // completion of the two row_indices staging buffers
  uint32_t heavy;         // some token of this block has more rows than its bucket
  uint32_t failed;        // a staging wait expired
  uint32_t n_bad;         // block 0: source rows outside x seen by the scan
  uint32_t next_unit;     // runs: the next (token, step) unit to claim
  uint32_t bad_d[kTqBadList];
  int32_t bad_src[kTqBadList];
};

// Launch constants of the token kernel (host-computed).
struct TqArgs {
  int64_t n_tok;  // source rows split over the blocks
  int tpb;        // tokens per block at most (size of the buckets)
  int n_tab;      // NVFP4 experts with a factor table (0: every row divides)
  int stage_ints; // row_indices entries per staging buffer (a multiple of 4)
  int units;      // warps claim (token, step) units; else warp w takes tokens w, w + 32, ...
};

// Dynamic shared memory: TqShared, two row_indices staging buffers, the
// buckets (tpb counts and tpb x kTqBucket rows) and the NVFP4 tables.
__host__ __device__ constexpr size_t tq_smem_bytes(int tpb, int n_tab, int stage_ints) {
  return sizeof(TqShared) + static_cast<size_t>(stage_ints) * 8 + static_cast<size_t>(tpb) * (kTqBucket + 1) * 4 +
         static_cast<size_t>(n_tab) * 64;
}

// 1D bulk copy (TMA) of `bytes` (a multiple of 16, both addresses 16-byte
// aligned) from global to shared memory, completing on `bar`.
__device__ __forceinline__ void bulk_load(void* smem_dst, const void* gsrc, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_addr(smem_dst)),
      "l"(gsrc), "r"(bytes), "r"(smem_addr(bar))
      : "memory");
}

// Destination row d (< min(row_offsets[G], total_rows)) reading source row
// src: the checks of the other kernels, on group metadata in shared memory.
// True (with the 5D scale row and the expert) when d is to be quantized;
// BSQ_ERR_VALUE for inconsistent metadata and for a source row outside x in
// a kept group.
__device__ __forceinline__ bool tq_check(const GroupedArgs& a, const TqShared& sh, int64_t d, int64_t src,
                                         int64_t& srow_out, int& e_out) {
  int lo = 0, hi = a.G - 1;  // g = max{g : ro[g] <= d}
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (static_cast<int64_t>(sh.ro[mid + 1]) <= d) lo = mid + 1;
    else hi = mid;
  }
  const int64_t r_beg = sh.ro[lo], r_end = sh.ro[lo + 1], so_g = sh.so[lo], so_n = sh.so[lo + 1];
  const int e = sh.e[lo];
  const int64_t srow = so_g + (d - r_beg);
  if (r_end - r_beg < 0 || r_end - r_beg > so_n - so_g || r_end > a.total_rows ||
      srow >= a.total_scale_rows || d < r_beg || d >= r_end || (a.sf != nullptr && e >= a.num_experts)) {
    record_error(kErrValue);
    return false;
  }
  if (e < 0) return false;
  if (src < 0 || src >= a.in_rows) {
    record_error(kErrValue);
    return false;
  }
  srow_out = srow;
  e_out = e;
  return true;
}

// Lanes [0, n) hold candidate destination rows d of source row t; the valid
// ones become the warp's descriptors 0..(count-1).  Returns the count.
template <int FMT>
__device__ __forceinline__ int tq_describe(const GroupedArgs& a, TqShared& sh, TqDesc* desc, bool cand,
                                           int64_t d, int64_t t, int n_tab) {
  const int lane = threadIdx.x & 31;
  int64_t srow = 0;
  int e = 0;
  const bool ok = cand && tq_check(a, sh, d, t, srow, e);
  const uint32_t m = __ballot_sync(0xFFFFFFFFu, ok);
  if (ok) {
    TqDesc dd;
    dd.out = a.out + d * a.out_ld;
    dd.scale = a.scale_ws != nullptr
                   ? a.scale_ws + srow * static_cast<int64_t>(a.kt_atoms) * 4  // row-major staging row
                   : a.scales + (srow >> 7) * static_cast<int64_t>(a.kt_atoms) * 512 + (srow & 31) * 16 +
                         ((srow & 127) >> 5) * 4;
    dd.tsf = 1.0f;
    dd.tab = -1;
    if constexpr (FMT == kNVFP4) {
      dd.tsf = __ldg(a.sf + e);
      if (e < n_tab && tk_factor_table_ok(dd.tsf)) dd.tab = e * 16;
    }
    desc[__popc(m & ((1u << lane) - 1u))] = dd;
  }
  __syncwarp();
  return __popc(m);
}

// A lane's step data: one NVFP4 block (16 elements) or one MX block (32).
template <int FMT> struct TqChunk { uint4 v[Fmt<FMT>::SF / 8]; };

template <int FMT>
__device__ __forceinline__ void tq_load(TqChunk<FMT>& c, const uint16_t* p, bool vec32) {
#pragma unroll
  for (int i = 0; i < Fmt<FMT>::SF / 8; i += 2) {
    if (vec32) {
      ld_global_nc_v8(p + 8 * i, c.v[i], c.v[i + 1]);
    } else {
      c.v[i] = ld_global_nc_v4(p + 8 * i);
      c.v[i + 1] = ld_global_nc_v4(p + 8 * (i + 1));
    }
  }
}

template <int FMT>
__device__ __forceinline__ void tq_zero(TqChunk<FMT>& c) {
#pragma unroll
  for (int i = 0; i < Fmt<FMT>::SF / 8; ++i) c.v[i] = make_uint4(0u, 0u, 0u, 0u);
}

// 8 FP32 values (four pairs, element 0 first) -> 8 E2M1 codes in one word.
__device__ __forceinline__ uint32_t e2m1_word(float2 p0, float2 p1, float2 p2, float2 p3) {
  uint32_t r;
  asm("{\n\t.reg .b8 q0, q1, q2, q3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 q0, %2, %1;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 q1, %4, %3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 q2, %6, %5;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 q3, %8, %7;\n\t"
      "mov.b32 %0, {q0, q1, q2, q3};\n\t}"
      : "=r"(r)
      : "f"(p0.x), "f"(p0.y), "f"(p1.x), "f"(p1.y), "f"(p2.x), "f"(p2.y), "f"(p3.x), "f"(p3.y));
  return r;
}

// Scale-byte store with an L2 cache policy.
__device__ __forceinline__ void st_global_u8_policy(void* p, uint32_t v, uint64_t pol) {
  asm volatile("st.global.L2::cache_hint.u8 [%0], %1, %2;" ::"l"(p), "r"(v), "l"(pol) : "memory");
}
__device__ __forceinline__ void st_global_v2(void* p, uint32_t a, uint32_t b) {
  asm volatile("st.global.v2.b32 [%0], {%1, %2};" ::"l"(p), "r"(a), "r"(b) : "memory");
}

// The warp quantizes the scale blocks [jb, je) of source row in_row (jb a
// multiple of 32, je <= the row's blocks with a scale byte) into its nv
// described destination rows, 32 blocks per step, lane l on block jb + l,
// jb + 32 + l, ...  cur holds the lane's block of the first step; on return
// it holds the lane's block next_jb + l of next_row (zeros without one).
template <int FMT>
__device__ __forceinline__ void tq_row(const GroupedArgs& a, const uint16_t* in_row, TqChunk<FMT>& cur, int jb,
                                       int je, const TqDesc* desc, int nv, const float* div6_tab,
                                       const float* tabs, const uint16_t* next_row = nullptr, int next_jb = 0) {
  constexpr int SF = Fmt<FMT>::SF;
  const int lane = threadIdx.x & 31;
  const int S = a.K / SF;          // blocks with data
  const int S4 = a.kt_atoms * 4;   // blocks with a scale byte (the last atom's padding is 0x00)
  const bool vec32 = a.in_vec32 != 0;
  // Scale bytes are stored with an L2 evict_last hint: each 32-byte sector of
  // a 5D atom collects 4-byte pieces of 8 destination rows written by other
  // warps and blocks at other times, and the hint keeps it in L2 until it is
  // complete instead of letting it go back to memory partly written (the
  // next ordinary read, e.g. the consuming matmul's, returns the lines to
  // normal priority).
  const uint64_t keep = l2_policy_evict_last();
#pragma unroll 1
  for (int j = jb + lane; j - lane < je; j += 32) {
    TqChunk<FMT> nx;
    tq_zero(nx);
    if (j - lane + 32 < je) {
      if (j + 32 < S) tq_load(nx, in_row + SF * (j + 32), vec32);
    } else if (next_row != nullptr && next_jb + lane < S) {
      tq_load(nx, next_row + SF * (next_jb + lane), vec32);  // the first step of the warp's next run
    }
    const bool has = j < S, has_scale = j < S4;
    const int64_t sc_off = a.scale_ws != nullptr ? static_cast<int64_t>(j) : static_cast<int64_t>(j >> 2) * 512 + (j & 3);
    uint32_t acc = 0;
#pragma unroll
    for (int c = 0; c < SF / 8; ++c) {
      acc = absmax2(acc, cur.v[c].x); acc = absmax2(acc, cur.v[c].y);
      acc = absmax2(acc, cur.v[c].z); acc = absmax2(acc, cur.v[c].w);
    }
    const float amax = absmax_final(acc);
    if constexpr (FMT == kNVFP4) {
      const float a6 = amax_div6(amax, div6_tab);
      float2 y[8];
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        y[4 * c + 0] = make_float2(bf16_lo(cur.v[c].x), bf16_hi(cur.v[c].x));
        y[4 * c + 1] = make_float2(bf16_lo(cur.v[c].y), bf16_hi(cur.v[c].y));
        y[4 * c + 2] = make_float2(bf16_lo(cur.v[c].z), bf16_hi(cur.v[c].z));
        y[4 * c + 3] = make_float2(bf16_lo(cur.v[c].w), bf16_hi(cur.v[c].w));
      }
      const int64_t el_off = static_cast<int64_t>(j) * 8;
#pragma unroll 1
      for (int i = 0; i < nv; ++i) {
        const TqDesc dd = desc[i];
        const uint32_t b = f32_to_e4m3(__fmul_rn(a6, dd.tsf));
        float f;
        if (dd.tab < 0) {  // warp-uniform
          const float ds = e4m3_to_f32(b);
          f = ds == 0.0f ? 0.0f : __fdiv_rn(dd.tsf, ds);
        } else {
          f = tk_factor(tabs + dd.tab, b);
        }
        const float2 ff = make_float2(f, f);
        float2 z[8];
#pragma unroll
        for (int m = 0; m < 8; ++m) z[m] = __fmul2_rn(y[m], ff);
        if (has) st_global_v2(dd.out + el_off, e2m1_word(z[0], z[1], z[2], z[3]), e2m1_word(z[4], z[5], z[6], z[7]));
        if (has_scale) st_global_u8_policy(dd.scale + sc_off, b, keep);
      }
    } else {
      const MxScale sc = mx_scale<FMT == kMXFP4 ? 6 : 448>(amax);
      const uint32_t sbyte = has ? sc.byte : 0u;
      uint32_t o[8];
      if constexpr (FMT == kMXFP4) {
#pragma unroll
        for (int c = 0; c < 4; ++c) o[c] = quant8_e2m1_pow2(cur.v[c], sc.pow2);
      } else {
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const uint2 qq = quant8_e4m3_pow2(cur.v[c], sc.pow2);
          o[2 * c] = qq.x;
          o[2 * c + 1] = qq.y;
        }
      }
      const int64_t el_off = static_cast<int64_t>(j) * (FMT == kMXFP4 ? 16 : 32);
      const bool ov32 = a.out_vec32 != 0;
#pragma unroll 1
      for (int i = 0; i < nv; ++i) {
        uint8_t* dst = desc[i].out + el_off;
        if (has) {
          if constexpr (FMT == kMXFP4) {
            st_global_v4(dst, o[0], o[1], o[2], o[3]);
          } else if (ov32) {
            st_global_v8(dst, o);
          } else {
            st_global_v4(dst, o[0], o[1], o[2], o[3]);
            st_global_v4(dst + 16, o[4], o[5], o[6], o[7]);
          }
        }
        if (has_scale) st_global_u8_policy(desc[i].scale + sc_off, sbyte, keep);
      }
    }
    cur = nx;
  }
}

// Grid: gridDim.x blocks share q.n_tok source rows evenly (block b owns
// [b n / P, (b+1) n / P)); with no row_indices destination row d reads
// source row d and n_tok covers every destination row.
template <int FMT>
__global__ void __launch_bounds__(kTqThreads, 1) grouped_token_kernel(const GroupedArgs a, const TqArgs q) {
  extern __shared__ __align__(16) uint8_t tq_smem[];
  TqShared& sh = *reinterpret_cast<TqShared*>(tq_smem);
  int4* stage = reinterpret_cast<int4*>(tq_smem + sizeof(TqShared));  // 2 x stage_ints entries
  uint32_t* cnt = reinterpret_cast<uint32_t*>(tq_smem + sizeof(TqShared) + static_cast<size_t>(q.stage_ints) * 8);
  uint32_t* bkt = cnt + q.tpb;
  float* tabs = reinterpret_cast<float*>(bkt + static_cast<int64_t>(q.tpb) * kTqBucket);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t t_lo = static_cast<int64_t>(blockIdx.x) * q.n_tok / gridDim.x;
  const int64_t t_hi = static_cast<int64_t>(blockIdx.x + 1) * q.n_tok / gridDim.x;
  const int nt = static_cast<int>(t_hi - t_lo);
  const bool gather = a.row_indices != nullptr;
  if constexpr (FMT == kNVFP4) fill_div6_table(sh.div6_tab, threadIdx.x, kTqThreads);
  for (int i = threadIdx.x; i < nt; i += kTqThreads) cnt[i] = 0u;
  // row_indices: a scalar head up to its first 16-byte boundary, a 16-byte
  // body staged into shared memory by bulk copies (chunks of stage_ints
  // entries, two buffers), a scalar tail.  All total_rows entries are
  // staged; only those below min(row_offsets[G], total_rows) are filed.
  const int64_t mis = gather ? static_cast<int64_t>(((16 - (reinterpret_cast<uintptr_t>(a.row_indices) & 15)) & 15) >> 2) : 0;
  const int64_t head = mis < a.total_rows ? mis : a.total_rows;
  const int64_t nvec = gather ? (a.total_rows - head) >> 2 : 0;   // 16-byte vectors in the body
  const int64_t cvec = q.stage_ints >> 2;                         // vectors per chunk
  const int64_t n_chunks = (nvec + cvec - 1) / cvec;
  const int4* body = reinterpret_cast<const int4*>(a.row_indices + head);
  auto chunk_bytes = [&](int64_t c) { return static_cast<uint32_t>(min(cvec, nvec - c * cvec) * 16); };
  if (threadIdx.x == 0) {
    sh.heavy = 0u;
    sh.failed = 0u;
    sh.n_bad = 0u;
    sh.next_unit = kTqWarps;  // warp w starts on unit w
    mbar_init(&sh.stage_bar[0], 1);
    mbar_init(&sh.stage_bar[1], 1);
    fence_mbar_init();
  }
  __syncthreads();
  pdl_wait();
  if (threadIdx.x == 0) {
    for (int64_t c = 0; c < 2 && c < n_chunks; ++c) {
      mbar_arrive_expect_tx(&sh.stage_bar[c], chunk_bytes(c));
      bulk_load(stage + c * cvec, body + c * cvec, chunk_bytes(c), &sh.stage_bar[c]);
    }
  }

  // the first step of each warp's first token row (units: of unit w), in
  // flight during the scan
  const int steps = (a.kt_atoms * 4 + 31) / 32;  // 32-block steps per row
  TqChunk<FMT> pre;
  tq_zero(pre);
  {
    const int k0 = q.units ? warp / steps : warp;
    const int j0 = (q.units ? (warp % steps) * 32 : 0) + lane;
    if (k0 < nt && t_lo + k0 < a.in_rows && j0 < a.K / Fmt<FMT>::SF)
      tq_load(pre, a.in + (t_lo + k0) * a.ld_in + Fmt<FMT>::SF * j0, a.in_vec32 != 0);
  }

  if (blockIdx.x == 0 && threadIdx.x == 0) check_offsets(a);
  // The group metadata and the expert scales are loaded into registers now
  // and stored to shared memory after the scan, which needs only
  // row_offsets[G]: their latency hides behind the row_indices copies.
  // G <= kTqMaxGroups = kTqThreads, so thread i holds entries i and i + 1024.
  const int64_t ro_end = static_cast<int64_t>(__ldg(a.row_offsets + a.G));
  const int64_t rows = ro_end < a.total_rows ? ro_end : a.total_rows;
  uint32_t m_ro[2] = {0u, 0u}, m_so[2] = {0u, 0u};
  int32_t m_e[2] = {0, 0};
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    const int i = static_cast<int>(threadIdx.x) + k * kTqThreads;
    if (i <= a.G) {
      m_ro[k] = __ldg(a.row_offsets + i);
      m_so[k] = __ldg(a.scales_offsets + i);
      if (i < a.G) m_e[k] = __ldg(a.expert_ids + i);
    }
  }
  // NVFP4: thread e < n_tab (<= kTqTabExperts = kTqThreads) owns expert e's table
  const float m_sf = (FMT == kNVFP4 && static_cast<int>(threadIdx.x) < q.n_tab) ? __ldg(a.sf + threadIdx.x) : 0.0f;

  // (1) scan: file the destination rows of this block's tokens.  Every
  // block reads every entry, so the per-entry test is a 32-bit subtract and
  // compare (source rows and in_rows are below 2^31), four staged vectors
  // per thread at a time, with the rare hits filed afterwards; block 0 also
  // notes source rows outside x, which are checked (and reported when their
  // group is kept) once the metadata is in shared memory.
  int64_t done = 0;                              // staged chunks filed
  int64_t issued = n_chunks < 2 ? n_chunks : 2;  // staged chunks copied
  const bool reporter = blockIdx.x == 0;
  if (gather) {
    const uint32_t t_lo32 = static_cast<uint32_t>(t_lo), nt32 = static_cast<uint32_t>(nt);
    // (in_rows >= 2^31: every non-negative int32 source row is inside x)
    const uint32_t in_rows32 = static_cast<uint32_t>(a.in_rows < 0x80000000LL ? a.in_rows : 0x80000000LL);
    auto file = [&](int64_t d, int32_t src) {
      const uint32_t k = static_cast<uint32_t>(src) - t_lo32;
      if (k < nt32) {
        const uint32_t slot = atomicAdd(&cnt[k], 1u);
        if (slot < kTqBucket) bkt[k * kTqBucket + slot] = static_cast<uint32_t>(d);
      } else if (reporter && static_cast<uint32_t>(src) >= in_rows32) {
        const uint32_t j = atomicAdd(&sh.n_bad, 1u);
        if (j < kTqBadList) {
          sh.bad_d[j] = static_cast<uint32_t>(d);
          sh.bad_src[j] = src;
        }
      }
    };
    if (threadIdx.x < 8) {
      const int64_t d = threadIdx.x < 4 ? threadIdx.x : head + 4 * nvec + (threadIdx.x - 4);
      if ((threadIdx.x < 4 ? d < head : true) && d < rows) file(d, __ldg(a.row_indices + d));
    }
    // staged body vectors holding rows below `rows` (the scalar tail holds the rest)
    const int64_t rows_vec = min(nvec, rows > head ? (rows - head + 3) >> 2 : int64_t(0));
#pragma unroll 1
    for (int64_t c = 0; c < n_chunks && c * cvec < rows_vec; ++c) {
      const int b = static_cast<int>(c & 1);
      if (!mbar_wait_bounded(&sh.stage_bar[b], static_cast<uint32_t>((c >> 1) & 1))) {
        record_error(kErrTimeout);
        sh.failed = 1u;
      }
      if (!__syncthreads_or(sh.failed != 0u)) {
        const int4* buf = stage + b * cvec;
        const int64_t v0 = c * cvec;
        const int nv = static_cast<int>(min(cvec, rows_vec - v0));  // vectors of this chunk with rows to file
        const int nfull = static_cast<int>(max(int64_t(0), min(static_cast<int64_t>(nv), (rows - head) / 4 - v0)));  // all 4 below rows
        const uint32_t d0 = static_cast<uint32_t>(head + 4 * v0);
#pragma unroll 1
        for (int v = threadIdx.x; v < nfull; v += kTqScanVec * kTqThreads) {
          int4 qv[kTqScanVec];
          bool in[kTqScanVec];
#pragma unroll
          for (int j = 0; j < kTqScanVec; ++j) {
            in[j] = v + j * kTqThreads < nfull;
            qv[j] = in[j] ? buf[v + j * kTqThreads] : make_int4(0, 0, 0, 0);
          }
          uint32_t hit = 0u;
#pragma unroll
          for (int j = 0; j < kTqScanVec; ++j) {
            const uint32_t s4[4] = {static_cast<uint32_t>(qv[j].x), static_cast<uint32_t>(qv[j].y),
                                    static_cast<uint32_t>(qv[j].z), static_cast<uint32_t>(qv[j].w)};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const bool h = s4[e] - t_lo32 < nt32 || (reporter && s4[e] >= in_rows32);
              hit |= (in[j] && h) ? (1u << (4 * j + e)) : 0u;
            }
          }
          if (hit != 0u) {
#pragma unroll
            for (int j = 0; j < kTqScanVec; ++j) {
              const uint32_t h = (hit >> (4 * j)) & 15u;
              if (h != 0u) {
                const uint32_t d = d0 + 4u * static_cast<uint32_t>(v + j * kTqThreads);
                if (h & 1u) file(d, qv[j].x);
                if (h & 2u) file(d + 1, qv[j].y);
                if (h & 4u) file(d + 2, qv[j].z);
                if (h & 8u) file(d + 3, qv[j].w);
              }
            }
          }
        }
        for (int v = nfull + static_cast<int>(threadIdx.x); v < nv; v += kTqThreads) {
          const int4 qv = buf[v];
          const int64_t d = head + 4 * (v0 + v);
          if (d < rows) file(d, qv.x);
          if (d + 1 < rows) file(d + 1, qv.y);
          if (d + 2 < rows) file(d + 2, qv.z);
          if (d + 3 < rows) file(d + 3, qv.w);
        }
      }
      __syncthreads();  // buffer b is free again
      if (c + 2 < n_chunks) {
        if (threadIdx.x == 0) {
          mbar_arrive_expect_tx(&sh.stage_bar[b], chunk_bytes(c + 2));
          bulk_load(stage + b * cvec, body + (c + 2) * cvec, chunk_bytes(c + 2), &sh.stage_bar[b]);
        }
        issued = c + 3;
      }
      done = c + 1;
    }
  }
  // chunks [done, issued) were copied but not consumed (rows past
  // min(row_offsets[G], total_rows), or an expired wait): their copies land
  // before the block may exit
  if (threadIdx.x == 0) {
    for (int64_t c = done; c < issued; ++c)
      if (!mbar_wait_bounded(&sh.stage_bar[c & 1], static_cast<uint32_t>((c >> 1) & 1))) record_error(kErrTimeout);
  }
  // the metadata and the NVFP4 factor tables into shared memory
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    const int i = static_cast<int>(threadIdx.x) + k * kTqThreads;
    if (i <= a.G) {
      sh.ro[i] = m_ro[k];
      sh.so[i] = m_so[k];
      if (i < a.G) sh.e[i] = m_e[k];
    }
  }
  if constexpr (FMT == kNVFP4) {
    if (static_cast<int>(threadIdx.x) < q.n_tab) {
      float* t = tabs + threadIdx.x * 16;
      t[0] = 0.0f;
#pragma unroll
      for (int m = 1; m < 16; ++m) t[m] = __fdiv_rn(m_sf, static_cast<float>(m));
    }
  }
  __syncthreads();
  if (sh.failed != 0u) return;  // block-uniform; reported as BSQ_ERR_TIMEOUT
  if (a.scale_ws != nullptr) {  // the staged rows of each band, for grouped_scale_ws_kernel
    const int64_t n_bands = a.total_scale_rows / 128;
    for (int64_t b = static_cast<int64_t>(blockIdx.x) * kTqThreads + threadIdx.x; b < n_bands;
         b += static_cast<int64_t>(gridDim.x) * kTqThreads)
      ws_band_rows(a)[b] = band_rows_written(a, sh.ro, sh.so, sh.e, b);
  }
  if (gather && reporter) {
    // source rows outside x: reported when their row belongs to a kept group
    const uint32_t nb = sh.n_bad;
    if (nb <= static_cast<uint32_t>(kTqBadList)) {
      for (uint32_t j = threadIdx.x; j < nb; j += kTqThreads) {
        int64_t sr;
        int e;
        tq_check(a, sh, sh.bad_d[j], sh.bad_src[j], sr, e);
      }
    } else {
      for (int64_t d = threadIdx.x; d < rows; d += kTqThreads) {  // more than the list holds: look again
        const int32_t src = __ldg(a.row_indices + d);
        if (src < 0 || src >= a.in_rows) {
          int64_t sr;
          int e;
          tq_check(a, sh, d, src, sr, e);
        }
      }
    }
  }

  const float* div6 = sh.div6_tab;
  if (q.units) {
    // (2) each warp describes tokens w, w + 32 into the freed staging area ...
    TqDesc* tdesc = reinterpret_cast<TqDesc*>(stage);                   // nt x kTqBucket
    int* tnv = reinterpret_cast<int*>(tdesc + static_cast<int64_t>(nt) * kTqBucket);  // nt
#pragma unroll 1
    for (int k = warp; k < nt; k += kTqWarps) {
      const int64_t t = t_lo + k;
      int n;
      int64_t d = -1;
      if (gather) {
        n = static_cast<int>(cnt[k]);
        if (n > kTqBucket) {  // warp-uniform: left to the re-scan
          if (lane == 0) {
            sh.heavy = 1u;
            tnv[k] = 0;
          }
          continue;
        }
        if (lane < n) d = bkt[k * kTqBucket + lane];
      } else {
        n = t < rows ? 1 : 0;
        d = t;
      }
      const int nv = tq_describe<FMT>(a, sh, tdesc + k * kTqBucket, lane < n, d, t, q.n_tab);
      if (lane == 0) tnv[k] = nv;
    }
    __syncthreads();
    // (3) ... then claims (token, step) units: the warps of a block share
    // its tokens' work evenly however few tokens it has.  Unit u is step
    // u % steps of token u / steps; warp w starts on unit w (prefetched),
    // and the first step of the next unit is loaded during the last step
    // of the current one.
    const int n_units = nt * steps;
    int u = warp;
#pragma unroll 1
    while (u < n_units) {
      int nxt = 0;
      if (lane == 0) nxt = static_cast<int>(atomicAdd(&sh.next_unit, 1u));
      nxt = __shfl_sync(0xFFFFFFFFu, nxt, 0);
      const int k = u / steps, c = u - k * steps;
      const int nv = tnv[k];
      const uint16_t* next_row = nullptr;
      int next_jb = 0;
      if (nxt < n_units) {
        const int nk = nxt / steps;
        if (t_lo + nk < a.in_rows) {  // (without row_indices, tokens past x have no rows)
          next_row = a.in + (t_lo + nk) * a.ld_in;
          next_jb = (nxt - nk * steps) * 32;
        }
      }
      if (nv == 0) {  // warp-uniform: no rows to write; load the next unit's first step
        tq_zero(pre);
        if (next_row != nullptr && next_jb + lane < a.K / Fmt<FMT>::SF)
          tq_load(pre, next_row + Fmt<FMT>::SF * (next_jb + lane), a.in_vec32 != 0);
      } else {
        const int jb = c * 32;
        const int je = min(jb + 32, a.kt_atoms * 4);
        tq_row<FMT>(a, a.in + (t_lo + k) * a.ld_in, pre, jb, je, tdesc + k * kTqBucket, nv, div6, tabs, next_row,
                    next_jb);
      }
      __syncwarp();
      u = nxt;
    }
  }
  // (2) + (3) without units: warp w takes tokens w, w + 32, ...
  TqDesc* desc = sh.desc[warp];
#pragma unroll 1
  for (int k = q.units ? nt : warp; k < nt; k += kTqWarps) {
    const int64_t t = t_lo + k;
    int n;
    int64_t d = -1;
    if (gather) {
      n = static_cast<int>(cnt[k]);
      if (n > kTqBucket) {  // warp-uniform: left to the re-scan
        if (lane == 0) sh.heavy = 1u;
        continue;
      }
      if (lane < n) d = bkt[k * kTqBucket + lane];
    } else {
      n = t < rows ? 1 : 0;
      d = t;
    }
    const int nv = tq_describe<FMT>(a, sh, desc, lane < n, d, t, q.n_tab);
    if (nv == 0) continue;  // warp-uniform
    if (k != warp) {
      tq_zero(pre);
      if (lane < a.K / Fmt<FMT>::SF) tq_load(pre, a.in + t * a.ld_in + Fmt<FMT>::SF * lane, a.in_vec32 != 0);
    }
    tq_row<FMT>(a, a.in + t * a.ld_in, pre, 0, a.kt_atoms * 4, desc, nv, div6, tabs);
    __syncwarp();
  }

  // (4) tokens with more destination rows than a bucket holds: re-scan and
  // quantize each of their rows on its own (warp-collective).
  __syncthreads();
  if (!gather || sh.heavy == 0u) return;  // block-uniform
#pragma unroll 1
  for (int64_t d0 = 0; d0 < rows; d0 += kTqThreads) {
    const int64_t dm = d0 + threadIdx.x;
    int32_t src = 0;
    bool hit = false;
    if (dm < rows) {
      src = __ldg(a.row_indices + dm);
      const int64_t k = src - t_lo;
      hit = k >= 0 && k < nt && cnt[k] > static_cast<uint32_t>(kTqBucket);
    }
    uint32_t m = __ballot_sync(0xFFFFFFFFu, hit);
    while (m != 0u) {
      const int l = __ffs(m) - 1;
      m &= m - 1u;
      const int64_t dd = __shfl_sync(0xFFFFFFFFu, dm, l);
      const int32_t ss = __shfl_sync(0xFFFFFFFFu, src, l);
      const int nv = tq_describe<FMT>(a, sh, desc, lane == 0, dd, ss, q.n_tab);
      if (nv == 0) continue;  // warp-uniform
      TqChunk<FMT> c;
      tq_zero(c);
      if (lane < a.K / Fmt<FMT>::SF)
        tq_load(c, a.in + static_cast<int64_t>(ss) * a.ld_in + Fmt<FMT>::SF * lane, a.in_vec32 != 0);
      tq_row<FMT>(a, a.in + static_cast<int64_t>(ss) * a.ld_in, c, 0, a.kt_atoms * 4, desc, nv, div6, tabs);
      __syncwarp();
    }
  }
}

// ------------------------------------------------- grouped_scale_ws_kernel --

// Block (b, c): 5D band b (scale rows 128 b ..), atoms kIlvAtoms c ..  The
// token kernel stored n = band_rows_written(b) in the workspace after the
// staged rows; those n rows (row-major, 4 Kt bytes each) go to their 5D
// positions: a 16-byte store per chunk whose four rows were all written,
// 4-byte stores otherwise; the other rows' bytes are not touched.  VEC:
// bytes per staging load (16 when the rows allow it, else 4).
template <int VEC>
__global__ void __launch_bounds__(kIlvThreads) grouped_scale_ws_kernel(const GroupedArgs a) {
  __shared__ __align__(16) uint8_t tile[128 * kIlvPitch];
  const int64_t s0 = static_cast<int64_t>(blockIdx.x) * 128;
  pdl_wait();
  const int n = __ldcg(ws_band_rows(a) + blockIdx.x);  // written by the token kernel
  if (n <= 0 || n > 128) return;  // block-uniform

  const int kt = a.kt_atoms;
  const int a0 = blockIdx.y * kIlvAtoms;
  const int na = min(kIlvAtoms, kt - a0);
  const int64_t S4 = static_cast<int64_t>(kt) * 4;
  const uint8_t* src = a.scale_ws + s0 * S4 + 4 * a0;  // staged row r, this run's first byte
  // rows r < n, bytes 0 .. 4 na - 1 of the run, into the padded tile
  constexpr int kPerRow = kIlvCols / VEC;
  for (int idx = threadIdx.x; idx < 128 * kPerRow; idx += kIlvThreads) {
    const int r = idx / kPerRow, w = idx % kPerRow;
    if (r < n && VEC * w < 4 * na) {
      if constexpr (VEC == 16) {
        const uint4 x = __ldg(reinterpret_cast<const uint4*>(src + r * S4 + VEC * w));
        uint32_t* t = reinterpret_cast<uint32_t*>(tile + r * kIlvPitch + VEC * w);
        t[0] = x.x; t[1] = x.y; t[2] = x.z; t[3] = x.w;
      } else {
        *reinterpret_cast<uint32_t*>(tile + r * kIlvPitch + VEC * w) =
            __ldg(reinterpret_cast<const uint32_t*>(src + r * S4 + VEC * w));
      }
    }
  }
  __syncthreads();
  uint8_t* dst = a.scales + (static_cast<int64_t>(blockIdx.x) * kt + a0) * 512;
  for (int idx = threadIdx.x; idx < na * 32; idx += kIlvThreads) {
    const int at = idx >> 5, r32 = idx & 31;
    if (r32 >= n) continue;
    const uint8_t* t = tile + r32 * kIlvPitch + at * 4;
    uint8_t* chunk = dst + at * 512 + r32 * 16;
    if (r32 + 96 < n) {
      st_global_v4(chunk, *reinterpret_cast<const uint32_t*>(t), *reinterpret_cast<const uint32_t*>(t + 32 * kIlvPitch),
                   *reinterpret_cast<const uint32_t*>(t + 64 * kIlvPitch),
                   *reinterpret_cast<const uint32_t*>(t + 96 * kIlvPitch));
    } else {
      for (int sb = 0; sb < 4 && r32 + 32 * sb < n; ++sb)
        *reinterpret_cast<uint32_t*>(chunk + 4 * sb) = *reinterpret_cast<const uint32_t*>(t + 32 * sb * kIlvPitch);
    }
  }
}

}  // namespace bsq
