// NVFP4 tensor scales on the GPU: tensor_sf = fl32(448 * 6 / amax), amax the
// exact max |x| of a BF16 tensor (or, per expert, over the expert's gathered
// rows), 1.0 for an all-zero tensor.  These are the FP32 tensor_sf / per-expert
// sf_tensor inputs of the NVFP4 quantize kernels, computed where the data is.
//
// Dense: warps stride over rows, lanes over 16-byte chunks (four loads in
// flight per lane), max.xorsign.abs BF16 pairs, warp and block reductions;
// every block folds its maximum into the workspace with one atomic max, and
// the last block to finish (fenced atomic counter) writes {amax, tensor_sf}.
// Grouped: one warp per destination row, its group by a binary search over
// row_offsets, an atomic max per expert (non-negative FP32
// maxima order like their bit patterns), and the last block writes sf_tensor;
// when a gather reuses source rows over few tokens, a token-major variant
// reads each source row once and scans row_indices instead.  All leave their
// workspace zeroed for the next launch.
#pragma once

#include "cluster.cuh"
#include "device_common.cuh"

namespace bsq {

constexpr int kAmaxThreads = 256;
constexpr int kAmaxWarps = kAmaxThreads / 32;
constexpr int kAmaxMaxBlocks = 1024;

// Dense workspace: a completion counter and the running maximum (FP32 bits;
// each block folds its maximum in with one atomic max).  The caller zeroes
// it once; the last block of every launch sets both back to zero, so
// consecutive launches need no memset in between.  A stale counter c > 0 (a
// workspace never zeroed) hands some block a ticket >= gridDim.x, which
// records BSQ_ERR_VALUE; with c >= gridDim.x no block is last and nothing is
// written, with a smaller c the block holding ticket gridDim.x - 1 may
// finish before the remaining blocks have folded in their maxima (that
// launch's outputs are reported as invalid).  A stale maximum under a zero
// counter is not detected (as for the per-expert maxima of the grouped
// workspace): the workspace must be zeroed whole.  The rest of the
// workspace (its size is part of the interface) is unused.
struct AmaxWorkspace {
  unsigned int counter;
  unsigned int amax_bits;
  unsigned int pad[2];
  unsigned int unused[kAmaxMaxBlocks];
};

__device__ __forceinline__ float tensor_sf_of(float amax) {
  return amax > 0.0f ? __fdiv_rn(2688.0f, amax) : 1.0f;
}

// max |x| over one row of K BF16 elements (K % 8 == 0), as two BF16 halves.
// The loads keep their lines in L2 (evict_last) for the quantize pass that
// follows over the same tensor.
__device__ __forceinline__ uint32_t row_absmax(const uint16_t* row, int K, int lane, uint64_t pol) {
  uint32_t acc = 0;
  const int chunks = K >> 3;
  int c = lane;
  for (; c + 96 < chunks; c += 128) {
    const uint4 v0 = ld_global_nc_v4_policy(row + 8 * c, pol), v1 = ld_global_nc_v4_policy(row + 8 * (c + 32), pol);
    const uint4 v2 = ld_global_nc_v4_policy(row + 8 * (c + 64), pol), v3 = ld_global_nc_v4_policy(row + 8 * (c + 96), pol);
    acc = absmax2(acc, v0.x); acc = absmax2(acc, v0.y); acc = absmax2(acc, v0.z); acc = absmax2(acc, v0.w);
    acc = absmax2(acc, v1.x); acc = absmax2(acc, v1.y); acc = absmax2(acc, v1.z); acc = absmax2(acc, v1.w);
    acc = absmax2(acc, v2.x); acc = absmax2(acc, v2.y); acc = absmax2(acc, v2.z); acc = absmax2(acc, v2.w);
    acc = absmax2(acc, v3.x); acc = absmax2(acc, v3.y); acc = absmax2(acc, v3.z); acc = absmax2(acc, v3.w);
  }
  for (; c < chunks; c += 32) {
    const uint4 v = ld_global_nc_v4_policy(row + 8 * c, pol);
    acc = absmax2(acc, v.x); acc = absmax2(acc, v.y); acc = absmax2(acc, v.z); acc = absmax2(acc, v.w);
  }
  return acc;
}

// Warp max of non-negative FP32 values, on their bit patterns.
__device__ __forceinline__ uint32_t warp_max_bits(uint32_t b) {
#pragma unroll
  for (int x = 16; x > 0; x >>= 1) b = max(b, __shfl_xor_sync(0xFFFFFFFFu, b, x));
  return b;
}

__global__ void __launch_bounds__(kAmaxThreads)
    tensor_amax_kernel(const uint16_t* __restrict__ in, int64_t M, int K, int64_t ld,
                       AmaxWorkspace* ws, float* out) {
  __shared__ uint32_t warp_max[kAmaxWarps];
  __shared__ bool last;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  pdl_wait();
  uint32_t acc = 0;
  const uint64_t pol = l2_policy_evict_last();
  for (int64_t r = static_cast<int64_t>(blockIdx.x) * kAmaxWarps + warp; r < M;
       r += static_cast<int64_t>(gridDim.x) * kAmaxWarps)
    acc = absmax2(acc, row_absmax(in + r * ld, K, lane, pol));
  pdl_trigger();  // this block's reads are done: the next kernel may launch
  const uint32_t wm = warp_max_bits(__float_as_uint(absmax_final(acc)));
  if (lane == 0) warp_max[warp] = wm;
  __syncthreads();
  if (threadIdx.x == 0) {
    uint32_t bm = 0;
    for (int w = 0; w < kAmaxWarps; ++w) bm = max(bm, warp_max[w]);
    if (bm != 0u) atomicMax(&ws->amax_bits, bm);  // non-negative FP32 maxima order like their bits
    __threadfence();
    const unsigned int ticket = atomicAdd(&ws->counter, 1u);
    if (ticket >= gridDim.x) record_error(kErrValue);
    last = ticket == gridDim.x - 1;
  }
  __syncthreads();
  if (!last) return;
  // last block: every block's maximum is in
  __threadfence();
  if (threadIdx.x == 0) {
    const uint32_t m = __ldcg(&ws->amax_bits);
    ws->amax_bits = 0u;
    const float amax = __uint_as_float(m);
    out[0] = amax;
    out[1] = tensor_sf_of(amax);
    ws->counter = 0;
  }
}

struct GroupedAmaxArgs {
  const uint16_t* in;
  int64_t ld_in, in_rows;
  int K;
  const uint32_t* row_offsets;
  const int32_t* expert_ids;
  const int32_t* row_indices;  // may be null
  int G;
  int64_t total_rows;
  int num_experts;
  unsigned int* amax_bits;     // workspace: num_experts maxima (zero at launch, zeroed again)
  unsigned int* counter;       // workspace: completion counter (zero at launch, zeroed again)
  float* sf;                   // out: num_experts tensor scales
};

__global__ void __launch_bounds__(kAmaxThreads) grouped_amax_kernel(const GroupedAmaxArgs a) {
  __shared__ bool last;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  pdl_wait();
  const int64_t ro_end = a.G > 0 ? static_cast<int64_t>(__ldg(a.row_offsets + a.G)) : 0;  // no groups: no rows
  const int64_t rows = ro_end < a.total_rows ? ro_end : a.total_rows;
  const uint64_t pol = l2_policy_evict_last();
  for (int64_t d = static_cast<int64_t>(blockIdx.x) * kAmaxWarps + warp; d < rows;
       d += static_cast<int64_t>(gridDim.x) * kAmaxWarps) {
    int e = -1;
    int64_t src = -1;
    if (lane == 0) {
      int lo = 0, hi = a.G - 1;  // g = max{g : ro[g] <= d}
      while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if (static_cast<int64_t>(__ldg(a.row_offsets + mid + 1)) <= d) lo = mid + 1;
        else hi = mid;
      }
      e = __ldg(a.expert_ids + lo);
      src = a.row_indices ? static_cast<int64_t>(__ldg(a.row_indices + d)) : d;
      if (d < static_cast<int64_t>(__ldg(a.row_offsets + lo)) || e >= a.num_experts ||
          (e >= 0 && (src < 0 || src >= a.in_rows))) {
        record_error(kErrValue);
        e = -1;
      }
    }
    e = __shfl_sync(0xFFFFFFFFu, e, 0);
    src = __shfl_sync(0xFFFFFFFFu, src, 0);
    if (e < 0) continue;  // warp-uniform
    const uint32_t m =
        warp_max_bits(__float_as_uint(absmax_final(row_absmax(a.in + src * a.ld_in, a.K, lane, pol))));
    if (lane == 0 && m != 0u) atomicMax(a.amax_bits + e, m);
  }
  pdl_trigger();  // this block's reads are done: the next kernel may launch
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    const unsigned int ticket = atomicAdd(a.counter, 1u);
    if (ticket >= gridDim.x) record_error(kErrValue);
    last = ticket == gridDim.x - 1;
  }
  __syncthreads();
  if (!last) return;
  __threadfence();
  for (int e = threadIdx.x; e < a.num_experts; e += kAmaxThreads) {
    a.sf[e] = tensor_sf_of(__uint_as_float(__ldcg(a.amax_bits + e)));
    a.amax_bits[e] = 0u;  // ready for the next launch
  }
  if (threadIdx.x == 0) *a.counter = 0u;
}

// Per-expert maxima, token-major (a row_indices gather that reuses source
// rows, e.g. top-k routing).  A cluster of kAtCluster blocks owns
// kAtCluster * kAtTokens consecutive source rows: each block reduces the max
// |x| of its kAtTokens rows once (one warp per row) into shared memory; then
// each block of the cluster scans its contiguous share of row_indices (the
// entries to visit compacted per warp and shared out over its lanes), and
// each destination row whose source row the cluster owns folds that row's
// maximum (read from the owning block's shared memory) into a per-group
// maximum in shared memory; the block then issues one atomic max per group
// it touched.  The same maxima as grouped_amax_kernel (max is exact and
// order-free), with each source row read once instead of once per
// destination row, and row_indices read once per cluster, in 16-byte
// vectors.  Metadata errors of a destination row are reported by the cluster
// owning its source row (a source row outside x: by the first cluster), as
// in grouped_amax_kernel.
constexpr int kAtThreads = 512;
constexpr int kAtTokens = kAtThreads / 32;
constexpr int kAtCluster = 8;
constexpr int kAtClusterTokens = kAtCluster * kAtTokens;
constexpr int kAtMaxGroups = 1024;

constexpr int kAtScanU = 2;  // 16-byte row_indices loads in flight per thread
struct AtShared {
  uint32_t ro[kAtMaxGroups + 1];
  int32_t e[kAtMaxGroups];
  uint32_t gmax[kAtMaxGroups];  // per-group maximum found by this block's scan
  uint32_t rowmax[kAtTokens];
  // per warp, one scan iteration's entries to visit (destination offset, source row)
  uint32_t hit_d[kAtThreads / 32][32 * 4 * kAtScanU];
  int32_t hit_s[kAtThreads / 32][32 * 4 * kAtScanU];
};

// max |x| over one row (K % 8 == 0): eight 16-byte loads in flight per lane,
// the last round predicated.
__device__ __forceinline__ uint32_t row_absmax_wide(const uint16_t* row, int K, int lane, uint64_t pol) {
  uint32_t acc = 0;
  const int chunks = K >> 3;
  for (int c = lane; c < chunks; c += 256) {
    uint4 v[8];
#pragma unroll
    for (int k = 0; k < 8; ++k)
      v[k] = c + 32 * k < chunks ? ld_global_nc_v4_policy(row + 8 * (c + 32 * k), pol) : make_uint4(0, 0, 0, 0);
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      acc = absmax2(acc, v[k].x); acc = absmax2(acc, v[k].y);
      acc = absmax2(acc, v[k].z); acc = absmax2(acc, v[k].w);
    }
  }
  return acc;
}

// rowmax[k] of block `rank` of this cluster (distributed shared memory).
__device__ __forceinline__ uint32_t cluster_rowmax(const AtShared& sh, int rank, int k) {
  return cluster_ld_u32(cluster_map(&sh.rowmax[k], rank));
}

// Destination row d gathers source row src; fold it in if this cluster owns src.
__device__ __forceinline__ void at_visit(const GroupedAmaxArgs& a, AtShared& sh, int64_t c0,
                                         bool first_cluster, int64_t d, int64_t src) {
  const bool bad_src = src < 0 || src >= a.in_rows;
  const int64_t k = src - c0;
  if (bad_src ? !first_cluster : (k < 0 || k >= kAtClusterTokens)) return;
  int lo = 0, hi = a.G - 1;  // g = max{g : ro[g] <= d}
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (static_cast<int64_t>(sh.ro[mid + 1]) <= d) lo = mid + 1;
    else hi = mid;
  }
  const int e = sh.e[lo];
  if (d < static_cast<int64_t>(sh.ro[lo]) || e >= a.num_experts || (e >= 0 && bad_src)) {
    record_error(kErrValue);
    return;
  }
  if (e < 0 || bad_src) return;
  const uint32_t m = cluster_rowmax(sh, static_cast<int>(k / kAtTokens), static_cast<int>(k % kAtTokens));
  if (m != 0u) atomicMax(&sh.gmax[lo], m);
}

// Grid: a multiple of kAtCluster blocks covering in_rows source rows.  The
// first batch of row_indices loads is issued before the row maxima are
// reduced, so that the scan's L2 latency hides under the HBM reads.
__global__ void __cluster_dims__(kAtCluster, 1, 1) __launch_bounds__(kAtThreads, 2)
    grouped_amax_token_kernel(const GroupedAmaxArgs a) {
  __shared__ AtShared sh;
  __shared__ bool last;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int rank = static_cast<int>(blockIdx.x % kAtCluster);
  const int64_t c0 = static_cast<int64_t>(blockIdx.x / kAtCluster) * kAtClusterTokens;
  const bool first_cluster = blockIdx.x < kAtCluster;
  pdl_wait();
  const int64_t ro_end = a.G > 0 ? static_cast<int64_t>(__ldg(a.row_offsets + a.G)) : 0;
  const int64_t rows = ro_end < a.total_rows ? ro_end : a.total_rows;
  // row_indices: a scalar head up to a 16-byte boundary and a scalar tail
  // (first block of the cluster), and a 16-byte body in kAtCluster contiguous
  // shares, one per block
  const int64_t mis = static_cast<int64_t>(((16 - (reinterpret_cast<uintptr_t>(a.row_indices) & 15)) & 15) >> 2);
  const int64_t head = mis < rows ? mis : rows;
  const int64_t nvec = (rows - head) >> 2;
  const int4* body = reinterpret_cast<const int4*>(a.row_indices + head);
  const int64_t share = (nvec + kAtCluster - 1) / kAtCluster;
  const int64_t vb = share * rank;
  const int64_t ve = vb + share < nvec ? vb + share : nvec;
  constexpr int U = kAtScanU;
  int4 q[U];
#pragma unroll
  for (int u = 0; u < U; ++u) {
    const int64_t v = vb + threadIdx.x + u * kAtThreads;
    q[u] = v < ve ? __ldg(body + v) : make_int4(0, 0, 0, 0);
  }
  for (int i = threadIdx.x; i <= a.G; i += kAtThreads) {
    sh.ro[i] = __ldg(a.row_offsets + i);
    if (i < a.G) {
      sh.e[i] = __ldg(a.expert_ids + i);
      sh.gmax[i] = 0u;
    }
  }
  {
    const int64_t t = static_cast<int64_t>(blockIdx.x) * kAtTokens + warp;
    uint32_t m = 0;
    if (t < a.in_rows)
      m = warp_max_bits(
          __float_as_uint(absmax_final(row_absmax_wide(a.in + t * a.ld_in, a.K, lane, l2_policy_evict_last()))));
    if (lane == 0) sh.rowmax[warp] = m;
  }
  __syncthreads();
  cluster_sync_all();  // every block's rowmax is visible to the cluster
  if (rank == 0 && threadIdx.x < head) at_visit(a, sh, c0, first_cluster, threadIdx.x, __ldg(a.row_indices + threadIdx.x));
  for (int64_t v0 = vb; v0 < ve; v0 += static_cast<int64_t>(kAtThreads) * U) {
    if (v0 > vb) {
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int64_t v = v0 + threadIdx.x + u * kAtThreads;
        q[u] = v < ve ? __ldg(body + v) : make_int4(0, 0, 0, 0);
      }
    }
    // The entries at_visit does not skip at once are compacted per warp and
    // shared out over its lanes: row_indices lists each group's rows in
    // token order, so a cluster's hits come in runs that would otherwise
    // fall to a few lanes, each paying a search and a remote load per hit.
    uint32_t hm = 0u;
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t v = v0 + threadIdx.x + u * kAtThreads;
      if (v >= ve) continue;
      const int32_t s4[4] = {q[u].x, q[u].y, q[u].z, q[u].w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const bool bad = s4[e] < 0 || s4[e] >= a.in_rows;
        const int64_t k = static_cast<int64_t>(s4[e]) - c0;
        if (bad ? first_cluster : (k >= 0 && k < kAtClusterTokens)) hm |= 1u << (4 * u + e);
      }
    }
    const int nh = __popc(hm);
    int incl = nh;  // inclusive prefix count over the warp's lanes
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int t = __shfl_up_sync(0xFFFFFFFFu, incl, o);
      if (lane >= o) incl += t;
    }
    const int total = __shfl_sync(0xFFFFFFFFu, incl, 31);
    if (total > 0) {  // warp-uniform
      int pos = incl - nh;
#pragma unroll
      for (int b = 0; b < 4 * U; ++b) {
        if ((hm >> b) & 1u) {
          const int u = b >> 2, e = b & 3;
          sh.hit_d[warp][pos] = static_cast<uint32_t>(4 * (threadIdx.x + u * kAtThreads) + e);  // d - (head + 4 v0)
          sh.hit_s[warp][pos] = e == 0 ? q[u].x : e == 1 ? q[u].y : e == 2 ? q[u].z : q[u].w;
          ++pos;
        }
      }
      __syncwarp();
      for (int i = lane; i < total; i += 32)
        at_visit(a, sh, c0, first_cluster, head + 4 * v0 + sh.hit_d[warp][i], sh.hit_s[warp][i]);
      __syncwarp();
    }
  }
  if (rank == 0)
    for (int64_t d = head + 4 * nvec + threadIdx.x; d < rows; d += kAtThreads)
      at_visit(a, sh, c0, first_cluster, d, __ldg(a.row_indices + d));
  __syncthreads();
  for (int i = threadIdx.x; i < a.G; i += kAtThreads)
    if (sh.gmax[i] != 0u) atomicMax(a.amax_bits + sh.e[i], sh.gmax[i]);
  pdl_trigger();  // this block's reads are done: the next kernel may launch
  __syncthreads();
  cluster_sync_all();  // no block leaves while another may read its rowmax
  if (threadIdx.x == 0) {
    __threadfence();
    const unsigned int ticket = atomicAdd(a.counter, 1u);
    if (ticket >= gridDim.x) record_error(kErrValue);
    last = ticket == gridDim.x - 1;
  }
  __syncthreads();
  if (!last) return;
  __threadfence();
  for (int e = threadIdx.x; e < a.num_experts; e += kAtThreads) {
    a.sf[e] = tensor_sf_of(__uint_as_float(__ldcg(a.amax_bits + e)));
    a.amax_bits[e] = 0u;  // ready for the next launch
  }
  if (threadIdx.x == 0) *a.counter = 0u;
}

}  // namespace bsq
