// Dense block-scaled quantization: BF16 (M, K) -> packed NVFP4 / MXFP4 /
// MXFP8 elements + scales in the 5D TCGEN layout.
//
// Design (sm_103a): a persistent kernel, one producer warp + eight consumer
// warps per CTA.  The work unit is a tile of 128 rows x 128 columns (one 5D
// scale-tile row band, 2 atoms for NVFP4 / 1 atom for MX).  The producer's
// elected lane streams tiles into a STAGES-deep shared-memory ring with 2D TMA
// loads (two 128-row x 64-column boxes per tile, 128-byte swizzle,
// out-of-range rows/columns zero-filled), completing on a "full" mbarrier.
// Consumer warps 0-3 take box 0 and warps 4-7 box 1 of every tile; each
// consumer lane owns one row of its box: it reads its row conflict-free
// (the swizzle spreads a quarter-warp over all banks), reduces each block's
// amax in registers, computes the block scale, encodes the elements with the
// hardware cvt instructions and stores its packed bytes as whole 32-byte
// sectors.  The lane -> row mapping is chosen so that the 32 lanes of a warp
// hold 128 contiguous bytes of each 512-byte scale atom, written by one
// coalesced 4-byte-per-lane store.  Consumer warps release a stage with one
// arrive each on its "empty" mbarrier.  Zero-filled padding yields zero blocks,
// whose scale bytes are 0x00, so the padding of the 5D buffer is written
// without extra work.
#pragma once

#include "box_quant.cuh"
#include "device_common.cuh"

namespace bsq {

constexpr int kDenseTileRows = 128;
constexpr int kDenseTileCols = 128;
constexpr int kDenseBoxCols = 64;                               // 128 bytes of BF16
constexpr int kDenseBoxBytes = kDenseTileRows * kDenseBoxCols * 2;  // 16 KB
constexpr int kDenseStageBytes = 2 * kDenseBoxBytes;               // 32 KB
constexpr int kDenseConsumerWarps = 8;
constexpr int kDenseThreads = (kDenseConsumerWarps + 1) * 32;

template <int STAGES>
constexpr int dense_smem_bytes() {
  // stages + alignment slack + mbarriers + NVFP4 element-scale and amax/6 tables
  return STAGES * kDenseStageBytes + 1024 + 2 * STAGES * 8 + (256 + 128) * 4;
}

struct DenseArgs {
  uint8_t* out;        // packed elements, row stride = packed row bytes
  uint8_t* scales;     // 5D scales
  int64_t out_ld;      // packed row bytes
  int M, K;
  int tiles_k;         // ceil(K / 128)
  int num_tiles;       // ceil(M / 128) * tiles_k
  int kt_atoms;        // 5D atoms per 128-row band: ceil(K / SF / 4)
  int vec32;           // packed rows allow 32-byte stores
  float tsf;
  const float* tsf_dev;  // NVFP4: tensor_sf read from device memory (or null: use tsf)
};

template <int FMT, int STAGES>
__global__ void __launch_bounds__(kDenseThreads)
    dense_quant_tma_kernel(const __grid_constant__ CUtensorMap tmap, const DenseArgs a) {
  extern __shared__ uint8_t smem_raw[];
  // 1024-byte alignment (128-byte swizzle atoms) by an offset from the shared
  // array itself, so that every access below stays a shared-space load
  const uint32_t base = static_cast<uint32_t>(__cvta_generic_to_shared(smem_raw));
  uint8_t* smem = smem_raw + ((1024u - (base & 1023u)) & 1023u);
  uint64_t* full_bar = reinterpret_cast<uint64_t*>(smem + STAGES * kDenseStageBytes);
  uint64_t* empty_bar = full_bar + STAGES;
  float* factor_tab = reinterpret_cast<float*>(empty_bar + STAGES);
  float* div6_tab = factor_tab + 256;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], kDenseConsumerWarps);
    }
    fence_mbar_init();
  }
  __syncthreads();  // barriers ready: the producer starts streaming at once

  if (warp == kDenseConsumerWarps) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      prefetch_tensormap(&tmap);
      // the first tiles' input into L2 while the previous kernel finishes
      for (int t = blockIdx.x, i = 0; t < a.num_tiles && i < STAGES; t += gridDim.x, ++i) {
        const int mt = t / a.tiles_k, col0 = (t - mt * a.tiles_k) * kDenseTileCols;
        tma_prefetch_2d(&tmap, col0, mt * kDenseTileRows);
        if (col0 + kDenseBoxCols < a.K) tma_prefetch_2d(&tmap, col0 + kDenseBoxCols, mt * kDenseTileRows);
      }
      pdl_wait();
      int stage = 0;
      uint32_t phase = 0;
      uint32_t used = 0, last_parity = 0;  // per-stage bit masks
      for (int t = blockIdx.x; t < a.num_tiles; t += gridDim.x) {
        if (!mbar_wait_bounded(&empty_bar[stage], phase ^ 1u)) {
          record_error(kErrTimeout);
          break;
        }
        const int mt = t / a.tiles_k, kt = t - mt * a.tiles_k;
        const int col0 = kt * kDenseTileCols;
        const bool second = col0 + kDenseBoxCols < a.K;
        uint8_t* dst = smem + stage * kDenseStageBytes;
        mbar_arrive_expect_tx(&full_bar[stage], second ? kDenseStageBytes : kDenseBoxBytes);
        tma_load_2d(dst, &tmap, col0, mt * kDenseTileRows, &full_bar[stage]);
        if (second)
          tma_load_2d(dst + kDenseBoxBytes, &tmap, col0 + kDenseBoxCols, mt * kDenseTileRows,
                      &full_bar[stage]);
        used |= 1u << stage;
        last_parity = (last_parity & ~(1u << stage)) | (phase << stage);
        if (++stage == STAGES) {
          stage = 0;
          phase ^= 1u;
        }
      }
      // the next kernel may launch once every tile load is issued (earlier,
      // its blocks would sit beside these CTAs for the whole launch)
      pdl_trigger();
      // Never leave the CTA with a TMA write still landing in shared memory.
      for (int s = 0; s < STAGES; ++s)
        if ((used >> s) & 1u)
          if (!mbar_wait_bounded(&full_bar[s], (last_parity >> s) & 1u)) record_error(kErrTimeout);
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  // NVFP4 scale tables, filled while the first tiles are in flight; named
  // barrier 1 synchronizes the consumer warps only.
  float tsf = a.tsf;
  bool store_ok = true;
  if constexpr (FMT == kNVFP4) {
    if (a.tsf_dev != nullptr) {
      // written by an earlier kernel in the stream: wait for it, read past L1
      pdl_wait();
      tsf = __ldcg(a.tsf_dev);
      if (!(tsf > 0.0f && tsf <= 3.4028234663852886e38f)) {
        if (threadIdx.x == 0) record_error(kErrValue);
        store_ok = false;
        tsf = 1.0f;
      }
    }
    fill_nvfp4_factor_table(factor_tab, tsf, threadIdx.x, 32 * kDenseConsumerWarps);
    fill_div6_table(div6_tab, threadIdx.x, 32 * kDenseConsumerWarps);
    asm volatile("bar.sync 1, %0;" ::"n"(32 * kDenseConsumerWarps) : "memory");
  }
  pdl_wait();

  // warp -> box h; lane -> row: r32 = 8*(warp%4) + lane%8, r4 = lane/8,
  // row = r32 + 32*r4, so a warp's 32 scale words fill 128 contiguous bytes.
  const int h = warp >> 2;
  const int r32 = 8 * (warp & 3) + (lane & 7);
  const int r4 = lane >> 3;
  const int row = r32 + 32 * r4;
  const int atom_off = r32 * 16 + r4 * 4;  // this row's word inside a 512-byte atom
  const NvScale ns{tsf, factor_tab, div6_tab};

  int stage = 0;
  uint32_t phase = 0;
  for (int t = blockIdx.x; t < a.num_tiles; t += gridDim.x) {
    if (!mbar_wait_bounded(&full_bar[stage], phase)) {
      record_error(kErrTimeout);
      break;
    }
    const int mt = t / a.tiles_k, kt = t - mt * a.tiles_k;
    const int col0 = kt * kDenseTileCols + h * kDenseBoxCols;
    const bool valid = col0 < a.K;
    const int64_t grow = static_cast<int64_t>(mt) * kDenseTileRows + row;
    uint32_t sbytes = 0;
    if (valid) {
      uint8_t* dst = grow < a.M && store_ok ? a.out + grow * a.out_ld +
                                      (Fmt<FMT>::OUT_BITS == 4 ? (col0 >> 1) : col0)
                                : nullptr;
      sbytes = quant_box_row<FMT, true>(smem + stage * kDenseStageBytes + h * kDenseBoxBytes + row * 128,
                                        row, min(kDenseBoxCols, a.K - col0), dst, a.vec32 != 0, ns);
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty_bar[stage]);

    uint8_t* band = a.scales + static_cast<int64_t>(mt) * a.kt_atoms * 512 + atom_off;
    if (!store_ok) {
      // invalid device tensor_sf: nothing is written
    } else if constexpr (FMT == kNVFP4) {
      // one atom (64 columns) per box
      if (valid) *reinterpret_cast<uint32_t*>(band + (2 * kt + h) * 512) = sbytes;
    } else {
      // one atom per tile: box h holds its blocks 2h and 2h+1
      *reinterpret_cast<uint16_t*>(band + kt * 512 + 2 * h) = static_cast<uint16_t>(sbytes);
    }
    if (++stage == STAGES) {
      stage = 0;
      phase ^= 1u;
    }
  }
}

}  // namespace bsq
