// A producer with the quantize in its epilogue: C = A * B^T (BF16 operands,
// FP32 accumulation, C rounded to BF16) quantized block-wise along N into
// packed codes and 5D scales, with no BF16 C written to memory.  The
// block_scaled_quantization module page (function list,
// block_scaled_matmul_with_epilogue) runs elementwise epilogues of its
// block-scaled matmul as a separate kernel, and its quantize kernels read a
// BF16 tensor stored by an earlier kernel; here the quantize is the epilogue
// of the producing matmul.
//
// Blackwell 5th-generation tensor cores (sm_103a), one CTA per SM,
// persistent over 128 (M) x 256 (N) output tiles:
//  * warp 0, one lane: TMA producer.  Per 64-wide K step it loads the A box
//    (64 x 128 rows) and the B box (64 x 256 rows), both with the 128-byte
//    swizzle, into a kGmStages-deep ring of shared-memory stages ("full" /
//    "empty" mbarriers);
//  * warp 1: allocates the tensor memory (two 256-column FP32 accumulators,
//    all 512 columns) and, from one lane, issues tcgen05.mma (kind::f16,
//    BF16 x BF16 -> FP32, M = 128, N = 256, K = 16; four per stage), reading
//    both operands from shared memory through matrix descriptors;
//    tcgen05.commit returns each stage to the producer and announces each
//    finished accumulator;
//  * warps 2-5: the epilogue.  Warp w reads TMEM lanes 32 (w % 4) ..
//    32 (w % 4) + 31 (tcgen05.ld 32x32b), so each thread holds one output
//    row; it rounds 64 columns at a time to BF16 in registers and quantizes
//    them with the dense kernel's box routine (4 NVFP4 or 2 MX scale
//    blocks), storing the packed bytes and the scale word at its 5D offset,
//    while the tensor cores already accumulate the next tile in the other
//    accumulator.
// Every mbarrier wait is bounded (about a second); an expired wait records
// BSQ_ERR_TIMEOUT, stops every role, waits (bounded) for the copies and
// tensor-core operations already issued, frees the tensor memory and returns.
#pragma once

#include "box_quant.cuh"
#include "device_common.cuh"

namespace bsq {

constexpr int kGmBM = 128, kGmBN = 256, kGmBK = 64;  // tile rows, tile columns, K per stage
constexpr int kGmStages = 4;
constexpr int kGmThreads = 192;                      // producer, MMA and four epilogue warps
constexpr int kGmABytes = kGmBM * kGmBK * 2;         // 16 KB
constexpr int kGmBBytes = kGmBN * kGmBK * 2;         // 32 KB
constexpr int kGmStageBytes = kGmABytes + kGmBBytes; // 48 KB
constexpr int kGmTmemCols = 2 * kGmBN;               // two FP32 accumulators

__host__ __device__ constexpr int gemm_smem_bytes() {
  // stages (1024-byte aligned) + alignment slack + barriers + tables + TMEM address
  return kGmStages * kGmStageBytes + 1024 + (2 * kGmStages + 4 + 1) * 8 + (256 + 128) * 4 + 32;
}

struct GemmQuantArgs {
  int64_t M;
  int N, K;
  float tsf;          // NVFP4 tensor scale
  uint8_t* out;       // M x out_ld packed codes
  int64_t out_ld;
  uint8_t* scales;    // 5D scales, kt_atoms atoms per 128-row band
  int kt_atoms;
  uint16_t* c;        // optional M x N BF16 copy of C (tests), row stride N
  int vec32;          // packed rows allow 32-byte stores
  int tiles_m, tiles_n;
};

// ------------------------------------------------------------- tcgen05 --

// Shared-memory matrix descriptor of a K-major operand tile laid out by a
// TMA load with the 128-byte swizzle: rows of 64 BF16 (128 bytes), groups of
// 8 rows 1024 bytes apart (stride byte offset), start address advanced by
// 32 bytes per K = 16 slice inside the swizzle atom.  Fields: start address
// >> 4 (bits 0-13), leading byte offset >> 4 (16-29; unused for swizzled
// K-major tiles, 1), stride byte offset >> 4 (32-45), the fixed 0b001 at
// 46-48, swizzle mode 2 = 128 bytes (61-63).
__device__ __forceinline__ uint64_t umma_desc_sw128(uint32_t saddr) {
  return static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4) | (static_cast<uint64_t>(1) << 16) |
         (static_cast<uint64_t>(1024 >> 4) << 32) | (static_cast<uint64_t>(1) << 46) |
         (static_cast<uint64_t>(2) << 61);
}

// Instruction descriptor of kind::f16: D FP32 (bits 4-5 = 1), A and B BF16
// (7-9 = 1, 10-12 = 1), both K-major (bits 15, 16 = 0), N >> 3 at 17-22,
// M >> 4 at 24-28.
constexpr uint32_t kGmIdesc = (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(kGmBN >> 3) << 17) |
                              (static_cast<uint32_t>(kGmBM >> 4) << 24);

__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(kGmIdesc), "r"(accumulate)
      : "memory");
}

// Arrive once on `bar` when every tcgen05 operation this thread issued so far
// has completed.
__device__ __forceinline__ void umma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_addr(bar))
               : "memory");
}

__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }

// 32 consecutive FP32 columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// The epilogue of one 64-column box of this thread's row m: BF16 rounding,
// quantize, packed bytes (rows < M), scale word (every row of the band), and
// the optional BF16 copy of C.
template <int FMT>
__device__ __forceinline__ void gm_box(const GemmQuantArgs& p, const uint32_t (&lo)[32], const uint32_t (&hi)[32],
                                       int64_t m, int n0, const NvScale& ns) {
  uint4 v[8];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    v[q] = make_uint4(pack_bf16x2(__uint_as_float(lo[8 * q]), __uint_as_float(lo[8 * q + 1])),
                      pack_bf16x2(__uint_as_float(lo[8 * q + 2]), __uint_as_float(lo[8 * q + 3])),
                      pack_bf16x2(__uint_as_float(lo[8 * q + 4]), __uint_as_float(lo[8 * q + 5])),
                      pack_bf16x2(__uint_as_float(lo[8 * q + 6]), __uint_as_float(lo[8 * q + 7])));
    v[4 + q] = make_uint4(pack_bf16x2(__uint_as_float(hi[8 * q]), __uint_as_float(hi[8 * q + 1])),
                          pack_bf16x2(__uint_as_float(hi[8 * q + 2]), __uint_as_float(hi[8 * q + 3])),
                          pack_bf16x2(__uint_as_float(hi[8 * q + 4]), __uint_as_float(hi[8 * q + 5])),
                          pack_bf16x2(__uint_as_float(hi[8 * q + 6]), __uint_as_float(hi[8 * q + 7])));
  }
  const bool live = m < p.M;
  if (live && p.c != nullptr) {
    uint4* cd = reinterpret_cast<uint4*>(p.c + m * p.N + n0);
#pragma unroll
    for (int q = 0; q < 8; ++q) cd[q] = v[q];
  }
  uint8_t* dst = live ? p.out + m * p.out_ld + (Fmt<FMT>::OUT_BITS == 4 ? n0 / 2 : n0) : nullptr;
  const uint32_t sbytes = quant_box_regs<FMT>(v, 64, dst, p.vec32 != 0, ns);
  const int64_t s0 = n0 / Fmt<FMT>::SF;  // first scale column of the box
  uint8_t* word = p.scales + ((m >> 7) * p.kt_atoms + (s0 >> 2)) * 512 + (m & 31) * 16 + ((m & 127) >> 5) * 4;
  if constexpr (FMT == kNVFP4) {
    *reinterpret_cast<uint32_t*>(word) = sbytes;
  } else {
    *reinterpret_cast<uint16_t*>(word + (s0 & 3)) = static_cast<uint16_t>(sbytes);
  }
}

// Grid: min(tiles, SMs) CTAs of kGmThreads; tile t covers rows
// 128 (t / tiles_n) and columns 256 (t % tiles_n).
template <int FMT>
__global__ void __launch_bounds__(kGmThreads, 1)
    gemm_quant_kernel(const __grid_constant__ CUtensorMap tma_a, const __grid_constant__ CUtensorMap tma_b,
                      const GemmQuantArgs p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t base = static_cast<uint32_t>(__cvta_generic_to_shared(smem_raw));
  uint8_t* smem = smem_raw + ((1024u - (base & 1023u)) & 1023u);
  uint64_t* full_bar = reinterpret_cast<uint64_t*>(smem + kGmStages * kGmStageBytes);
  uint64_t* empty_bar = full_bar + kGmStages;
  uint64_t* acc_full = empty_bar + kGmStages;   // [2]: accumulator ready for the epilogue
  uint64_t* acc_empty = acc_full + 2;           // [2]: accumulator drained by the epilogue
  uint64_t* drain_bar = acc_empty + 2;          // the MMA warp's last operations, before the TMEM is freed
  float* factor_tab = reinterpret_cast<float*>(drain_bar + 1);
  float* div6_tab = factor_tab + 256;
  volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(div6_tab + 128);
  volatile uint32_t* abort_flag = tmem_slot + 1;
  volatile uint32_t* counts = tmem_slot + 2;  // [0] stages filled, [1] stages consumed

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int num_tiles = p.tiles_m * p.tiles_n;
  const int kb_total = (p.K + kGmBK - 1) / kGmBK;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kGmStages; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&acc_full[b], 1);
      mbar_init(&acc_empty[b], 4);
    }
    mbar_init(drain_bar, 1);
    *abort_flag = 0u;
    counts[0] = counts[1] = 0u;
    fence_mbar_init();
  }
  if (warp >= 2) {
    if constexpr (FMT == kNVFP4) {
      fill_div6_table(div6_tab, threadIdx.x - 64, 128);
      fill_nvfp4_factor_table(factor_tab, p.tsf, threadIdx.x - 64, 128);
    }
  }
  if (warp == 1) {  // the whole warp allocates the tensor memory
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_addr(const_cast<uint32_t*>(tmem_slot))),
                 "r"(kGmTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  pdl_wait();

  if (warp == 0) {
    // ---- TMA producer
    if (lane == 0) {
      prefetch_tensormap(&tma_a);
      prefetch_tensormap(&tma_b);
      uint32_t stage = 0, phase = 0, fills = 0;
      for (int t = blockIdx.x; t < num_tiles && *abort_flag == 0u; t += gridDim.x) {
        const int m0 = (t / p.tiles_n) * kGmBM, n0 = (t % p.tiles_n) * kGmBN;
        for (int kb = 0; kb < kb_total; ++kb) {
          if (!mbar_wait_bounded(&empty_bar[stage], phase ^ 1u)) {
            record_error(kErrTimeout);
            *abort_flag = 1u;
            break;
          }
          uint8_t* st = smem + stage * kGmStageBytes;
          mbar_arrive_expect_tx(&full_bar[stage], kGmStageBytes);
          tma_load_2d(st, &tma_a, kb * kGmBK, m0, &full_bar[stage]);
          tma_load_2d(st + kGmABytes, &tma_b, kb * kGmBK, n0, &full_bar[stage]);
          ++fills;
          if (++stage == kGmStages) { stage = 0; phase ^= 1u; }
        }
      }
      counts[0] = fills;
    }
  } else if (warp == 1) {
    // ---- MMA issuer
    if (lane == 0) {
      uint32_t stage = 0, phase = 0, consumed = 0;
      int it = 0;
      for (int t = blockIdx.x; t < num_tiles && *abort_flag == 0u; t += gridDim.x, ++it) {
        const uint32_t acc = it & 1, acc_phase = (it >> 1) & 1;
        if (!mbar_wait_bounded(&acc_empty[acc], acc_phase ^ 1u)) {
          record_error(kErrTimeout);
          *abort_flag = 1u;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * kGmBN;
        bool ok = true;
        for (int kb = 0; kb < kb_total; ++kb) {
          if (!mbar_wait_bounded(&full_bar[stage], phase)) {
            record_error(kErrTimeout);
            *abort_flag = 1u;
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a_addr = smem_addr(smem + stage * kGmStageBytes);
          const uint32_t b_addr = a_addr + kGmABytes;
#pragma unroll
          for (int k = 0; k < kGmBK / 16; ++k)
            umma_bf16(d_tmem, umma_desc_sw128(a_addr + 32 * k), umma_desc_sw128(b_addr + 32 * k),
                      (kb > 0 || k > 0) ? 1u : 0u);
          umma_commit(&empty_bar[stage]);  // the stage is free once these MMAs are done
          ++consumed;
          if (++stage == kGmStages) { stage = 0; phase ^= 1u; }
        }
        if (!ok) break;
        umma_commit(&acc_full[acc]);  // the accumulator is complete
      }
      umma_commit(drain_bar);  // every MMA issued has completed when this arrives
      if (!mbar_wait_bounded(drain_bar, 0)) record_error(kErrTimeout);
      counts[1] = consumed;
    }
  } else {
    // ---- epilogue: warp w owns TMEM lanes 32 (w % 4) .. + 31
    const int quarter = warp & 3;
    const NvScale ns{p.tsf, factor_tab, div6_tab};
    int it = 0;
    for (int t = blockIdx.x; t < num_tiles; t += gridDim.x, ++it) {
      const uint32_t acc = it & 1, acc_phase = (it >> 1) & 1;
      bool ok = true;
      if (lane == 0) ok = mbar_wait_bounded(&acc_full[acc], acc_phase);
      ok = __shfl_sync(0xFFFFFFFFu, ok ? 1 : 0, 0) != 0;
      if (!ok || *abort_flag != 0u) {  // warp-uniform
        if (lane == 0 && !ok) {
          record_error(kErrTimeout);
          *abort_flag = 1u;
        }
        break;
      }
      __syncwarp();
      tc_fence_after();
      const int64_t m = static_cast<int64_t>(t / p.tiles_n) * kGmBM + 32 * quarter + lane;
      const int n_tile = (t % p.tiles_n) * kGmBN;
      const uint32_t taddr = tmem_base + (static_cast<uint32_t>(32 * quarter) << 16) + acc * kGmBN;
#pragma unroll 1
      for (int bx = 0; bx < kGmBN / 64; ++bx) {
        if (n_tile + 64 * bx >= p.N) break;  // warp-uniform
        uint32_t lo[32], hi[32];
        tmem_ld32(taddr + 64 * bx, lo);
        tmem_ld32(taddr + 64 * bx + 32, hi);
        tmem_ld_wait();
        gm_box<FMT>(p, lo, hi, m, n_tile + 64 * bx, ns);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acc_empty[acc]);
    }
  }

  __syncthreads();
  // loads issued but never consumed (only after an expired wait) land
  // before the CTA may finish: fill f sits in stage f % kGmStages, phase f / kGmStages
  if (threadIdx.x == 0) {
    for (uint32_t f = counts[1]; f < counts[0]; ++f)
      if (!mbar_wait_bounded(&full_bar[f % kGmStages], (f / kGmStages) & 1u)) record_error(kErrTimeout);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) {
    __syncwarp();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(kGmTmemCols)
                 : "memory");
  }
}

}  // namespace bsq
