// A producer with the quantize in its epilogue: C = A * B^T (BF16 operands,
// FP32 accumulation, C rounded to BF16) quantized block-wise along N into
// packed codes and 5D scales, with no BF16 C written to memory.  The
// block_scaled_quantization module page (function list,
// block_scaled_matmul_with_epilogue) runs elementwise epilogues of its
// block-scaled matmul as a separate kernel, and its quantize kernels read a
// BF16 tensor stored by an earlier kernel; here the quantize is the epilogue
// of the producing matmul.
//
// Block tile 64 (M) x 64 (N), K in steps of 32, four warps of 32 x 32 on the
// mma.sync m16n8k16 BF16 tensor-core path (operands staged in shared memory,
// fragments by ldmatrix, the next K step loaded into registers while the
// current one multiplies).  Epilogue: the FP32 tile rounded to BF16 into
// shared memory, then one thread per row quantizes its 64 columns with the
// dense kernel's per-row box routine (4 NVFP4 or 2 MX scale blocks) and
// writes the packed bytes and the row's scale word (NVFP4) or half word (MX)
// at its 5D offset.  Rows past M (up to the end of the last 128-row band)
// get zero scales and no packed bytes.  The mainloop is the legacy warp-level
// tensor-core path, not tcgen05: the contraction here only feeds the fused
// epilogue.
#pragma once

#include "box_quant.cuh"
#include "device_common.cuh"

namespace bsq {

constexpr int kGqBM = 64, kGqBN = 64, kGqBK = 32;
constexpr int kGqThreads = 128;
constexpr int kGqPitch = kGqBK + 8;  // operand tile row pitch (elements): 80 bytes
constexpr int kGqCPitch = kGqBN + 8; // C tile row pitch (elements): 144 bytes

struct GemmQuantArgs {
  const uint16_t* a;  // M x K BF16, row stride lda
  const uint16_t* b;  // N x K BF16, row stride ldb
  int64_t M;
  int N, K;
  int64_t lda, ldb;
  float tsf;          // NVFP4 tensor scale
  uint8_t* out;       // M x out_ld packed codes
  int64_t out_ld;
  uint8_t* scales;    // 5D scales, kt_atoms atoms per 128-row band
  int kt_atoms;
  uint16_t* c;        // optional M x N BF16 copy of C (tests), row stride N
  int vec32;          // packed rows allow 32-byte stores
};

__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], const void* p) {
  const uint32_t s = static_cast<uint32_t>(__cvta_generic_to_shared(p));
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(s));
}

__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// One K step of the block's operand tiles into registers: thread tid moves
// 16-byte chunks tid and tid + 128 of each 64 x 32 tile (row c / 4, columns
// 8 * (c % 4)); A rows past M read as zeros.
__device__ __forceinline__ void gq_load(const GemmQuantArgs& p, int64_t m0, int n0, int k0, int tid, uint4 (&ra)[2],
                                        uint4 (&rb)[2]) {
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const int c = tid + i * kGqThreads, row = c >> 2, col = (c & 3) * 8;
    const int64_t gm = m0 + row;
    ra[i] = gm < p.M ? ld_global_nc_v4(p.a + gm * p.lda + k0 + col) : make_uint4(0u, 0u, 0u, 0u);
    rb[i] = ld_global_nc_v4(p.b + static_cast<int64_t>(n0 + row) * p.ldb + k0 + col);
  }
}

// Grid: (N / 64, 2 * ceil(M / 128)) blocks of kGqThreads.
template <int FMT>
__global__ void __launch_bounds__(kGqThreads) gemm_quant_kernel(const GemmQuantArgs p) {
  __shared__ __align__(16) uint16_t As[kGqBM][kGqPitch];
  __shared__ __align__(16) uint16_t Bs[kGqBN][kGqPitch];
  __shared__ __align__(16) uint16_t Cs[kGqBM][kGqCPitch];
  __shared__ float factor_tab[256];
  __shared__ float div6_tab[128];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int wm = warp >> 1, wn = warp & 1;  // warp tile: rows 32*wm, cols 32*wn
  const int n0 = blockIdx.x * kGqBN;
  const int64_t m0 = static_cast<int64_t>(blockIdx.y) * kGqBM;
  if constexpr (FMT == kNVFP4) {
    fill_div6_table(div6_tab, tid, kGqThreads);
    fill_nvfp4_factor_table(factor_tab, p.tsf, tid, kGqThreads);
  }
  pdl_wait();

  float acc[2][4][4];
#pragma unroll
  for (int i = 0; i < 2; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j)
#pragma unroll
      for (int r = 0; r < 4; ++r) acc[i][j][r] = 0.0f;

  if (m0 < p.M) {
    uint4 ra[2], rb[2];
    gq_load(p, m0, n0, 0, tid, ra, rb);
    for (int k0 = 0; k0 < p.K; k0 += kGqBK) {
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const int c = tid + i * kGqThreads, row = c >> 2, col = (c & 3) * 8;
        *reinterpret_cast<uint4*>(&As[row][col]) = ra[i];
        *reinterpret_cast<uint4*>(&Bs[row][col]) = rb[i];
      }
      __syncthreads();
      if (k0 + kGqBK < p.K) gq_load(p, m0, n0, k0 + kGqBK, tid, ra, rb);  // next step in flight
#pragma unroll
      for (int kk = 0; kk < kGqBK; kk += 16) {
        uint32_t af[2][4], bf[2][4];
#pragma unroll
        for (int i = 0; i < 2; ++i)  // 16 x 16 A tiles: lanes 0-15 rows, 16-31 the upper 8 columns
          ldsm_x4(af[i], &As[32 * wm + 16 * i + (lane & 15)][kk + 8 * (lane >> 4)]);
#pragma unroll
        for (int j = 0; j < 2; ++j)  // two n8 x k16 B tiles per load
          ldsm_x4(bf[j], &Bs[32 * wn + 16 * j + (lane & 7) + 8 * (lane >> 4)][kk + 8 * ((lane >> 3) & 1)]);
#pragma unroll
        for (int i = 0; i < 2; ++i)
#pragma unroll
          for (int j = 0; j < 4; ++j) mma_bf16_16816(acc[i][j], af[i], bf[j >> 1][2 * (j & 1)], bf[j >> 1][2 * (j & 1) + 1]);
      }
      __syncthreads();
    }
  }

  // epilogue: C rounded to BF16 into shared memory (m16n8 accumulator
  // layout: rows lane/4 and lane/4 + 8, columns 2 * (lane % 4) + {0, 1})
#pragma unroll
  for (int i = 0; i < 2; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int r = 32 * wm + 16 * i + (lane >> 2), c = 32 * wn + 8 * j + 2 * (lane & 3);
      *reinterpret_cast<uint32_t*>(&Cs[r][c]) = pack_bf16x2(acc[i][j][0], acc[i][j][1]);
      *reinterpret_cast<uint32_t*>(&Cs[r + 8][c]) = pack_bf16x2(acc[i][j][2], acc[i][j][3]);
    }
  __syncthreads();
  if (tid < kGqBM) {
    const int64_t m = m0 + tid;
    const bool live = m < p.M;
    uint8_t* dst = live ? p.out + m * p.out_ld + (Fmt<FMT>::OUT_BITS == 4 ? n0 / 2 : n0) : nullptr;
    const NvScale ns{p.tsf, factor_tab, div6_tab};
    const uint32_t sbytes =
        quant_box_row<FMT, false>(reinterpret_cast<const uint8_t*>(&Cs[tid][0]), tid, kGqBN, dst, p.vec32 != 0, ns);
    const int64_t s0 = n0 / Fmt<FMT>::SF;  // first scale column of the tile
    uint8_t* word = p.scales + ((m >> 7) * p.kt_atoms + (s0 >> 2)) * 512 + (m & 31) * 16 + ((m & 127) >> 5) * 4;
    if constexpr (FMT == kNVFP4) {
      *reinterpret_cast<uint32_t*>(word) = sbytes;
    } else {
      *reinterpret_cast<uint16_t*>(word + (s0 & 3)) = static_cast<uint16_t>(sbytes);
    }
    if (live && p.c != nullptr) {
      const uint4* src = reinterpret_cast<const uint4*>(&Cs[tid][0]);
      uint4* cd = reinterpret_cast<uint4*>(p.c + m * p.N + n0);
#pragma unroll
      for (int q = 0; q < kGqBN / 8; ++q) cd[q] = src[q];
    }
  }
}

}  // namespace bsq
