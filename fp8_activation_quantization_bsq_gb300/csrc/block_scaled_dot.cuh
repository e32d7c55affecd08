// Naive block-scaled matmul on the GPU, a consumer-side validator of the
// quantized operands: C[m][n] = sum_k deq(A)[m][k] * deq(B)[n][k], with A
// (M x K) and B (N x K) packed NVFP4 / MXFP4 / MXFP8 rows and their scales
// read through the 5D layout, the way the tensor cores read them.
//
// One thread per output, FP64 arithmetic: the product of two decoded
// elements and of two decoded block scales is exact in FP64, each block's
// element dot is exact, and blocks are accumulated in order of k.  The
// elements are decoded with the hardware conversions (cvt.rn.f16x2.e2m1x2 /
// .e4m3x2), E8M0 scales as exact powers of two.  Not a performance path.
#pragma once

#include "device_common.cuh"

namespace bsq {

// Two E2M1 codes (one packed byte, element 2k in the low nibble) -> FP32.
__device__ __forceinline__ float2 e2m1x2_to_f32(uint32_t byte) {
  uint32_t h2;
  asm("{\n\t.reg .b8 q;\n\tcvt.u8.u32 q, %1;\n\tcvt.rn.f16x2.e2m1x2 %0, q;\n\t}" : "=r"(h2) : "r"(byte));
  return make_float2(__half2float(__ushort_as_half(static_cast<unsigned short>(h2 & 0xFFFFu))),
                     __half2float(__ushort_as_half(static_cast<unsigned short>(h2 >> 16))));
}

// E8M0 byte b (0..254) -> 2^(b - 127), exact in FP64.
__device__ __forceinline__ double e8m0_to_f64(uint32_t b) {
  return __longlong_as_double(static_cast<long long>(b - 127 + 1023) << 52);
}

__device__ __forceinline__ int64_t offset5d(int64_t m, int64_t s, int64_t Kt) {
  return ((m >> 7) * Kt + (s >> 2)) * 512 + (m & 31) * 16 + ((m & 127) >> 5) * 4 + (s & 3);
}

template <int FMT>
__global__ void __launch_bounds__(256) block_scaled_dot_kernel(const uint8_t* __restrict__ a,
                                                               const uint8_t* __restrict__ sa,
                                                               const uint8_t* __restrict__ b,
                                                               const uint8_t* __restrict__ sb, int64_t M,
                                                               int64_t N, int K, double inv_tsf,
                                                               double* __restrict__ c) {
  constexpr int SF = Fmt<FMT>::SF;
  const int64_t n = static_cast<int64_t>(blockIdx.x) * 16 + (threadIdx.x & 15);
  const int64_t m = static_cast<int64_t>(blockIdx.y) * 16 + (threadIdx.x >> 4);
  pdl_wait();
  if (m >= M || n >= N) return;
  const int S = K / SF;
  const int64_t Kt = (S + 3) / 4;
  const int64_t row_bytes = Fmt<FMT>::OUT_BITS == 4 ? K / 2 : K;
  const uint8_t* ar = a + m * row_bytes;
  const uint8_t* br = b + n * row_bytes;
  double acc = 0.0;
  for (int s = 0; s < S; ++s) {
    double dot = 0.0;  // exact: sums of products of E2M1 / E4M3 values
    if constexpr (Fmt<FMT>::OUT_BITS == 4) {
      for (int i = 0; i < SF / 2; ++i) {
        const float2 x = e2m1x2_to_f32(__ldg(ar + s * (SF / 2) + i));
        const float2 y = e2m1x2_to_f32(__ldg(br + s * (SF / 2) + i));
        dot += static_cast<double>(x.x) * y.x + static_cast<double>(x.y) * y.y;
      }
    } else {
      for (int i = 0; i < SF; ++i)
        dot += static_cast<double>(e4m3_to_f32(__ldg(ar + s * SF + i))) * e4m3_to_f32(__ldg(br + s * SF + i));
    }
    const uint32_t ba = __ldg(sa + offset5d(m, s, Kt)), bb = __ldg(sb + offset5d(n, s, Kt));
    const double scale = FMT == kNVFP4 ? static_cast<double>(e4m3_to_f32(ba)) * e4m3_to_f32(bb)
                                       : e8m0_to_f64(ba) * e8m0_to_f64(bb);
    acc += dot * scale;
  }
  c[m * N + n] = acc * inv_tsf;
}

}  // namespace bsq
