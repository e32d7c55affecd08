// Device helpers shared by the libbsq kernels (sm_103a): format traits,
// conversions through the hardware cvt instructions, bounded mbarrier waits
// and TMA loads written as inline PTX.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

namespace bsq {

enum : int { kNVFP4 = 0, kMXFP4 = 1, kMXFP8 = 2 };
enum : unsigned { kErrValue = 4u, kErrTimeout = 6u };

// Block-scaled format traits.  SF: elements per scale factor.  ATOM_COLS:
// input columns covered by one 5D scale atom column (4 scale factors).
template <int FMT> struct Fmt;
template <> struct Fmt<kNVFP4> { static constexpr int SF = 16, ATOM_COLS = 64, OUT_BITS = 4; };
template <> struct Fmt<kMXFP4> { static constexpr int SF = 32, ATOM_COLS = 128, OUT_BITS = 4; };
template <> struct Fmt<kMXFP8> { static constexpr int SF = 32, ATOM_COLS = 128, OUT_BITS = 8; };

// ---------------------------------------------------------------- errors --
// One error word per device; the first recorded code wins.
__device__ unsigned int g_error_word;

__device__ __forceinline__ void record_error(unsigned code) {
  atomicCAS(&g_error_word, 0u, code);
}

// ------------------------------------------------------------ conversion --
// BF16 pair (one 32-bit word) -> two FP32 values (exact).
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Running max of |x| over BF16 pairs; the result is two BF16 magnitudes.
__device__ __forceinline__ uint32_t absmax2(uint32_t acc, uint32_t w) {
  uint32_t r;
  asm("max.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(acc), "r"(w & 0x7FFF7FFFu));
  return r;
}
// Reduce the two halves of an absmax2 accumulator to one FP32 amax.  The
// halves are non-negative BF16 values, which order like their bit patterns.
__device__ __forceinline__ float absmax_final(uint32_t acc) {
  return __uint_as_float(max(acc << 16, acc & 0xFFFF0000u));
}

// FP32 -> E4M3 (round to nearest even, saturate to +-448), result in the low byte.
__device__ __forceinline__ uint32_t f32_to_e4m3(float s) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(0.0f), "f"(s));
  return r & 0xFFu;
}

// E4M3 byte -> FP32 (exact: E4M3 is a subset of FP16).
__device__ __forceinline__ float e4m3_to_f32(uint32_t b) {
  uint32_t h2;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(static_cast<uint16_t>(b)));
  return __half2float(__ushort_as_half(static_cast<unsigned short>(h2 & 0xFFFFu)));
}

// Eight FP32 values -> eight E2M1 codes packed in one word, element 0 in the
// low nibble.  cvt ...e2m1x2 puts its first source in the high nibble.
__device__ __forceinline__ uint32_t pack_e2m1x8(float a0, float a1, float a2, float a3,
                                                float a4, float a5, float a6, float a7) {
  uint32_t r;
  asm("{\n\t.reg .b8 q0, q1, q2, q3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 q0, %2, %1;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 q1, %4, %3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 q2, %6, %5;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 q3, %8, %7;\n\t"
      "mov.b32 %0, {q0, q1, q2, q3};\n\t}"
      : "=r"(r)
      : "f"(a0), "f"(a1), "f"(a2), "f"(a3), "f"(a4), "f"(a5), "f"(a6), "f"(a7));
  return r;
}

// Four FP32 values -> four E4M3 bytes in one word, element 0 in the low byte.
__device__ __forceinline__ uint32_t pack_e4m3x4(float a0, float a1, float a2, float a3) {
  uint32_t r;
  asm("{\n\t.reg .b16 h0, h1;\n\t"
      "cvt.rn.satfinite.e4m3x2.f32 h0, %2, %1;\n\t"
      "cvt.rn.satfinite.e4m3x2.f32 h1, %4, %3;\n\t"
      "mov.b32 %0, {h0, h1};\n\t}"
      : "=r"(r)
      : "f"(a0), "f"(a1), "f"(a2), "f"(a3));
  return r;
}

// Scale the 8 BF16 elements of `w` by f (each product rounded to FP32) and
// encode them as 8 E2M1 codes (one word).
__device__ __forceinline__ uint32_t quant8_e2m1(uint4 w, float f) {
  return pack_e2m1x8(__fmul_rn(bf16_lo(w.x), f), __fmul_rn(bf16_hi(w.x), f),
                     __fmul_rn(bf16_lo(w.y), f), __fmul_rn(bf16_hi(w.y), f),
                     __fmul_rn(bf16_lo(w.z), f), __fmul_rn(bf16_hi(w.z), f),
                     __fmul_rn(bf16_lo(w.w), f), __fmul_rn(bf16_hi(w.w), f));
}

// Same for E4M3: 8 bytes (two words).
__device__ __forceinline__ uint2 quant8_e4m3(uint4 w, float f) {
  uint2 r;
  r.x = pack_e4m3x4(__fmul_rn(bf16_lo(w.x), f), __fmul_rn(bf16_hi(w.x), f),
                    __fmul_rn(bf16_lo(w.y), f), __fmul_rn(bf16_hi(w.y), f));
  r.y = pack_e4m3x4(__fmul_rn(bf16_lo(w.z), f), __fmul_rn(bf16_hi(w.z), f),
                    __fmul_rn(bf16_lo(w.w), f), __fmul_rn(bf16_hi(w.w), f));
  return r;
}

// ----------------------------------------------------------- block scales --
struct BlockScale {
  uint32_t byte;  // scale factor as stored (E4M3 or E8M0)
  float factor;   // multiplier applied to the elements before encoding
};

// NVFP4: s = fl32(fl32(amax / 6) * tensor_sf) -> E4M3; element scale
// tensor_sf / decoded scale (0 when the decoded scale is 0).
__device__ __forceinline__ BlockScale nvfp4_scale(float amax, float tsf) {
  const float s = __fmul_rn(__fdiv_rn(amax, 6.0f), tsf);
  const uint32_t b = f32_to_e4m3(s);
  const float ds = e4m3_to_f32(b);
  return {b, ds == 0.0f ? 0.0f : __fdiv_rn(tsf, ds)};
}

// MX: e = ceil(log2(fl32(amax / Qmax))) clamped to [-127, 127] (-127 for a
// zero block), taken exactly from the FP32 bits of the quotient; byte e+127,
// element factor 2^-e.
template <int QMAX>
__device__ __forceinline__ BlockScale mx_scale(float amax) {
  const float s = __fdiv_rn(amax, static_cast<float>(QMAX));
  const uint32_t bits = __float_as_uint(s);
  const int ex = static_cast<int>(bits >> 23);
  int e;
  if (ex == 0) {
    // zero or subnormal: s <= 2^-127 -> -127 (after the clamp), else -126
    e = bits > 0x00400000u ? -126 : -127;
  } else {
    e = ex - 127 + ((bits & 0x007FFFFFu) != 0u ? 1 : 0);
    e = min(e, 127);
  }
  // 2^-e: normal for -e >= -126; 2^-127 is the subnormal 0x00400000
  const uint32_t fbits = (e == 127) ? 0x00400000u : static_cast<uint32_t>(127 - e) << 23;
  return {static_cast<uint32_t>(e + 127), __uint_as_float(fbits)};
}

// ------------------------------------------------------------------- PTX --
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count));
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0u;
}

// Wait until the phase with the given parity has completed, for at most
// about one second; false when the limit expired.
constexpr uint64_t kWaitLimitNs = 1000000000ull;
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (globaltimer_ns() - t0 > kWaitLimitNs) return false;
  }
}

// 2D TMA tile load into shared memory, completing on `bar` (tx bytes).
// x is the innermost (element) coordinate, y the row.
__device__ __forceinline__ void tma_load_2d(void* smem_dst, const CUtensorMap* map, int32_t x,
                                            int32_t y, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_addr(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_addr(bar))
      : "memory");
}

__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// 32-byte and 16-byte global stores.
__device__ __forceinline__ void st_global_v8(void* p, const uint32_t (&v)[8]) {
  asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(p), "r"(v[0]),
               "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7])
               : "memory");
}
__device__ __forceinline__ void st_global_v4(void* p, uint32_t a, uint32_t b, uint32_t c,
                                             uint32_t d) {
  asm volatile("st.global.v4.b32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(a), "r"(b), "r"(c),
               "r"(d)
               : "memory");
}

// Read-only 16-byte global load that does not allocate in L1.
__device__ __forceinline__ uint4 ld_global_nc_v4(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.b32 {%0, %1, %2, %3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

}  // namespace bsq
