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

// Running max of |x| over BF16 pairs: max.xorsign.abs keeps max(|acc|, |w|)
// per half (its sign bit is the XOR of the inputs' signs and is masked off at
// the end).  NaN inputs are outside the contract.
__device__ __forceinline__ uint32_t absmax2(uint32_t acc, uint32_t w) {
  uint32_t r;
  asm("max.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(acc), "r"(w));
  return r;
}
// Reduce the two halves of an absmax2 accumulator to one FP32 amax.  The
// halves are BF16 magnitudes (after the sign mask), which order like their
// bit patterns.
__device__ __forceinline__ float absmax_final(uint32_t acc) {
  acc &= 0x7FFF7FFFu;
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

// Scale the 8 BF16 elements of `w` by f (each product rounded to FP32, two
// at a time with mul.rn.f32x2) and encode them as 8 E2M1 codes (one word,
// element 0 in the low nibble).
__device__ __forceinline__ uint32_t quant8_e2m1(uint4 w, float f) {
  uint32_t r;
  asm("{\n\t.reg .b32 l0, h0, l1, h1, l2, h2, l3, h3;\n\t"
      ".reg .b64 p0, p1, p2, p3, ff;\n\t"
      ".reg .b8 q0, q1, q2, q3;\n\t"
      "shl.b32 l0, %1, 16;\n\tand.b32 h0, %1, 0xFFFF0000;\n\t"
      "shl.b32 l1, %2, 16;\n\tand.b32 h1, %2, 0xFFFF0000;\n\t"
      "shl.b32 l2, %3, 16;\n\tand.b32 h2, %3, 0xFFFF0000;\n\t"
      "shl.b32 l3, %4, 16;\n\tand.b32 h3, %4, 0xFFFF0000;\n\t"
      "mov.b64 ff, {%5, %5};\n\t"
      "mov.b64 p0, {l0, h0};\n\tmul.rn.f32x2 p0, p0, ff;\n\tmov.b64 {l0, h0}, p0;\n\t"
      "mov.b64 p1, {l1, h1};\n\tmul.rn.f32x2 p1, p1, ff;\n\tmov.b64 {l1, h1}, p1;\n\t"
      "mov.b64 p2, {l2, h2};\n\tmul.rn.f32x2 p2, p2, ff;\n\tmov.b64 {l2, h2}, p2;\n\t"
      "mov.b64 p3, {l3, h3};\n\tmul.rn.f32x2 p3, p3, ff;\n\tmov.b64 {l3, h3}, p3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 q0, h0, l0;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 q1, h1, l1;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 q2, h2, l2;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 q3, h3, l3;\n\t"
      "mov.b32 %0, {q0, q1, q2, q3};\n\t}"
      : "=r"(r)
      : "r"(w.x), "r"(w.y), "r"(w.z), "r"(w.w), "f"(f));
  return r;
}

// Products of BF16 elements with a power of two p (given as BF16 bits, so p
// is exact in BF16): fma.rn.f32.bf16(x, p, -0) is the exact product rounded
// once to FP32, i.e. fl32(x * p), taking the BF16 halves of a word directly;
// the -0 addend keeps the sign of zero products.
#define BSQ_POW2_PRODUCTS_8                                                   \
  ".reg .b16 x0, x1, x2, x3, x4, x5, x6, x7, pw;\n\t"                         \
  ".reg .f32 y0, y1, y2, y3, y4, y5, y6, y7;\n\t"                             \
  "mov.b16 pw, %5;\n\t"                                                        \
  "mov.b32 {x0, x1}, %1;\n\tmov.b32 {x2, x3}, %2;\n\t"                         \
  "mov.b32 {x4, x5}, %3;\n\tmov.b32 {x6, x7}, %4;\n\t"                         \
  "fma.rn.f32.bf16 y0, x0, pw, 0f80000000;\n\t"                                \
  "fma.rn.f32.bf16 y1, x1, pw, 0f80000000;\n\t"                                \
  "fma.rn.f32.bf16 y2, x2, pw, 0f80000000;\n\t"                                \
  "fma.rn.f32.bf16 y3, x3, pw, 0f80000000;\n\t"                                \
  "fma.rn.f32.bf16 y4, x4, pw, 0f80000000;\n\t"                                \
  "fma.rn.f32.bf16 y5, x5, pw, 0f80000000;\n\t"                                \
  "fma.rn.f32.bf16 y6, x6, pw, 0f80000000;\n\t"                                \
  "fma.rn.f32.bf16 y7, x7, pw, 0f80000000;\n\t"

// 8 BF16 elements x 2^k -> 8 E2M1 codes (one word, element 0 low).
__device__ __forceinline__ uint32_t quant8_e2m1_pow2(uint4 w, uint16_t p_bf16) {
  uint32_t r;
  asm("{\n\t" BSQ_POW2_PRODUCTS_8
      ".reg .b8 q0, q1, q2, q3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 q0, y1, y0;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 q1, y3, y2;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 q2, y5, y4;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 q3, y7, y6;\n\t"
      "mov.b32 %0, {q0, q1, q2, q3};\n\t}"
      : "=r"(r)
      : "r"(w.x), "r"(w.y), "r"(w.z), "r"(w.w), "h"(p_bf16));
  return r;
}

// 8 BF16 elements x 2^k -> 8 E4M3 bytes (two words, element 0 low).
__device__ __forceinline__ uint2 quant8_e4m3_pow2(uint4 w, uint16_t p_bf16) {
  uint64_t r;
  asm("{\n\t" BSQ_POW2_PRODUCTS_8
      ".reg .b16 q0, q1, q2, q3;\n\t"
      "cvt.rn.satfinite.e4m3x2.f32 q0, y1, y0;\n\t"
      "cvt.rn.satfinite.e4m3x2.f32 q1, y3, y2;\n\t"
      "cvt.rn.satfinite.e4m3x2.f32 q2, y5, y4;\n\t"
      "cvt.rn.satfinite.e4m3x2.f32 q3, y7, y6;\n\t"
      "mov.b64 %0, {q0, q1, q2, q3};\n\t}"
      : "=l"(r)
      : "r"(w.x), "r"(w.y), "r"(w.z), "r"(w.w), "h"(p_bf16));
  return make_uint2(static_cast<uint32_t>(r), static_cast<uint32_t>(r >> 32));
}

// ----------------------------------------------------------- block scales --
struct BlockScale {
  uint32_t byte;  // scale factor as stored (E4M3 or E8M0)
  float factor;   // NVFP4: FP32 multiplier applied to the elements before encoding
};

struct MxScale {
  uint32_t byte;  // E8M0 scale byte e + 127
  uint16_t pow2;  // 2^-e as BF16 bits (exact)
};

// MX: e = ceil(log2(fl32(amax / Qmax))) clamped to [-127, 127] (-127 for a
// zero block); byte e+127, element factor 2^-e.
//
// No division is needed.  amax is a BF16 magnitude (8 significant bits) and
// Qmax = 1.5 * 2^2 (E2M1) or 1.75 * 2^8 (E4M3).  The exact quotient r is a
// power of two only when amax's significand equals Qmax's; otherwise r is at
// least a relative 2^-9 away from every power of two, so rounding r to FP32
// cannot reach one and ceil(log2(fl32(r))) = ceil(log2(r)).  With
// amax = 1.f * 2^E: e = E - log2(Qmax / 1.q) + (1.f > 1.q), where 1.q is
// Qmax's significand.  Zero and subnormal amax give e < -127 (clamped).
template <int QMAX>
__device__ __forceinline__ MxScale mx_scale(float amax) {
  static_assert(QMAX == 6 || QMAX == 448, "Qmax is 6 (E2M1) or 448 (E4M3)");
  constexpr int kExpQ = QMAX == 6 ? 2 : 8;                        // Qmax = 1.q * 2^kExpQ
  constexpr uint32_t kSigQ = QMAX == 6 ? 0x00400000u : 0x00600000u;  // 1.q fraction bits
  const uint32_t bits = __float_as_uint(amax);
  int e = static_cast<int>(bits >> 23) - 127 - kExpQ + ((bits & 0x007FFFFFu) > kSigQ ? 1 : 0);
  e = max(e, -127);
  // 2^-e is a normal BF16 value for e in [-127, 126], the range reachable here
  return {static_cast<uint32_t>(e + 127), static_cast<uint16_t>((127 - e) << 7)};
}

// NVFP4 element-scale table: os[b] = tensor_sf / decode(b) for every E4M3
// byte b (0 when the decoded value is 0; NaN codes are never produced by the
// block-scale encode).  Filled once per thread block in shared memory so that
// each block scale costs one lookup instead of a division.
__device__ __forceinline__ void fill_nvfp4_factor_table(float* tab, float tsf, int tid, int nthreads) {
  for (int b = tid; b < 256; b += nthreads) {
    const float ds = e4m3_to_f32(static_cast<uint32_t>(b));
    tab[b] = (ds == 0.0f || b == 0x7F || b == 0xFF) ? 0.0f : __fdiv_rn(tsf, fabsf(ds));
  }
}

// fl32(amax / 6) without a division for BF16 amax.  With
// amax = (1 + f/128) * 2^(E-127) (E the biased exponent, f the 7 fraction
// bits), amax / 6 = ((128 + f) / 192) * 2^(E-129): the quotient of the
// significands, rounded once, scaled by a power of two.  Scaling is exact
// while the result stays normal (E >= 5); smaller amax take the division.
// div6_tab[f] = fl32((128 + f) / 192).
__device__ __forceinline__ void fill_div6_table(float* tab, int tid, int nthreads) {
  for (int f = tid; f < 128; f += nthreads) tab[f] = __fdiv_rn(static_cast<float>(128 + f), 192.0f);
}
__device__ __forceinline__ float amax_div6(float amax, const float* div6_tab) {
  const uint32_t bits = __float_as_uint(amax);
  const uint32_t e = bits >> 23;
  if (e < 5u) return __fdiv_rn(amax, 6.0f);
  return __fmul_rn(div6_tab[(bits >> 16) & 0x7Fu], __uint_as_float((e - 2u) << 23));
}

// ------------------------------------------------------------------- PTX --

// Programmatic dependent launch.  pdl_wait(): block until the grids this one
// depends on (the previous kernels in the stream) have completed and their
// memory is visible; every kernel calls it before its first global memory
// access, so that only its prologue overlaps the previous kernel's tail (a
// no-op when the launch was not programmatic).  pdl_trigger(): allow the next
// kernel in the stream to launch now (it still waits for this grid's
// completion before touching memory).
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
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

// Prefetch a 2D TMA tile into L2 (no shared memory, no completion).  L2 is
// the point of coherence for global memory, so a prefetch issued before a
// dependent-launch wait cannot make a later read see stale data.
__device__ __forceinline__ void tma_prefetch_2d(const CUtensorMap* map, int32_t x, int32_t y) {
  asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(x), "r"(y)
               : "memory");
}

__device__ __forceinline__ void prefetch_l2(const void* p) {
  asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
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

// Read-only 32-byte global load that does not allocate in L1.
__device__ __forceinline__ void ld_global_nc_v8(const void* p, uint4& lo, uint4& hi) {
  asm volatile("ld.global.nc.L1::no_allocate.v8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
               : "=r"(lo.x), "=r"(lo.y), "=r"(lo.z), "=r"(lo.w), "=r"(hi.x), "=r"(hi.y),
                 "=r"(hi.z), "=r"(hi.w)
               : "l"(p));
}

// L2 cache policy for loads: keep the lines (evict_last) for a following
// pass over the same data -- the tensor-scale reduction before quantizing
// the same tensor.
__device__ __forceinline__ uint64_t l2_policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// Read-only 16-byte global load, no L1 allocation, with an L2 policy.
__device__ __forceinline__ uint4 ld_global_nc_v4_policy(const void* p, uint64_t pol) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.v4.b32 {%0, %1, %2, %3}, [%4], %5;"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p), "l"(pol));
  return r;
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
