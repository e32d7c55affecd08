// Rank-2 -> 5D TCGEN scale reinterleave (a pure byte permutation).
//
// Thread block (band, chunk) stages 128 rows x (4 * kIlvAtoms) scale bytes in
// shared memory (zero outside M x S), then writes the chunk's atoms, which are
// contiguous in the 5D buffer, as 16-byte stores: store j of an atom holds the
// 4 bytes of rows j, j+32, j+64, j+96.  The staging rows are padded to 68
// bytes so that the transposed 4-byte reads hit 32 distinct banks.
#pragma once

#include "device_common.cuh"

namespace bsq {

constexpr int kIlvAtoms = 16;                 // atoms (4 scale columns each) per block
constexpr int kIlvCols = 4 * kIlvAtoms;       // 64 scale bytes per row
constexpr int kIlvPitch = kIlvCols + 4;       // padded staging row (bytes)
constexpr int kIlvThreads = 128;

// VEC: bytes per staging load (16, 4 or 1); the launcher picks the widest one
// that the base address, ld and S allow.
template <int VEC>
__global__ void __launch_bounds__(kIlvThreads)
    interleave_kernel(const uint8_t* __restrict__ in, int64_t M, int64_t S, int64_t ld,
                      uint8_t* __restrict__ out, int kt_atoms) {
  __shared__ __align__(16) uint8_t tile[128 * kIlvPitch];
  const int64_t m0 = static_cast<int64_t>(blockIdx.x) * 128;
  const int a0 = blockIdx.y * kIlvAtoms;
  const int64_t s0 = static_cast<int64_t>(a0) * 4;
  // the block's rows into L2 while the previous kernel finishes (L2 is the
  // point of coherence: a later read after the wait still sees its writes)
  for (int r = threadIdx.x; r < 128; r += kIlvThreads)
    if (m0 + r < M && s0 < S) prefetch_l2(in + (m0 + r) * ld + s0);
  pdl_wait();
  pdl_trigger();

  if constexpr (VEC > 1) {
    // every load of the thread is issued before the first shared-memory store
    constexpr int kPerRow = kIlvCols / VEC;
    constexpr int kN = 128 * kPerRow / kIlvThreads;
    uint32_t val[kN][VEC / 4];
#pragma unroll
    for (int j = 0; j < kN; ++j) {
      const int idx = threadIdx.x + j * kIlvThreads;
      const int r = idx / kPerRow, w = idx % kPerRow;
      const int64_t m = m0 + r, s = s0 + VEC * w;
      const bool in_range = m < M && s < S;
      if constexpr (VEC == 16) {
        uint4 x = make_uint4(0u, 0u, 0u, 0u);
        if (in_range) x = __ldg(reinterpret_cast<const uint4*>(in + m * ld + s));
        val[j][0] = x.x; val[j][1] = x.y; val[j][2] = x.z; val[j][3] = x.w;
      } else {
        val[j][0] = in_range ? __ldg(reinterpret_cast<const uint32_t*>(in + m * ld + s)) : 0u;
      }
    }
#pragma unroll
    for (int j = 0; j < kN; ++j) {
      const int idx = threadIdx.x + j * kIlvThreads;
      const int r = idx / kPerRow, w = idx % kPerRow;
#pragma unroll
      for (int k = 0; k < VEC / 4; ++k)
        *reinterpret_cast<uint32_t*>(tile + r * kIlvPitch + VEC * w + 4 * k) = val[j][k];
    }
  } else {
    constexpr int kB = 16;
    for (int base = 0; base < 128 * kIlvCols; base += kB * kIlvThreads) {
      uint8_t val[kB];
#pragma unroll
      for (int j = 0; j < kB; ++j) {
        const int idx = base + threadIdx.x + j * kIlvThreads;
        const int r = idx / kIlvCols, c = idx % kIlvCols;
        const int64_t m = m0 + r, s = s0 + c;
        val[j] = (m < M && s < S) ? __ldg(in + m * ld + s) : uint8_t(0);
      }
#pragma unroll
      for (int j = 0; j < kB; ++j) {
        const int idx = base + threadIdx.x + j * kIlvThreads;
        tile[(idx / kIlvCols) * kIlvPitch + idx % kIlvCols] = val[j];
      }
    }
  }
  __syncthreads();

  const int natoms = min(kIlvAtoms, kt_atoms - a0);
  uint8_t* dst = out + (static_cast<int64_t>(blockIdx.x) * kt_atoms + a0) * 512;
  for (int idx = threadIdx.x; idx < natoms * 32; idx += kIlvThreads) {
    const int atom = idx >> 5, r32 = idx & 31;
    const uint8_t* src = tile + r32 * kIlvPitch + atom * 4;
    st_global_v4(dst + atom * 512 + r32 * 16,
                 *reinterpret_cast<const uint32_t*>(src),
                 *reinterpret_cast<const uint32_t*>(src + 32 * kIlvPitch),
                 *reinterpret_cast<const uint32_t*>(src + 64 * kIlvPitch),
                 *reinterpret_cast<const uint32_t*>(src + 96 * kIlvPitch));
  }
}

}  // namespace bsq
