// Thread-block cluster primitives (sm_90 and later): a full cluster barrier
// and distributed shared memory, i.e. loads, stores and atomics on another
// block's shared memory.  The token-major kernels use them to let the blocks
// of a cluster share one scan of row_indices.
#pragma once

#include <cstdint>

namespace bsq {

// Every thread of every block of the cluster arrives; shared-memory writes
// before it are visible to the whole cluster after it.
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// The address of *p (this block's shared memory) in block `rank` of the cluster.
__device__ __forceinline__ uint32_t cluster_map(const void* p, int rank) {
  const uint32_t local = static_cast<uint32_t>(__cvta_generic_to_shared(p));
  uint32_t remote;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(local), "r"(rank));
  return remote;
}

__device__ __forceinline__ uint32_t cluster_ld_u32(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
  return v;
}

__device__ __forceinline__ void cluster_st_u32(uint32_t addr, uint32_t v) {
  asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}

// Returns the old value.
__device__ __forceinline__ uint32_t cluster_atomic_add_u32(uint32_t addr, uint32_t v) {
  uint32_t old;
  asm volatile("atom.shared::cluster.add.u32 %0, [%1], %2;" : "=r"(old) : "r"(addr), "r"(v) : "memory");
  return old;
}

}  // namespace bsq
