// Thread-block cluster helpers: rank, a full cluster barrier (or its two halves), and 4-byte
// loads from and stores to a peer CTA's shared memory (distributed shared memory).
#pragma once

#include <cstdint>

namespace cxa {

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// Every thread of every CTA of the cluster arrives and waits (release / acquire).
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// The two halves of cluster_sync, for work placed between them: arrive publishes this
// thread's earlier shared-memory writes (release); wait returns once every thread of
// the cluster has arrived and makes their writes visible (acquire).
__device__ __forceinline__ void cluster_arrive() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// The float at the same shared-memory offset as `local`, in cluster CTA `rank`.
__device__ __forceinline__ float ld_dsmem(const float* local, uint32_t rank) {
  uint32_t laddr = static_cast<uint32_t>(__cvta_generic_to_shared(local)), raddr;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(raddr) : "r"(laddr), "r"(rank));
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(raddr) : "memory");
  return v;
}

// Store v at the same shared-memory offset as `local`, in cluster CTA `rank`.
__device__ __forceinline__ void st_dsmem(float* local, uint32_t rank, float v) {
  uint32_t laddr = static_cast<uint32_t>(__cvta_generic_to_shared(local)), raddr;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(raddr) : "r"(laddr), "r"(rank));
  asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(raddr), "f"(v) : "memory");
}

}  // namespace cxa
