// Device helpers for thread-block clusters: rank and size, the hardware
// cluster barrier, stores into another CTA's shared memory, and the kept
// test of a selection given the k-th chunk.
#pragma once

#include <stdint.h>

namespace fc {

__device__ __forceinline__ uint32_t cluster_rank()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

__device__ __forceinline__ uint32_t cluster_size()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
    return r;
}

// Every thread of every CTA of the cluster arrives; memory operations
// before the barrier (shared, distributed shared and global) are visible to
// every thread of the cluster after it.
__device__ __forceinline__ void cluster_sync()
{
    asm volatile(
        "barrier.cluster.arrive.release.aligned;\n\t"
        "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Stores v at the address of `local` (a shared variable) in CTA `rank` of
// the cluster.
__device__ __forceinline__ void st_cluster_u32(const void *local, uint32_t rank, uint32_t v)
{
    const uint32_t a = (uint32_t)__cvta_generic_to_shared(local);
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(rank));
    asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(r), "r"(v) : "memory");
}

// Chunk c is kept iff it comes before the k-th chunk (tau, c_tau) in
// (key descending, index ascending) order, or is that chunk.
__device__ __forceinline__ bool is_kept(uint32_t key, int64_t c, uint32_t tau, int64_t ctau)
{
    return key > tau || (key == tau && c <= ctau);
}

}  // namespace fc
