// Device helpers for the one-launch steps: thread-block cluster rank and
// size, the hardware cluster barrier, stores into another CTA's shared
// memory, a bounded barrier over the CTAs of a cooperative launch, and the
// kept test of a selection given the k-th chunk.
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

__device__ __forceinline__ uint32_t ld_acquire_gpu(const unsigned *p)
{
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ uint64_t globaltimer_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ uint32_t atom_add_acq_rel_gpu(unsigned *p, uint32_t v)
{
    uint32_t old;
    asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v)
                 : "memory");
    return old;
}

__device__ __forceinline__ void st_release_gpu(unsigned *p, uint32_t v)
{
    asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ void st_relaxed_gpu(unsigned *p, uint32_t v)
{
    asm volatile("st.relaxed.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Waits (one thread) until *p == v, at most limit_ns; false if it ran out.
__device__ __forceinline__ bool wait_equal_gpu(const unsigned *p, uint32_t v, uint64_t limit_ns)
{
    if (ld_acquire_gpu(p) == v) return true;
    const uint64_t t0 = globaltimer_ns();
    while (ld_acquire_gpu(p) != v)
        if (globaltimer_ns() - t0 > limit_ns) return false;
    return true;
}

// Barrier over all nblocks CTAs of a cooperative launch (every CTA resident
// at once), on two words in global memory: bar[0] counts arrivals (zero
// between barriers), bar[1] is the generation.  Thread 0 of each CTA reads
// the generation g and arrives with an acquire-release add, which also
// publishes the CTA's writes (ordered before it by the CTA barrier); the
// last CTA to arrive clears the count and releases generation g + 1, for
// which the others wait, at most limit_ns.  Returns false, in every thread
// of the CTA, if that wait ran out (the caller then gives up the step);
// *gen_out is g + 1.
__device__ __forceinline__ bool grid_sync(unsigned *bar, unsigned nblocks, uint64_t limit_ns,
                                          volatile uint32_t *s_ok, volatile uint32_t *s_gen)
{
    __syncthreads();
    if (threadIdx.x == 0) {
        const unsigned g = ld_acquire_gpu(bar + 1);
        bool ok = true;
        if (atom_add_acq_rel_gpu(bar, 1u) == nblocks - 1) {
            st_relaxed_gpu(bar, 0u);
            st_release_gpu(bar + 1, g + 1u);
        } else {
            ok = wait_equal_gpu(bar + 1, g + 1u, limit_ns);
        }
        *s_gen = g + 1u;
        *s_ok = ok ? 1u : 0u;
    }
    __syncthreads();
    return *s_ok != 0u;
}

// Chunk c is kept iff it comes before the k-th chunk (tau, c_tau) in
// (key descending, index ascending) order, or is that chunk.
__device__ __forceinline__ bool is_kept(uint32_t key, int64_t c, uint32_t tau, int64_t ctau)
{
    return key > tau || (key == tau && c <= ctau);
}

}  // namespace fc
