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

__device__ __forceinline__ uint64_t ld_acquire_gpu_u64(const unsigned long long *p)
{
    uint64_t v;
    asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}

// Barrier over all n CTAs of a cooperative launch on a 64-bit arrival count
// that only grows (zero in a fresh workspace).  Each completed launch adds
// n per barrier, so between launches the count is a multiple of n, and
// *s_base, read by thread 0 at launch start and rounded down to a multiple
// of n, is the count before this launch even if other CTAs have already
// arrived.  At barrier k (1, 2, ...) thread 0 of each CTA adds one with a
// release reduction (no return value to wait for) and waits, at most
// limit_ns, until the count reaches *s_base + k n.  Returns false, in every
// thread of the CTA, if that wait ran out (a launch that gave up leaves the
// count off its multiple of n, so the workspace must be zeroed again).
__device__ __forceinline__ bool grid_arrive_wait(unsigned long long *count, const uint64_t *s_base,
                                                 unsigned k, uint64_t limit_ns,
                                                 volatile uint32_t *s_ok)
{
    __syncthreads();
    if (threadIdx.x == 0) {
        const uint64_t target = *s_base + (uint64_t)k * gridDim.x;
        asm volatile("red.release.gpu.global.add.u64 [%0], 1;" ::"l"(count) : "memory");
        bool ok = ld_acquire_gpu_u64(count) >= target;
        if (!ok) {
            const uint64_t t0 = globaltimer_ns();
            while (!(ok = ld_acquire_gpu_u64(count) >= target))
                if (globaltimer_ns() - t0 > limit_ns) break;
        }
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
