// Phase 1 (a2 + unit sums of squares) with TMA staging, for 4, 8 or 16
// workers and layouts where every layer is 16-byte aligned for every worker
// and starts at a multiple of 8 elements, N is a multiple of 8 and the chunk
// size a multiple of 256.
//
// One CTA per SM: a producer warp streams tiles of TT fused elements of all
// W workers (and the residual) from HBM into a ring of S shared-memory stages
// with bulk copies (cp.async.bulk, completion counted on an mbarrier); eight
// consumer warps take one 256-element unit each per tile, add the workers in
// the same binary tree as the register kernel (k_reduce) from shared memory,
// and write `a` and the unit sums of squares exactly as k_reduce does, so the
// results are bit-identical.  The copies keep S-1 tiles of every worker in
// flight per SM regardless of register pressure.
//
// Every wait on an mbarrier gives up after a time limit (read from the
// global timer); the kernel then records the failure in `err` and returns,
// the producer first waiting (again with a limit) for the copies it issued.
#include <atomic>
#include <mutex>

#include "fc_internal.h"

namespace fc {

namespace {

__device__ __forceinline__ uint32_t smem_u32(const void *p)
{
    return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_test(uint32_t bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ uint64_t global_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Waits until the phase of the given parity has completed; false if that
// takes longer than limit_ns.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, uint64_t limit_ns)
{
    if (mbar_test(bar, parity)) return true;
    const uint64_t t0 = global_ns();
    while (!mbar_test(bar, parity))
        if (global_ns() - t0 > limit_ns) return false;
    return true;
}

__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void *src, uint32_t bytes,
                                         uint32_t bar)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
        "l"(src), "r"(bytes), "r"(bar)
        : "memory");
}

// Test hook (fc_test_stage_loss): a one-shot tile to drop and the wait limit
// that goes with it.
std::atomic<int64_t> g_drop_tile{-1};
std::atomic<uint64_t> g_drop_limit_ns{0};

constexpr int kConsumerWarps = 8;
constexpr int kThreads = 32 * (kConsumerWarps + 1);
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s: far beyond any tile

}  // namespace

// drop_tile >= 0 (test hook only, see fc_test_stage_loss): the producer
// issues no copies for that tile, so the bounded waits on it run out.
template <class Tab, int WT, int MAXH>
__global__ void __launch_bounds__(kThreads, 1)
    k_reduce_tma(const __grid_constant__ Tab tab, const UnitGeom G, const int TT,
                 const int S, const float u, const float *resid, float *out,
                 float *partials, unsigned *err, const int64_t drop_tile,
                 const uint64_t limit_ns)
{
    extern __shared__ __align__(128) unsigned char smem[];
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem);  // full[S], empty[S]
    unsigned char *stages = smem + 128;
    const int W = WT > 0 ? WT : tab.W;
    const int L = tab.L;
    const size_t gbytes = (size_t)W * TT * 2;
    const size_t sbytes = gbytes + (size_t)TT * 4;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t N = G.N;
    const int64_t ntiles = (N + TT - 1) / TT;

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(smem_u32(&bars[s]), 1);
            mbar_init(smem_u32(&bars[S + s]), kConsumerWarps);
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    // Launched after whatever the stream ran before (programmatic
    // serialisation): no global memory is touched before that work is done.
    wait_for_prior_grid();
    allow_dependent_launch();
    __syncthreads();

    if (warp == kConsumerWarps) {
        // producer
        if (lane != 0) return;
        int it = 0;
        for (int64_t t = blockIdx.x; t < ntiles; t += gridDim.x, ++it) {
            const int s = it % S;
            if (it >= S && !mbar_wait(smem_u32(&bars[S + s]), ((it / S) - 1) & 1, limit_ns)) {
                atomicOr(err, 1u);
                break;
            }
            if (t == drop_tile) continue;
            const int64_t f0 = t * TT;
            const int64_t f1 = f0 + TT < N ? f0 + TT : N;
            const uint32_t full = smem_u32(&bars[s]);
            mbar_expect_tx(full, (uint32_t)((f1 - f0) * (2 * W + (resid ? 4 : 0))));
            unsigned char *st = stages + (size_t)s * sbytes;
            int l = find_layer(tab, f0);
            for (int64_t fa = f0; fa < f1;) {
                while (tab.off[l + 1] <= fa) ++l;
                const int64_t fb = tab.off[l + 1] < f1 ? tab.off[l + 1] : f1;
                for (int w = 0; w < W; ++w)
                    bulk_g2s(smem_u32(st + ((size_t)w * TT + (size_t)(fa - f0)) * 2),
                             tab.ptr[w * L + l] + (fa - tab.off[l]), (uint32_t)((fb - fa) * 2), full);
                fa = fb;
            }
            if (resid) bulk_g2s(smem_u32(st + gbytes), resid + f0, (uint32_t)((f1 - f0) * 4), full);
        }
        // No copy may still be landing in shared memory when the CTA exits:
        // wait for every stage still in flight (each wait bounded; a stage
        // that gives up does not stop the waits for the others).
        for (int j = it > S ? it - S : 0; j < it; ++j)
            if (!mbar_wait(smem_u32(&bars[j % S]), (j / S) & 1, limit_ns))
                atomicOr(err, 2u);
        return;
    }

    // consumers
    int it = 0;
    for (int64_t t = blockIdx.x; t < ntiles; t += gridDim.x, ++it) {
        const int s = it % S;
        if (!mbar_wait(smem_u32(&bars[s]), (it / S) & 1, limit_ns)) {
            if (lane == 0) atomicOr(err, 4u);
            return;
        }
        const int64_t f0 = t * TT;
        const int64_t f1 = f0 + TT < N ? f0 + TT : N;
        const unsigned char *st = stages + (size_t)s * sbytes;
        for (int64_t lo = f0 + (int64_t)warp * FC_UNIT; lo < f1;
             lo += (int64_t)kConsumerWarps * FC_UNIT) {
            const int64_t hi = lo + FC_UNIT < f1 ? lo + FC_UNIT : f1;
            const int64_t f = lo + 8 * lane;
            float tss = 0.f;
            if (f < hi) {  // f + 8 <= hi: N and every unit start are multiples of 8
                const size_t off = (size_t)(f - f0);
                float a[8];
                tree_sum<WT, MAXH, 8>(
                    W,
                    [&](int w, float(&x)[8]) {
                        unpack8(*reinterpret_cast<const uint4 *>(st + ((size_t)w * TT + off) * 2), x);
                    },
                    a);
                float r[8];
                if (resid) {
                    const float4 *rr = reinterpret_cast<const float4 *>(st + gbytes + off * 4);
                    const float4 r0 = rr[0], r1 = rr[1];
                    r[0] = r0.x; r[1] = r0.y; r[2] = r0.z; r[3] = r0.w;
                    r[4] = r1.x; r[5] = r1.y; r[6] = r1.z; r[7] = r1.w;
                }
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    a[e] = __fmul_rn(a[e], u);
                    if (resid) a[e] = __fadd_rn(a[e], r[e]);
                }
                reinterpret_cast<float4 *>(out + f)[0] = make_float4(a[0], a[1], a[2], a[3]);
                reinterpret_cast<float4 *>(out + f)[1] = make_float4(a[4], a[5], a[6], a[7]);
                tss = __fadd_rn(tss, group_sumsq(a));
            }
            if (partials) {
                tss = warp_sum_f32(tss);
                if (lane == 0) partials[lo / FC_UNIT] = tss;
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&bars[S + s]));
    }
}

// Tile size and stage count for W workers: a stage holds W*TT fp16 values and
// TT fp32 residuals, about 64 KB of gradients, and as many stages as fit.
static void tma_shape(int W, int &TT, int &S, size_t &smem)
{
    TT = 2048;
    while (TT > FC_UNIT && (size_t)W * TT * 2 > 65536) TT /= 2;
    const size_t sbytes = (size_t)W * TT * 2 + (size_t)TT * 4;
    const size_t cap = 227 * 1024 - 128;
    S = (int)(cap / sbytes);
    if (S > 4) S = 4;
    smem = 128 + (size_t)S * sbytes;
}

template <class Tab>
bool tma_eligible(const Tab &tab, const UnitGeom &G, const float *partials)
{
    if (partials && G.cs % FC_UNIT != 0) return false;
    if (G.N % 8 != 0) return false;
    for (int l = 0; l < tab.L; ++l) {
        if (tab.off[l] % 8 != 0) return false;
        if (tab.off[l + 1] > tab.off[l] && !((tab.vec[l >> 5] >> (l & 31)) & 1u)) return false;
    }
    int TT, S;
    size_t smem;
    tma_shape(tab.W, TT, S, smem);
    return S >= 2;
}

template <class Tab, int WT, int MAXH>
static cudaError_t launch_tma_w(const Tab &tab, const UnitGeom &G, float u,
                                const float *resid, float *out, float *partials,
                                unsigned *err, cudaStream_t s)
{
    int TT, S;
    size_t smem;
    tma_shape(tab.W, TT, S, smem);
    auto kern = k_reduce_tma<Tab, WT, MAXH>;
    static std::mutex mu;
    static bool attr_set[64];
    int dev = 0;
    cudaGetDevice(&dev);
    {
        std::lock_guard<std::mutex> lock(mu);
        if (dev < 64 && !attr_set[dev]) {
            cudaError_t e = cudaFuncSetAttribute((const void *)kern,
                                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 227 * 1024);
            if (e != cudaSuccess) return e;
            attr_set[dev] = true;
        }
    }
    const int64_t tiles = (G.N + TT - 1) / TT;
    const int grid = grid_for((const void *)kern, kThreads, smem, tiles);
    const int64_t drop = g_drop_tile.exchange(-1);
    const uint64_t limit = drop >= 0 ? g_drop_limit_ns.load() : kWaitLimitNs;
    return launch_after_prior(kern, (unsigned)grid, kThreads, smem, s, tab, G, TT, S, u,
                              resid, out, partials, err, drop, limit);
}

template <class Tab>
cudaError_t launch_reduce_tma(const Tab &tab, const UnitGeom &G, float u,
                              const float *resid, float *out, float *partials,
                              unsigned *err, cudaStream_t s)
{
    switch (tab.W) {
    case 4: return launch_tma_w<Tab, 4, 3>(tab, G, u, resid, out, partials, err, s);
    case 8: return launch_tma_w<Tab, 8, 4>(tab, G, u, resid, out, partials, err, s);
    case 16: return launch_tma_w<Tab, 16, 5>(tab, G, u, resid, out, partials, err, s);
    default: break;
    }
    return cudaErrorNotSupported;
}

}  // namespace fc

extern "C" fc_status fc_test_stage_loss(int64_t tile, uint64_t wait_limit_ns)
{
    if (tile >= 0 && (wait_limit_ns < 1000000ull || wait_limit_ns > 2000000000ull))
        return fc::set_error(FC_ERR_INVALID_ARG, "wait_limit_ns must be in [1 ms, 2 s]");
    fc::g_drop_limit_ns.store(wait_limit_ns);
    fc::g_drop_tile.store(tile < 0 ? -1 : tile);
    return FC_OK;
}

namespace fc {

template bool tma_eligible<TableS>(const TableS &, const UnitGeom &, const float *);
template bool tma_eligible<TableL>(const TableL &, const UnitGeom &, const float *);
template cudaError_t launch_reduce_tma<TableS>(const TableS &, const UnitGeom &, float,
                                               const float *, float *, float *,
                                               unsigned *, cudaStream_t);
template cudaError_t launch_reduce_tma<TableL>(const TableL &, const UnitGeom &, float,
                                               const float *, float *, float *,
                                               unsigned *, cudaStream_t);

}  // namespace fc
