// fc_step in one launch for small problems (a few hundred thousand
// elements), instead of three kernels.  The three-kernel pipeline pays
// three launches and two full-device hand-offs per step, which bounds a
// 133K-element step at 17 us whatever the kernels do.
//
// Two kernels share the same per-unit code (below) and so give the same
// bits as the three kernels (the GPU tests compare all of them and the
// oracle):
//  * k_step_grid: one cooperative launch, one CTA per SM, with one grid
//    barrier on a workspace arrival count after the norms and the k-th
//    chunk handed to every CTA through one tag word (both waits bounded);
//  * k_step_small: one thread-block cluster (16 CTAs where the GPU allows,
//    else 8) with hardware cluster barriers and distributed shared memory,
//    for devices that run no cooperative launch.
// Both run the same four steps:
//  1. reduce: each warp takes 256-element units with the tree, unscale and
//     residual of the register kernel (`k_reduce`), and writes `a` and the
//     unit sums of squares;
//  2. norms: chunk norms from the unit sums in the fixed float-float order
//     of the selection kernel (at once, by the reducing warp, when a chunk
//     is a single unit);
//  3. select: every chunk's rank in (norm descending, index ascending)
//     order is counted against all C keys, which each CTA holds; the chunk
//     of rank k-1 gives the threshold tau and its index c_tau to every CTA.
//     Chunk c is kept iff key_c > tau, or key_c == tau and c <= c_tau:
//     exactly the k chunks first in that order, the same set the radix
//     select of the pipeline finds;
//  4. update: each warp updates its own units again (re-reading the `a` it
//     wrote), with each kept chunk's send-buffer slot counted from the keys
//     (kept chunks before it), exactly as the update kernel does.
#include <atomic>
#include <mutex>

#include "fc_cluster.cuh"
#include "fc_internal.h"

namespace fc {

struct SmallArgs {
    UnitGeom G;
    float u;
    const float *resid;
    float *a;
    float *partials;
    float *norms;
    int64_t k;
    int32_t *idx;
    uint8_t *mask;
    float *threshold;
    unsigned *status;
    float lr, mu;
    float *r, *v, *w;
    __half *w16;
    float *packed;
    __half *packed16;
    float send_scale;
    int inplace;
    unsigned *bar;      // grid kernel: 64-bit arrival count (words 0-1), tau, c_tau, tau's tag
    uint64_t limit_ns;  // grid kernel: longest wait at a barrier
    int drop_cta;       // grid kernel, test hook: this CTA skips its first barrier (-1: none)
};

// ---- per-unit work shared by the cluster and the grid kernels ----------------

// a2 on one 256-element unit [lo, hi) by a whole warp (lane: elements
// lo + 8*lane ..+8) with the register kernel's arithmetic (chunk sizes are
// multiples of 8, so a unit has at most 32 groups of 8); writes `a` and
// returns the unit's sum of squares (every lane).
template <class Tab, int WT, int MAXH>
__device__ __forceinline__ float reduce_unit(const Tab &tab, const SmallArgs &A, int64_t lo,
                                             int64_t hi, int lane)
{
    const int W = WT > 0 ? WT : tab.W;
    const int L = tab.L;
    const int64_t f0 = lo + 8 * (int64_t)lane;
    float tss = 0.f;
    if (f0 < hi) {
        float a[8];
        int l = find_layer(tab, f0);
        if (f0 + 8 <= hi && f0 + 8 <= tab.off[l + 1] && ((tab.vec[l >> 5] >> (l & 31)) & 1u)) {
            const int64_t j = f0 - tab.off[l];
            tree_sum<WT, MAXH, 8>(
                W,
                [&](int wk, float(&x)[8]) {
                    unpack8(__ldg(reinterpret_cast<const uint4 *>(tab.ptr[wk * L + l] + j)), x);
                },
                a);
            float r[8];
            if (A.resid) {
                const float4 r0 = __ldcs(reinterpret_cast<const float4 *>(A.resid + f0));
                const float4 r1 = __ldcs(reinterpret_cast<const float4 *>(A.resid + f0 + 4));
                r[0] = r0.x; r[1] = r0.y; r[2] = r0.z; r[3] = r0.w;
                r[4] = r1.x; r[5] = r1.y; r[6] = r1.z; r[7] = r1.w;
            }
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                a[e] = __fmul_rn(a[e], A.u);
                if (A.resid) a[e] = __fadd_rn(a[e], r[e]);
            }
            reinterpret_cast<float4 *>(A.a + f0)[0] = make_float4(a[0], a[1], a[2], a[3]);
            reinterpret_cast<float4 *>(A.a + f0)[1] = make_float4(a[4], a[5], a[6], a[7]);
        } else {
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const int64_t f = f0 + e;
                if (f >= hi) {
                    a[e] = 0.f;
                    continue;
                }
                while (tab.off[l + 1] <= f) ++l;
                const int64_t j = f - tab.off[l];
                float s1[1];
                tree_sum<WT, MAXH, 1>(
                    W,
                    [&](int wk, float(&x)[1]) {
                        x[0] = ld_half_as_float(tab.ptr[wk * L + l] + j);
                    },
                    s1);
                float val = __fmul_rn(s1[0], A.u);
                if (A.resid) val = __fadd_rn(val, __ldcs(A.resid + f));
                A.a[f] = val;
                a[e] = val;
            }
        }
        tss = __fadd_rn(tss, group_sumsq(a));
    }
    return warp_sum_f32(tss);
}

// The norm of a chunk that is a single unit, from that unit's sum of squares
// (lane 0's) with the selection kernel's float-float butterfly, so the bits
// are those of the pipeline; the key (bit pattern) in every lane.
__device__ __forceinline__ uint32_t single_unit_key(float tss, int lane, float &n)
{
    FF ss = {0.f, 0.f};
    if (lane == 0) ss = ff_add(ss, tss);
    n = norm_from_sumsq(warp_sum_ff(ss));
    return __shfl_sync(0xffffffffu, __float_as_uint(n), 0);
}

// Norms of chunks c0, c0 + nw, ... (warp gw = c0 of nw) from the unit sums,
// up to four chunks' sums in flight before the first addition; the additions
// follow the fixed order (lane t: units t, t+32, ... in float-float, then
// the butterfly).  put(c, key) is called by every lane.
template <class Put>
__device__ __forceinline__ void chunk_norms_from_units(const SmallArgs &A, int64_t gw, int64_t nw,
                                                       int lane, Put &&put)
{
    const UnitGeom &G = A.G;
    const int64_t C = G.C;
    for (int64_t c0 = gw; c0 < C; c0 += 4 * nw) {
        float x[4][8];
        int64_t Uc[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int64_t c = c0 + q * nw;
            Uc[q] = c < C ? units_of_chunk(G, c) : 0;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int64_t jj = lane + 32 * i;
                x[q][i] = jj < Uc[q] ? __ldcg(A.partials + c * G.U + jj) : 0.f;
            }
        }
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int64_t c = c0 + q * nw;
            if (c >= C) break;
            float n;
            if (Uc[q] <= 256) {
                FF ss = {0.f, 0.f};
#pragma unroll
                for (int i = 0; i < 8; ++i)
                    if (lane + 32 * i < Uc[q]) ss = ff_add(ss, x[q][i]);
                n = norm_from_sumsq(warp_sum_ff(ss));
            } else {
                n = chunk_norm_from_units(G, A.partials, c, lane);
            }
            const uint32_t key = __shfl_sync(0xffffffffu, __float_as_uint(n), 0);
            if (lane == 0) A.norms[c] = n;
            put(c, key);
        }
    }
}

// The kept chunks as a bitmask (s_kept) and the kept chunks before each
// 32-chunk word (s_before), from the keys in shared memory; a whole CTA.
template <int NT>
__device__ __forceinline__ void kept_words(const uint32_t *skeys, int64_t C, uint32_t tau,
                                           int64_t ctau, uint32_t *s_kept, uint32_t *s_before)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int64_t nwords = (C + 31) / 32;
    for (int64_t wd = warp; wd < nwords; wd += NT / 32) {
        const int64_t c = 32 * wd + lane;
        const uint32_t bits = __ballot_sync(0xffffffffu, c < C && is_kept(skeys[c], c, tau, ctau));
        if (lane == 0) s_kept[wd] = bits;
    }
    __syncthreads();
    if (warp == 0) {
        const uint32_t cnt = lane < nwords ? (uint32_t)__popc(s_kept[lane]) : 0u;
        uint32_t inc = cnt;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t y = __shfl_up_sync(0xffffffffu, inc, o);
            if (lane >= o) inc += y;
        }
        if (lane < nwords) s_before[lane] = inc - cnt;
    }
    __syncthreads();
}

// a5 on unit un [lo, hi) of chunk c by a whole warp, re-reading the `a` the
// same lane wrote in reduce_unit; also the chunk's mask and idx entries (by
// the warp of its first unit) and its send-buffer slot.
__device__ __forceinline__ void update_unit(const SmallArgs &A, int64_t c, int64_t lo, int64_t hi,
                                            int lane, const uint32_t *s_kept,
                                            const uint32_t *s_before)
{
    const int64_t cs = A.G.cs;
    const uint32_t word = s_kept[c >> 5];
    const bool kept = (word >> (c & 31)) & 1u;
    // slot of chunk c in the send buffers: kept chunks before it
    const uint32_t slot = s_before[c >> 5] + (uint32_t)__popc(word & ((1u << (c & 31)) - 1u));
    if (lo == c * cs && lane == 0) {
        A.mask[c] = kept ? 1 : 0;
        if (kept) A.idx[slot] = (int32_t)c;
    }
    const bool pk = kept && (A.packed != nullptr || A.packed16 != nullptr);
    const int64_t pbase = pk ? (int64_t)slot * cs - c * cs : 0;
    const bool need_a = kept || !A.inplace;
    const int64_t f0 = lo + 8 * (int64_t)lane;
    if (f0 < hi) {
        if (f0 + 8 <= hi) {
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int64_t i0 = f0 + 4 * h;
                float4 av = make_float4(0.f, 0.f, 0.f, 0.f);
                if (need_a) av = *reinterpret_cast<const float4 *>(A.a + i0);  // this thread's own step-1 writes
                float4 vv = *reinterpret_cast<const float4 *>(A.v + i0);
                float4 ww = *reinterpret_cast<const float4 *>(A.w + i0);
                float4 rr;
                sgd1(av.x, kept, A.lr, A.mu, rr.x, vv.x, ww.x);
                sgd1(av.y, kept, A.lr, A.mu, rr.y, vv.y, ww.y);
                sgd1(av.z, kept, A.lr, A.mu, rr.z, vv.z, ww.z);
                sgd1(av.w, kept, A.lr, A.mu, rr.w, vv.w, ww.w);
                __stcs(reinterpret_cast<float4 *>(A.v + i0), vv);
                __stcs(reinterpret_cast<float4 *>(A.w + i0), ww);
                if (need_a) __stcs(reinterpret_cast<float4 *>(A.r + i0), rr);
                if (A.w16) {
                    __half2 h0 = __floats2half2_rn(ww.x, ww.y);
                    __half2 h1 = __floats2half2_rn(ww.z, ww.w);
                    uint2 hv;
                    hv.x = *reinterpret_cast<uint32_t *>(&h0);
                    hv.y = *reinterpret_cast<uint32_t *>(&h1);
                    __stcs(reinterpret_cast<uint2 *>(A.w16 + i0), hv);
                }
                if (pk && A.packed) __stcs(reinterpret_cast<float4 *>(A.packed + pbase + i0), av);
                if (pk && A.packed16) {
                    const __half2 s0 = __floats2half2_rn(__fmul_rn(av.x, A.send_scale),
                                                         __fmul_rn(av.y, A.send_scale));
                    const __half2 s1 = __floats2half2_rn(__fmul_rn(av.z, A.send_scale),
                                                         __fmul_rn(av.w, A.send_scale));
                    uint2 hv;
                    hv.x = *reinterpret_cast<const uint32_t *>(&s0);
                    hv.y = *reinterpret_cast<const uint32_t *>(&s1);
                    __stcs(reinterpret_cast<uint2 *>(A.packed16 + pbase + i0), hv);
                }
            }
        } else {
            for (int64_t i = f0; i < hi; ++i) {
                const float ai = need_a ? A.a[i] : 0.f;
                float vi = A.v[i], wi = A.w[i], ri;
                sgd1(ai, kept, A.lr, A.mu, ri, vi, wi);
                A.v[i] = vi;
                A.w[i] = wi;
                if (need_a) A.r[i] = ri;
                if (A.w16) A.w16[i] = __float2half_rn(wi);
                if (pk && A.packed) A.packed[pbase + i] = ai;
                if (pk && A.packed16)
                    A.packed16[pbase + i] = __float2half_rn(__fmul_rn(ai, A.send_scale));
            }
        }
    }
    // the short last chunk: zero its send-buffer slot past N
    if (pk && hi == A.G.N) {
        for (int64_t i = A.G.N + lane; i < c * cs + cs; i += 32) {
            if (A.packed) A.packed[pbase + i] = 0.f;
            if (A.packed16) A.packed16[pbase + i] = __float2half_rn(0.f);
        }
    }
}

// ---- the cluster kernel ---------------------------------------------------------

// NT threads per CTA: 1024 for up to 4 workers (the tree then fits in 64
// registers a thread), else 512.
template <class Tab, int WT, int MAXH, int NT>
__global__ void __launch_bounds__(NT, 1)
    k_step_small(const __grid_constant__ Tab tab, const SmallArgs A)
{
    constexpr int kSmallWarps = NT / 32;
    // the chunks' keys (norm bit patterns), padded with zeros to a multiple
    // of 4; the k-th chunk; the kept chunks as a bitmask and the number of
    // kept chunks before each 32-chunk word
    __shared__ __align__(16) uint32_t skeys[FC_SMALL_MAX_CHUNKS + 4];
    __shared__ uint32_t s_tau, s_ctau;
    __shared__ uint32_t s_kept[FC_SMALL_MAX_CHUNKS / 32], s_before[FC_SMALL_MAX_CHUNKS / 32];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const uint32_t crank = cluster_rank(), ncta = cluster_size();
    const int64_t gw = (int64_t)crank * kSmallWarps + warp;
    const int64_t nw = (int64_t)ncta * kSmallWarps;
    const UnitGeom &G = A.G;
    const int64_t C = G.C;
    // Every CTA of the cluster must be running before any writes to another
    // one's shared memory: arrive now, wait once the work ahead in the
    // stream is done (by then every CTA has arrived).
    asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
    // Launched after whatever the stream ran before (programmatic
    // serialisation): no global memory is touched before that work is done.
    wait_for_prior_grid();
    allow_dependent_launch();
    asm volatile("barrier.cluster.wait.aligned;" ::: "memory");
    if (threadIdx.x < 4) skeys[C + threadIdx.x] = 0u;

    // ---- 1. reduce.  With one unit per chunk (chunks of at most 256
    // elements) the warp that reduced a unit also finishes its chunk's norm
    // at once.
    for (int64_t un = gw; un < G.units; un += nw) {
        int64_t c, lo, hi;
        unit_range(G, un, c, lo, hi);
        const float tss = reduce_unit<Tab, WT, MAXH>(tab, A, lo, hi, lane);
        if (lane == 0) A.partials[un] = tss;
        if (G.U == 1) {
            float n;
            const uint32_t key = single_unit_key(tss, lane, n);
            if (lane == 0) A.norms[c] = n;
            if ((uint32_t)lane < ncta) st_cluster_u32(&skeys[c], (uint32_t)lane, key);
        }
    }

    // ---- 2. norms, and every norm's key into every CTA's shared memory
    if (G.U > 1) {
        cluster_sync();
        chunk_norms_from_units(A, gw, nw, lane, [&](int64_t c, uint32_t key) {
            if ((uint32_t)lane < ncta) st_cluster_u32(&skeys[c], (uint32_t)lane, key);
        });
    }
    cluster_sync();

    // ---- 3. select: the chunk of rank k-1.  Warp gw ranks chunks gw,
    // gw + nw, ...: lane t counts the chunks j = t, t+32, ... before it in
    // (key descending, index ascending) order.
    for (int64_t c = gw; c < C; c += nw) {
        const uint32_t kc = skeys[c];
        uint32_t above = 0;
        for (int64_t j = lane; j < C; j += 32) {
            const uint32_t kj = skeys[j];
            above += (kj > kc || (kj == kc && j < c)) ? 1u : 0u;
        }
        above = __reduce_add_sync(0xffffffffu, above);
        if ((int64_t)above == A.k - 1) {
            if ((uint32_t)lane < ncta) {
                st_cluster_u32(&s_tau, (uint32_t)lane, kc);
                st_cluster_u32(&s_ctau, (uint32_t)lane, (uint32_t)c);
            }
            if (lane == 0) {
                A.threshold[0] = __uint_as_float(kc);
                if (A.status) *A.status = 0u;  // the step is applied
            }
        }
    }
    cluster_sync();

    // ---- 4. update, unit by unit as in step 1
    kept_words<NT>(skeys, C, s_tau, (int64_t)s_ctau, s_kept, s_before);
    for (int64_t un = gw; un < G.units; un += nw) {
        int64_t c, lo, hi;
        unit_range(G, un, c, lo, hi);
        update_unit(A, c, lo, hi, lane, s_kept, s_before);
    }
}

// ---- the grid kernel ------------------------------------------------------------
//
// The same step over every SM: one cooperative launch (all CTAs resident at
// once) with a grid barrier after the norms (two when a chunk has several
// units) on an arrival count in the workspace (grid_arrive_wait).  The warp
// that finds the chunk of rank k-1 then publishes it (tau, c_tau) with a
// release store of a tag, the count this launch's last barrier waited for,
// and every CTA waits for that word alone instead of a second barrier.  Units and chunks are dealt to warps across the CTAs (warp index
// gw = warp * CTAs + CTA), so a small problem's units spread over all SMs.
// A barrier wait that runs out (only possible if the GPU stalls for
// limit_ns) ends every CTA that sees it without writing v, w or the
// outputs, and marks the step as not applied.
template <class Tab, int WT, int MAXH, int NT>
__global__ void __launch_bounds__(NT, 1)
    k_step_grid(const __grid_constant__ Tab tab, const SmallArgs A)
{
    constexpr int kWarps = NT / 32;
    __shared__ __align__(16) uint32_t skeys[FC_SMALL_MAX_CHUNKS + 4];
    __shared__ uint32_t s_kept[FC_SMALL_MAX_CHUNKS / 32], s_before[FC_SMALL_MAX_CHUNKS / 32];
    __shared__ uint32_t s_ok, s_tau, s_ctau;
    __shared__ uint64_t s_base;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int64_t gw = (int64_t)warp * gridDim.x + blockIdx.x;
    const int64_t nw = (int64_t)gridDim.x * kWarps;
    const UnitGeom &G = A.G;
    const int64_t C = G.C;
    auto give_up = [&]() {
        if (threadIdx.x == 0 && blockIdx.x == 0 && A.status) *A.status = 1u;
    };
    // Launched after whatever the stream ran before (programmatic
    // serialisation): no global memory is touched before that work is done.
    unsigned long long *count = reinterpret_cast<unsigned long long *>(A.bar);
    wait_for_prior_grid();
    allow_dependent_launch();
    // the barrier's arrival count before this launch (see grid_arrive_wait)
    if (threadIdx.x == 0) {
        const uint64_t c = ld_acquire_gpu_u64(count);
        s_base = c - c % gridDim.x;
    }

    // ---- 1. reduce (and, with one unit per chunk, the chunk's norm)
    for (int64_t un = gw; un < G.units; un += nw) {
        int64_t c, lo, hi;
        unit_range(G, un, c, lo, hi);
        const float tss = reduce_unit<Tab, WT, MAXH>(tab, A, lo, hi, lane);
        if (lane == 0) A.partials[un] = tss;
        if (G.U == 1) {
            float n;
            (void)single_unit_key(tss, lane, n);
            if (lane == 0) A.norms[c] = n;
        }
    }
    // test hook: this CTA never arrives, so the others' waits run out
    if ((int)blockIdx.x == A.drop_cta) return give_up();
    // ---- 2. norms of chunks of several units
    unsigned barriers = 1;
    if (G.U > 1) {
        if (!grid_arrive_wait(count, &s_base, barriers++, A.limit_ns, &s_ok)) return give_up();
        chunk_norms_from_units(A, gw, nw, lane, [](int64_t, uint32_t) {});
    }
    if (!grid_arrive_wait(count, &s_base, barriers, A.limit_ns, &s_ok)) return give_up();
    // this launch's last barrier count: differs from every earlier launch's
    const uint32_t tag = (uint32_t)(s_base + (uint64_t)barriers * gridDim.x);

    // every CTA takes all keys
    for (int64_t c = threadIdx.x; c < C; c += NT) skeys[c] = __float_as_uint(__ldcg(A.norms + c));
    if (threadIdx.x < 4) skeys[C + threadIdx.x] = 0u;
    __syncthreads();

    // ---- 3. warp gw ranks chunks gw, gw + nw, ... (lane t counts the chunks
    // j = t, t+32, ... before it in (key descending, index ascending) order);
    // the chunk of rank k-1 publishes itself.
    for (int64_t c = gw; c < C; c += nw) {
        const uint32_t kc = skeys[c];
        uint32_t above = 0;
        for (int64_t j = lane; j < C; j += 32) {
            const uint32_t kj = skeys[j];
            above += (kj > kc || (kj == kc && j < c)) ? 1u : 0u;
        }
        above = __reduce_add_sync(0xffffffffu, above);
        if ((int64_t)above == A.k - 1 && lane == 0) {
            A.threshold[0] = __uint_as_float(kc);
            if (A.status) *A.status = 0u;  // the step is applied
            st_relaxed_gpu(A.bar + 2, kc);
            st_relaxed_gpu(A.bar + 3, (uint32_t)c);
            st_release_gpu(A.bar + 4, tag);
        }
    }
    // wait for the k-th chunk (a word no earlier launch left at this tag)
    if (threadIdx.x == 0) {
        s_ok = wait_equal_gpu(A.bar + 4, tag, A.limit_ns) ? 1u : 0u;
        s_tau = ld_acquire_gpu(A.bar + 2);
        s_ctau = ld_acquire_gpu(A.bar + 3);
    }
    __syncthreads();
    if (!s_ok) return give_up();

    // ---- 4. update, unit by unit as in step 1
    kept_words<NT>(skeys, C, s_tau, (int64_t)s_ctau, s_kept, s_before);
    for (int64_t un = gw; un < G.units; un += nw) {
        int64_t c, lo, hi;
        unit_range(G, un, c, lo, hi);
        update_unit(A, c, lo, hi, lane, s_kept, s_before);
    }
}

namespace {

// Cluster size per (kernel, device): 16 CTAs where the GPU schedules such a
// cluster of this kernel, else 8, else 0 (one-launch path unavailable).
int cluster_ctas(const void *kern, int dev, int threads)
{
    struct Entry {
        const void *kern;
        int dev, ctas;
    };
    static std::mutex mu;
    static Entry cache[64];
    static int used = 0;
    std::lock_guard<std::mutex> lock(mu);
    for (int i = 0; i < used; ++i)
        if (cache[i].kern == kern && cache[i].dev == dev) return cache[i].ctas;
    int ctas = 0;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) !=
        cudaSuccess)
        (void)cudaGetLastError();
    for (int n : {16, 8}) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(n);
        cfg.blockDim = dim3(threads);
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = n;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        int clusters = 0;
        if (cudaOccupancyMaxActiveClusters(&clusters, kern, &cfg) == cudaSuccess && clusters >= 1) {
            ctas = n;
            break;
        }
        (void)cudaGetLastError();
    }
    if (used < 64) cache[used++] = Entry{kern, dev, ctas};
    return ctas;
}

// CTAs of the grid kernel per device: one per SM when the device runs
// cooperative launches and one CTA of the kernel fits on an SM, else 0.
int grid_ctas(const void *kern, int dev, int threads)
{
    struct Entry {
        const void *kern;
        int dev, ctas;
    };
    static std::mutex mu;
    static Entry cache[64];
    static int used = 0;
    std::lock_guard<std::mutex> lock(mu);
    for (int i = 0; i < used; ++i)
        if (cache[i].kern == kern && cache[i].dev == dev) return cache[i].ctas;
    int coop = 0, sms = 0, per_sm = 0;
    cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, threads, 0) != cudaSuccess)
        per_sm = 0;
    (void)cudaGetLastError();
    const int ctas = coop && per_sm >= 1 ? sms : 0;
    if (used < 64) cache[used++] = Entry{kern, dev, ctas};
    return ctas;
}

// Longest wait at a grid barrier before the step is given up: far beyond
// any step this kernel runs (a few microseconds).
constexpr uint64_t kGridWaitNs = 2000000000ull;

// Test hooks: force the cluster kernel (fc_test_one_launch_kind), and a
// one-shot CTA that skips the grid kernel's first barrier with the wait
// limit that goes with it (fc_test_barrier_loss).
std::atomic<int> g_force_cluster{0};
std::atomic<int> g_drop_cta{-1};
std::atomic<uint64_t> g_drop_cta_limit_ns{0};

template <class Tab, int WT, int MAXH>
cudaError_t launch_small_w(const Tab &tab, const SmallArgs &args_in, cudaStream_t s,
                           bool probe_only, int *kind)
{
    SmallArgs args = args_in;
    // the whole GPU, when the device allows a cooperative launch of it
    if (args.bar && !g_force_cluster.load()) {
        constexpr int NTG = (WT > 0 && WT <= 16) ? 512 : 256;
        auto kg = k_step_grid<Tab, WT, MAXH, NTG>;
        int dev = 0;
        cudaGetDevice(&dev);
        const int ctas = grid_ctas((const void *)kg, dev, NTG);
        const int64_t max_units = (int64_t)ctas * (NTG / 32) * FC_SMALL_UNITS_PER_WARP;
        if (ctas > 0 && args.G.units <= max_units) {
            *kind = FC_STEP_ONE_LAUNCH;
            if (probe_only) return cudaSuccess;
            const int drop = g_drop_cta.exchange(-1);
            if (drop >= 0) {
                args.drop_cta = drop < ctas ? drop : ctas - 1;
                args.limit_ns = g_drop_cta_limit_ns.load();
            }
            cudaLaunchConfig_t cfg = {};
            cfg.gridDim = dim3(ctas);
            cfg.blockDim = dim3(NTG);
            cfg.stream = s;
            cudaLaunchAttribute attr[2];
            attr[0].id = cudaLaunchAttributeCooperative;
            attr[0].val.cooperative = 1;
            attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
            attr[1].val.programmaticStreamSerializationAllowed = 1;
            cfg.attrs = attr;
            cfg.numAttrs = 2;
            return cudaLaunchKernelEx(&cfg, kg, tab, args);
        }
    }
    // else one thread-block cluster
    constexpr int NT = (WT > 0 && WT <= 4) ? 1024 : 512;
    constexpr int kSmallWarps = NT / 32;
    auto kern = k_step_small<Tab, WT, MAXH, NT>;
    int dev = 0;
    cudaGetDevice(&dev);
    const int ctas = cluster_ctas((const void *)kern, dev, NT);
    // units are taken one per warp and round
    const int64_t max_units = (int64_t)ctas * kSmallWarps * FC_SMALL_UNITS_PER_WARP;
    if (ctas <= 0 || args.G.units > max_units) return cudaSuccess;
    *kind = FC_STEP_ONE_CLUSTER;
    if (probe_only) return cudaSuccess;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(ctas);
    cfg.blockDim = dim3(NT);
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = ctas;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, kern, tab, args);
}

}  // namespace

template <class Tab>
cudaError_t launch_step_small(const Tab &tab, const SmallStep &st, cudaStream_t s,
                              bool probe_only, int *kind)
{
    *kind = FC_STEP_THREE_KERNELS;
    const UnitGeom &G = st.G;
    if (G.cs % 8 != 0 || G.C > FC_SMALL_MAX_CHUNKS || G.N > FC_SMALL_MAX_N || tab.W > 64)
        return cudaSuccess;
    SmallArgs A;
    A.G = G;
    A.u = st.u;
    A.resid = st.resid;
    A.a = st.a;
    A.partials = st.partials;
    A.norms = st.norms;
    A.k = st.k;
    A.idx = st.idx;
    A.mask = st.mask;
    A.threshold = st.threshold;
    A.status = st.status;
    A.lr = st.lr;
    A.mu = st.mu;
    A.r = st.r;
    A.v = st.v;
    A.w = st.w;
    A.w16 = st.w16;
    A.packed = st.packed;
    A.packed16 = st.packed16;
    A.send_scale = st.send_scale;
    A.inplace = st.a == st.r ? 1 : 0;
    A.bar = st.bar;
    A.limit_ns = kGridWaitNs;
    A.drop_cta = -1;
#define FC_S(WT, MAXH) launch_small_w<Tab, WT, MAXH>(tab, A, s, probe_only, kind)
    switch (tab.W) {
    case 1: return FC_S(1, 1);
    case 2: return FC_S(2, 2);
    case 4: return FC_S(4, 3);
    case 8: return FC_S(8, 4);
    case 16: return FC_S(16, 5);
    case 32: return FC_S(32, 6);
    case 64: return FC_S(64, 7);
    default: break;
    }
    if (tab.W < 32) return FC_S(0, 5);
    return FC_S(0, 7);
#undef FC_S
}

template cudaError_t launch_step_small<TableS>(const TableS &, const SmallStep &, cudaStream_t,
                                               bool, int *);
template cudaError_t launch_step_small<TableL>(const TableL &, const SmallStep &, cudaStream_t,
                                               bool, int *);

}  // namespace fc

extern "C" fc_status fc_test_one_launch_kind(int32_t kind)
{
    if (kind != FC_STEP_ONE_LAUNCH && kind != FC_STEP_ONE_CLUSTER)
        return fc::set_error(FC_ERR_INVALID_ARG, "kind must be FC_STEP_ONE_LAUNCH or FC_STEP_ONE_CLUSTER");
    fc::g_force_cluster.store(kind == FC_STEP_ONE_CLUSTER ? 1 : 0);
    return FC_OK;
}

extern "C" fc_status fc_test_barrier_loss(int32_t cta, uint64_t wait_limit_ns)
{
    if (cta >= 0 && (wait_limit_ns == 0 || wait_limit_ns > 10000000000ull))
        return fc::set_error(FC_ERR_INVALID_ARG, "wait_limit_ns must be in (0, 10 s]");
    fc::g_drop_cta_limit_ns.store(wait_limit_ns);
    fc::g_drop_cta.store(cta < 0 ? -1 : cta);
    return FC_OK;
}
