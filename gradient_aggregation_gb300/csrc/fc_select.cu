// a3 chunk norms and a4 top-k chunk selection + compaction.
//
// GradientFlow (arXiv 1902.06855), abstract: coarse-grained sparse
// communication sends only the chunks that matter.  The pages do not
// define importance or how many chunks; the engine scores a chunk by its L2
// norm and keeps the k chunks that come first in (norm descending, index
// ascending) order.
//
// GB300 mapping:
//  * norms: one block per chunk forms the chunk's unit sums with the same
//    warp/lane mapping and the same float-float order as the fused reduction
//    kernel, so both produce the same bits;
//  * select: in the pipeline, blocks of 32 warps first turn the reduction's
//    unit sums into chunk norms (one warp per chunk, the fixed float-float
//    order); the last block to finish then selects.  C is at most a few
//    thousand, so one 1024-thread block holds the norms in shared memory and
//    runs a 4-pass radix select (8 bits a pass) on their bit patterns, then
//    one block scan in index order gives the tie-broken kept set, the
//    ascending index list and each kept chunk's slot in the packed output;
//  * gather: a grid-wide copy of the kept chunks into their slots (fp32
//    and/or fp16 send buffers).
#include "fc_internal.h"

namespace fc {

// ---- a3 ------------------------------------------------------------------------

// One block of 8 warps per chunk.  Warp w forms the sums of the units
// j = w, w+8, w+16, ... of the chunk exactly as the reduction kernels do, and
// keeps four float-float running sums, one per residue class j mod 32 it
// sees (w, w+8, w+16, w+24), added in increasing j.  Those 32 class sums then
// go through the same butterfly as the selection kernel's chunk finish, so
// both produce the same bits.
__global__ void __launch_bounds__(FC_BLOCK)
    k_norms(const float *__restrict__ a, const UnitGeom G,
            float *__restrict__ norms)
{
    __shared__ float res_hi[32], res_lo[32];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    for (int64_t c = blockIdx.x; c < G.C; c += gridDim.x) {
        const int64_t Uc = units_of_chunk(G, c);
        FF acc[4] = {{0.f, 0.f}, {0.f, 0.f}, {0.f, 0.f}, {0.f, 0.f}};
        for (int64_t base = 0; base < Uc; base += 32) {
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int64_t j = base + warp + 8 * q;
                if (j >= Uc) continue;
                int64_t cc, lo, hi;
                unit_range(G, c * G.U + j, cc, lo, hi);
                float tss = 0.f;
                const int64_t g1 = (hi + 7) >> 3;
                for (int64_t g = (lo >> 3) + lane; g < g1; g += 32) {
                    const int64_t f0 = g << 3;
                    float v[8];
                    if (f0 >= lo && f0 + 8 <= hi) {
                        const float4 x0 = __ldg(reinterpret_cast<const float4 *>(a + f0));
                        const float4 x1 = __ldg(reinterpret_cast<const float4 *>(a + f0 + 4));
                        v[0] = x0.x; v[1] = x0.y; v[2] = x0.z; v[3] = x0.w;
                        v[4] = x1.x; v[5] = x1.y; v[6] = x1.z; v[7] = x1.w;
                    } else {
#pragma unroll
                        for (int e = 0; e < 8; ++e) {
                            const int64_t f = f0 + e;
                            v[e] = (f >= lo && f < hi) ? __ldg(a + f) : 0.f;
                        }
                    }
                    tss = __fadd_rn(tss, group_sumsq(v));
                }
                tss = warp_sum_f32(tss);
                acc[q] = ff_add(acc[q], tss);
            }
        }
        if (lane == 0) {
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                res_hi[warp + 8 * q] = acc[q].hi;
                res_lo[warp + 8 * q] = acc[q].lo;
            }
        }
        __syncthreads();
        if (warp == 0) {
            const FF ss = warp_sum_ff(FF{res_hi[lane], res_lo[lane]});
            if (lane == 0) norms[c] = norm_from_sumsq(ss);
        }
        __syncthreads();
    }
}

cudaError_t launch_norms(const float *a, const UnitGeom &G, float *norms,
                         cudaStream_t s)
{
    const int grid = grid_for((const void *)k_norms, FC_BLOCK, 0, G.C);
    k_norms<<<grid, FC_BLOCK, 0, s>>>(a, G, norms);
    return cudaGetLastError();
}

// ---- a4 ------------------------------------------------------------------------

#define SEL_THREADS 1024
#define SEL_ITEMS 4
#define SEL_SMEM_KEYS 11264

// Exclusive prefix sum over the 1024 threads; `total` gets the block sum.
__device__ __forceinline__ uint64_t block_excl_scan64(uint64_t x, uint64_t *sw,
                                                      uint64_t &total)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    uint64_t inc = x;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint64_t y = __shfl_up_sync(0xffffffffu, inc, o);
        if (lane >= o) inc += y;
    }
    __syncthreads();  // sw may still be read by the previous scan
    if (lane == 31) sw[warp] = inc;
    __syncthreads();
    if (warp == 0) {
        uint64_t t = sw[lane];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint64_t y = __shfl_up_sync(0xffffffffu, t, o);
            if (lane >= o) t += y;
        }
        sw[lane] = t;
    }
    __syncthreads();
    total = sw[31];
    return (warp ? sw[warp - 1] : 0ull) + inc - x;
}

// Selection kernel.  With partials != NULL every block first turns the unit
// sums of 32 chunks (one per warp) into norms; the block that finishes last
// (a count of finished blocks in `done`, reset by that block) then runs the
// selection.  With partials == NULL there is one block and the norms are an
// input.  No block ever waits for another.
//
// Selection: the norms' bit patterns (non-negative binary32 values order like
// their uint32 patterns) go to shared memory; four radix passes of 8 bits
// find the pattern tau of the k-th largest norm and how many chunks equal to
// tau are kept (`need`: the lowest-indexed ones); one block scan in index
// order then places every kept chunk: its slot is the number of kept chunks
// before it = (#greater before it) + min(#equal before it, need).
__global__ void __launch_bounds__(SEL_THREADS)
    k_select(const UnitGeom G, const float *__restrict__ partials,
             unsigned *__restrict__ done, float *norms, const int64_t k,
             int32_t *__restrict__ idx, uint8_t *__restrict__ mask,
             int32_t *__restrict__ slot, float *__restrict__ threshold,
             unsigned *__restrict__ err, unsigned *__restrict__ status)
{
    __shared__ uint32_t skeys[SEL_SMEM_KEYS];
    __shared__ uint32_t hist[3][256];
    __shared__ uint64_t sw[32];
    __shared__ uint32_t s_last, s_dr[2];
    const int tid = threadIdx.x;
    const int64_t C = G.C;
    wait_for_prior_grid();
    allow_dependent_launch();

    if (partials) {
        const int lane = tid & 31, warp = tid >> 5;
        for (int64_t c = (int64_t)blockIdx.x * 32 + warp; c < C;
             c += (int64_t)gridDim.x * 32) {
            const float n = chunk_norm_from_units(G, partials, c, lane);
            if (lane == 0) norms[c] = n;
        }
        // Publish this block's norms before counting it: the barrier orders
        // every warp's writes before thread 0's count, whose release makes
        // them visible device-wide with it; its acquire makes every earlier
        // block's norms visible to the block that counts last.
        __syncthreads();
        if (tid == 0) {
            unsigned seen;
            asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], 1;"
                         : "=r"(seen)
                         : "l"(done)
                         : "memory");
            s_last = seen == gridDim.x - 1 ? 1u : 0u;
            if (s_last) *done = 0u;  // ready for the next call
        }
        __syncthreads();
        if (!s_last) return;
        // A wait inside the staged reduction gave up (not expected to
        // happen): report it as a NaN threshold with nothing kept, and mark
        // the step as not applied, so that the update leaves the state alone.
        const bool failed = err && __ldcg(err) != 0u;
        if (tid == 0 && status) *status = failed ? 1u : 0u;
        if (failed) {
            for (int64_t c = tid; c < C; c += SEL_THREADS) {
                mask[c] = 0;
                if (slot) slot[c] = -1;
            }
            for (int64_t q = tid; q < k; q += SEL_THREADS) idx[q] = -1;
            __syncthreads();
            if (tid == 0) {
                threshold[0] = __int_as_float(0x7fc00000);
                *err = 0u;
            }
            return;
        }
    }

    const bool in_smem = C <= SEL_SMEM_KEYS;
    if (in_smem) {
        // all of a thread's loads in flight before its first store
        constexpr int R = (SEL_SMEM_KEYS + SEL_THREADS - 1) / SEL_THREADS;
        uint32_t v[R];
#pragma unroll
        for (int i = 0; i < R; ++i) {
            const int64_t c = tid + (int64_t)i * SEL_THREADS;
            v[i] = c < C ? __float_as_uint(__ldcg(norms + c)) : 0u;
        }
#pragma unroll
        for (int i = 0; i < R; ++i) {
            const int64_t c = tid + (int64_t)i * SEL_THREADS;
            if (c < C) skeys[c] = v[i];
        }
        __syncthreads();
    }
    auto key_at = [&](int64_t c) -> uint32_t {
        return in_smem ? skeys[c] : __float_as_uint(__ldcg(norms + c));
    };

    const int lane = tid & 31;
    if (k == C) {
        // Every chunk is kept: the threshold is the smallest norm, and chunk
        // c goes to slot c.  (The radix select and the scan below would give
        // the same outputs.)
        uint32_t lo = 0xffffffffu;
        for (int64_t c = tid; c < C; c += SEL_THREADS) {
            lo = min(lo, key_at(c));
            mask[c] = 1;
            if (slot) slot[c] = (int32_t)c;
            idx[c] = (int32_t)c;
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) lo = min(lo, __shfl_xor_sync(0xffffffffu, lo, o));
        if (lane == 0) hist[0][tid >> 5] = lo;
        __syncthreads();
        if (tid < 32) {
            lo = hist[0][tid];
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) lo = min(lo, __shfl_xor_sync(0xffffffffu, lo, o));
            if (tid == 0) threshold[0] = __uint_as_float(lo);
        }
        return;
    }

    // Radix passes.  Pass p counts into hist[p % 3] while the threads below
    // 256 clear hist[(p + 1) % 3] for the next pass (last read by the scan of
    // pass p - 2, finished before that pass's second barrier), so a pass
    // needs two barriers: after the counts, and after warp 0 has found the
    // digit.
    if (tid < 256) hist[0][tid] = 0;
    __syncthreads();
    uint32_t prefix = 0, rem = (uint32_t)k;
#pragma unroll 1
    for (int pass = 0; pass < 4; ++pass) {
        const int shift = 24 - 8 * pass;
        uint32_t *h = hist[pass % 3];
        if (tid < 256) hist[(pass + 1) % 3][tid] = 0;
        // Norms of similar size share their top bits, so many lanes hit the
        // same bin: lanes with equal digits are counted once per warp.
        for (int64_t base = tid & ~31; base < C; base += SEL_THREADS) {
            const int64_t c = base + lane;
            const uint32_t key = c < C ? key_at(c) : 0u;
            const bool in = c < C && (pass == 0 || (key >> (shift + 8)) == prefix);
            const uint32_t digit = in ? (key >> shift) & 255u : 256u;
            const uint32_t peers = __match_any_sync(0xffffffffu, digit);
            if (in && lane == __ffs(peers) - 1)
                atomicAdd(&h[digit], (uint32_t)__popc(peers));
        }
        __syncthreads();
        if (tid < 32) {
            uint32_t hv[8], local = 0;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                hv[i] = h[255 - 8 * lane - i];
                local += hv[i];
            }
            uint32_t inc = local;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const uint32_t y = __shfl_up_sync(0xffffffffu, inc, o);
                if (lane >= o) inc += y;
            }
            uint32_t above = inc - local;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                if (above < rem && rem <= above + hv[i]) {
                    s_dr[0] = (uint32_t)(255 - 8 * lane - i);
                    s_dr[1] = rem - above;
                }
                above += hv[i];
            }
        }
        __syncthreads();
        prefix = (prefix << 8) | s_dr[0];
        rem = s_dr[1];
    }
    const uint32_t tau = prefix;  // bit pattern of the k-th largest norm
    const uint32_t need = rem;    // chunks equal to tau that are kept

    uint32_t gt_carry = 0, eq_carry = 0;
    for (int64_t base = 0; base < C; base += SEL_THREADS * SEL_ITEMS) {
        uint32_t key[SEL_ITEMS];
        uint32_t ngt = 0, neq = 0;
#pragma unroll
        for (int i = 0; i < SEL_ITEMS; ++i) {
            const int64_t c = base + (int64_t)tid * SEL_ITEMS + i;
            key[i] = c < C ? key_at(c) : 0u;
            if (c < C) {
                ngt += key[i] > tau ? 1u : 0u;
                neq += key[i] == tau ? 1u : 0u;
            }
        }
        uint64_t tot;
        const uint64_t ex = block_excl_scan64(((uint64_t)neq << 32) | ngt, sw, tot);
        uint32_t gtb = (uint32_t)ex + gt_carry;
        uint32_t eqb = (uint32_t)(ex >> 32) + eq_carry;
#pragma unroll
        for (int i = 0; i < SEL_ITEMS; ++i) {
            const int64_t c = base + (int64_t)tid * SEL_ITEMS + i;
            if (c >= C) break;
            const bool gt = key[i] > tau, eq = key[i] == tau;
            const bool kept = gt || (eq && eqb < need);
            const uint32_t pos = gtb + (eqb < need ? eqb : need);
            mask[c] = kept ? 1 : 0;
            if (slot) slot[c] = kept ? (int32_t)pos : -1;
            if (kept && pos < (uint32_t)k) idx[pos] = (int32_t)c;
            gtb += gt ? 1u : 0u;
            eqb += eq ? 1u : 0u;
        }
        gt_carry += (uint32_t)tot;
        eq_carry += (uint32_t)(tot >> 32);
    }
    if (tid == 0) threshold[0] = __uint_as_float(tau);
}

cudaError_t launch_select(const UnitGeom &G, const float *partials,
                          unsigned *done, float *norms, int64_t k,
                          int32_t *idx, uint8_t *mask, int32_t *slot,
                          float *threshold, cudaStream_t s, unsigned *err,
                          unsigned *status)
{
    int64_t blocks = 1;
    if (partials) {
        blocks = (G.C + 31) / 32;
        const int cap = grid_for((const void *)k_select, SEL_THREADS, 0, blocks);
        if (blocks > cap) blocks = cap;  // all blocks resident: no queueing
    }
    return launch_after_prior(k_select, (unsigned)blocks, SEL_THREADS, 0, s, G,
                              partials, done, norms, k, idx, mask, slot, threshold,
                              err, status);
}

// ---- packed copy of the kept chunks ----------------------------------------------

__global__ void __launch_bounds__(FC_BLOCK)
    k_gather(const float *__restrict__ a, const int64_t N, const int64_t cs,
             const int64_t P, const int32_t *__restrict__ idx,
             const int64_t tiles, float *__restrict__ packed,
             __half *__restrict__ packed16, const float send_scale)
{
    const bool vec = (cs & 3) == 0;
    for (int64_t t = blockIdx.x; t < tiles; t += gridDim.x) {
        const int64_t q = t / P, j = t - q * P;
        const int64_t c = idx[q];
        const int64_t e0 = j * FC_TILE;
        const int64_t e1 = e0 + FC_TILE < cs ? e0 + FC_TILE : cs;
        const int64_t src = c * cs, dst = q * cs;
        if (vec) {
            for (int64_t e = e0 + 4 * (int64_t)threadIdx.x; e < e1; e += 4 * FC_BLOCK) {
                const int64_t i = src + e;
                float4 x;
                if (i + 4 <= N) {
                    x = __ldg(reinterpret_cast<const float4 *>(a + i));
                } else {
                    x.x = i < N ? a[i] : 0.f;
                    x.y = i + 1 < N ? a[i + 1] : 0.f;
                    x.z = i + 2 < N ? a[i + 2] : 0.f;
                    x.w = i + 3 < N ? a[i + 3] : 0.f;
                }
                if (packed) __stcs(reinterpret_cast<float4 *>(packed + dst + e), x);
                if (packed16) {
                    const __half2 s0 = __floats2half2_rn(__fmul_rn(x.x, send_scale),
                                                         __fmul_rn(x.y, send_scale));
                    const __half2 s1 = __floats2half2_rn(__fmul_rn(x.z, send_scale),
                                                         __fmul_rn(x.w, send_scale));
                    uint2 hv;
                    hv.x = *reinterpret_cast<const uint32_t *>(&s0);
                    hv.y = *reinterpret_cast<const uint32_t *>(&s1);
                    __stcs(reinterpret_cast<uint2 *>(packed16 + dst + e), hv);
                }
            }
        } else {
            for (int64_t e = e0 + threadIdx.x; e < e1; e += FC_BLOCK) {
                const int64_t i = src + e;
                const float x = i < N ? __ldg(a + i) : 0.f;
                if (packed) packed[dst + e] = x;
                if (packed16) packed16[dst + e] = __float2half_rn(__fmul_rn(x, send_scale));
            }
        }
    }
}

cudaError_t launch_gather(const float *a, int64_t N, int64_t cs, int64_t P,
                          const int32_t *idx, int64_t k, float *packed,
                          __half *packed16, float send_scale, cudaStream_t s)
{
    const int64_t tiles = k * P;
    const int grid = grid_for((const void *)k_gather, FC_BLOCK, 0, tiles);
    k_gather<<<grid, FC_BLOCK, 0, s>>>(a, N, cs, P, idx, tiles, packed, packed16,
                                       send_scale);
    return cudaGetLastError();
}

}  // namespace fc
