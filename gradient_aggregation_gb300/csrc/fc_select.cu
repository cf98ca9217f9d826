// a3 chunk norms and a4 top-k chunk selection + compaction.
//
// GradientFlow (arXiv 1902.06855), abstract: coarse-grained sparse
// communication sends only the important gradient chunks.  The pages do not
// define importance or how many chunks; the engine scores a chunk by its L2
// norm and keeps the k chunks that come first in (norm descending, index
// ascending) order.
//
// GB300 mapping:
//  * norms: one block per chunk walks the chunk's tiles with the same
//    thread/group mapping as the fused reduction kernel, so both produce the
//    same bits;
//  * select: C is at most a few thousand, so one 1024-thread block does a
//    3-pass radix select (11/11/10 bits) on the norms' bit patterns
//    (non-negative binary32 values order like their uint32 bits) with
//    shared-memory histograms, then two block scans in index order give the
//    tie-broken kept set, the ascending index list and each kept chunk's slot
//    in the packed output;
//  * gather: a grid-wide copy of the kept chunks into their slots.
#include "fc_internal.h"

namespace fc {

// ---- a3 ------------------------------------------------------------------------

__global__ void __launch_bounds__(FC_BLOCK)
    k_norms(const float *__restrict__ a, const TileGeom G, const int64_t C,
            float *__restrict__ norms)
{
    __shared__ float red8[FC_BLOCK / 32];
    for (int64_t c = blockIdx.x; c < C; c += gridDim.x) {
        double acc = 0.0;
        for (int64_t j = 0; j < G.P; ++j) {
            int64_t lo, hi, cc, hin;
            const bool any = tile_range(G, c * G.P + j, lo, hi, cc, hin);
            float tss = 0.f;
            if (any) {
                const int64_t g1 = (hi + 7) >> 3;
                for (int64_t g = (lo >> 3) + threadIdx.x; g < g1; g += FC_BLOCK) {
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
            }
            const double d = block_tile_sumsq(tss, red8);
            if (threadIdx.x == 0) acc = __dadd_rn(acc, d);
        }
        if (threadIdx.x == 0) norms[c] = norm_from_sumsq(acc);
    }
}

cudaError_t launch_norms(const float *a, const TileGeom &G, int64_t C,
                         float *norms, cudaStream_t s)
{
    const int grid = grid_for((const void *)k_norms, FC_BLOCK, 0, C);
    k_norms<<<grid, FC_BLOCK, 0, s>>>(a, G, C, norms);
    return cudaGetLastError();
}

// ---- a4 ------------------------------------------------------------------------

#define SEL_THREADS 1024
#define SEL_ITEMS 4

// Exclusive prefix sum over the 1024 threads; *total gets the block sum.
__device__ __forceinline__ uint32_t block_excl_scan(uint32_t x, uint32_t *sw,
                                                    uint32_t &total)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    uint32_t inc = x;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(0xffffffffu, inc, o);
        if (lane >= o) inc += y;
    }
    __syncthreads();  // sw may still be read by the previous scan
    if (lane == 31) sw[warp] = inc;
    __syncthreads();
    if (warp == 0) {
        uint32_t t = sw[lane];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t y = __shfl_up_sync(0xffffffffu, t, o);
            if (lane >= o) t += y;
        }
        sw[lane] = t;
    }
    __syncthreads();
    total = sw[31];
    return (warp ? sw[warp - 1] : 0u) + inc - x;
}

__global__ void __launch_bounds__(SEL_THREADS)
    k_select(const double *__restrict__ partials, const int64_t P,
             float *norms, const int64_t C, const int64_t k,
             int32_t *__restrict__ idx, uint8_t *__restrict__ mask,
             int32_t *__restrict__ slot, float *__restrict__ threshold)
{
    __shared__ uint32_t hist[2048];
    __shared__ uint32_t sw[32];
    __shared__ uint32_t s_digit, s_rem;
    const int tid = threadIdx.x;

    // finish the norms from the per-tile partial sums (same order as k_norms)
    if (partials) {
        for (int64_t c = tid; c < C; c += SEL_THREADS) {
            double ss = 0.0;
            for (int64_t j = 0; j < P; ++j) ss = __dadd_rn(ss, partials[c * P + j]);
            norms[c] = norm_from_sumsq(ss);
        }
        __syncthreads();
    }

    // radix select of the k-th largest key
    uint32_t prefix = 0, rem = (uint32_t)k;
#pragma unroll 1
    for (int pass = 0; pass < 3; ++pass) {
        const int shift = pass == 0 ? 21 : (pass == 1 ? 10 : 0);
        const int bits = pass == 2 ? 10 : 11;
        const int nb = 1 << bits;
        for (int b = tid; b < 2048; b += SEL_THREADS) hist[b] = 0;
        __syncthreads();
        for (int64_t c = tid; c < C; c += SEL_THREADS) {
            const uint32_t key = __float_as_uint(norms[c]);
            if (pass == 0 || (key >> (shift + bits)) == prefix)
                atomicAdd(&hist[(key >> shift) & (nb - 1)], 1u);
        }
        __syncthreads();
        const int per = nb / SEL_THREADS;  // 2 or 1 bins per thread, descending
        uint32_t local = 0;
        for (int i = 0; i < per; ++i) local += hist[nb - 1 - (per * tid + i)];
        uint32_t tot;
        uint32_t above = block_excl_scan(local, sw, tot);
        for (int i = 0; i < per; ++i) {
            const int b = nb - 1 - (per * tid + i);
            const uint32_t h = hist[b];
            if (above < rem && rem <= above + h) {
                s_digit = (uint32_t)b;
                s_rem = rem - above;
            }
            above += h;
        }
        __syncthreads();
        prefix = (prefix << bits) | s_digit;
        rem = s_rem;
        __syncthreads();
    }
    const uint32_t tau = prefix;  // bit pattern of the k-th largest norm
    const uint32_t need = rem;    // how many chunks equal to tau are kept

    // compaction in index order: ties kept from the lowest index up
    uint32_t eq_carry = 0, kept_carry = 0;
    for (int64_t base = 0; base < C; base += SEL_THREADS * SEL_ITEMS) {
        uint32_t key[SEL_ITEMS];
        bool valid[SEL_ITEMS], kept[SEL_ITEMS];
        uint32_t neq = 0;
#pragma unroll
        for (int i = 0; i < SEL_ITEMS; ++i) {
            const int64_t c = base + (int64_t)tid * SEL_ITEMS + i;
            valid[i] = c < C;
            key[i] = valid[i] ? __float_as_uint(norms[c]) : 0u;
            neq += (valid[i] && key[i] == tau) ? 1u : 0u;
        }
        uint32_t eq_tot;
        uint32_t eqr = block_excl_scan(neq, sw, eq_tot) + eq_carry;
        uint32_t nk = 0;
#pragma unroll
        for (int i = 0; i < SEL_ITEMS; ++i) {
            const bool eq = valid[i] && key[i] == tau;
            kept[i] = valid[i] && (key[i] > tau || (eq && eqr < need));
            eqr += eq ? 1u : 0u;
            nk += kept[i] ? 1u : 0u;
        }
        uint32_t k_tot;
        uint32_t pos = block_excl_scan(nk, sw, k_tot) + kept_carry;
#pragma unroll
        for (int i = 0; i < SEL_ITEMS; ++i) {
            const int64_t c = base + (int64_t)tid * SEL_ITEMS + i;
            if (!valid[i]) continue;
            mask[c] = kept[i] ? 1 : 0;
            if (slot) slot[c] = kept[i] ? (int32_t)pos : -1;
            if (kept[i]) {
                if (pos < (uint32_t)k) idx[pos] = (int32_t)c;  // always true
                ++pos;
            }
        }
        eq_carry += eq_tot;
        kept_carry += k_tot;
    }
    if (tid == 0) threshold[0] = __uint_as_float(tau);
}

cudaError_t launch_select(const double *partials, int64_t P, float *norms,
                          int64_t C, int64_t k, int32_t *idx, uint8_t *mask,
                          int32_t *slot, float *threshold, cudaStream_t s)
{
    k_select<<<1, SEL_THREADS, 0, s>>>(partials, P, norms, C, k, idx, mask,
                                       slot, threshold);
    return cudaGetLastError();
}

// ---- packed copy of the kept chunks ----------------------------------------------

__global__ void __launch_bounds__(FC_BLOCK)
    k_gather(const float *__restrict__ a, const int64_t N, const int64_t cs,
             const int64_t P, const int32_t *__restrict__ idx,
             const int64_t tiles, float *__restrict__ packed)
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
                __stcs(reinterpret_cast<float4 *>(packed + dst + e), x);
            }
        } else {
            for (int64_t e = e0 + threadIdx.x; e < e1; e += FC_BLOCK) {
                const int64_t i = src + e;
                packed[dst + e] = i < N ? __ldg(a + i) : 0.f;
            }
        }
    }
}

cudaError_t launch_gather(const float *a, int64_t N, int64_t cs, int64_t P,
                          const int32_t *idx, int64_t k, float *packed,
                          cudaStream_t s)
{
    const int64_t tiles = k * P;
    const int grid = grid_for((const void *)k_gather, FC_BLOCK, 0, tiles);
    k_gather<<<grid, FC_BLOCK, 0, s>>>(a, N, cs, P, idx, tiles, packed);
    return cudaGetLastError();
}

}  // namespace fc
