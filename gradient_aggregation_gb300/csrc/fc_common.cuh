// Device-side building blocks shared by the engine's kernels.
//
// Layout conventions:
//  * The fused vector has N elements; layer l occupies [off[l], off[l+1]).
//  * Chunks of `cs` elements split the fused vector (the last may be short).
//  * Reduction and norms work on units of at most FC_UNIT = 256 elements that
//    never straddle a chunk: chunk c owns units c*U .. with U = ceil(cs/256);
//    unit j of chunk c covers [c*cs + 256j, min(+256, c*cs+cs, N)).  One warp
//    handles one unit: lane t takes the 8-element groups [8g, 8g+8) (absolute
//    fused index, clipped to the unit) with g = floor(lo/8) + t + 32r.
//  * The sum of squares of a unit is the warp butterfly of the lanes' sums of
//    their groups (each group summed pairwise).  A chunk's sum of squares is
//    formed from its unit sums in float-float arithmetic in one fixed order:
//    lane t adds the units j = t, t+32, t+64, ... in turn, then a butterfly
//    over the 32 lanes (lane 0's result).  Every kernel that needs norms
//    follows this order, so the norms are bitwise identical across the fused
//    pipeline and the standalone calls.
//  * The update works on tiles of at most FC_TILE = 2048 elements that never
//    straddle a chunk (chunk c owns tiles c*P .. with P = ceil(cs/2048)).
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#define FC_TILE 2048
#define FC_UNIT 256
#define FC_BLOCK 256

namespace fc {

// Worker x layer pointer table, passed by value as a __grid_constant__
// kernel parameter (read from the constant bank, never copied).
template <int MAXP, int MAXL>
struct Table {
    int32_t W, L;
    int64_t off[MAXL + 1];               // fused offsets, off[L] = N
    uint32_t vec[(MAXL + 31) / 32];      // bit l: every worker's layer l is
                                         // 16-byte aligned at fused index 0 mod 8
    const __half *ptr[MAXP];             // ptr[w*L + l]
};
using TableS = Table<256, 64>;
using TableL = Table<3072, 512>;

struct TileGeom {
    int64_t N;   // elements
    int64_t cs;  // chunk size
    int64_t P;   // tiles per chunk
};

__device__ __forceinline__ bool tile_range(const TileGeom &G, int64_t t,
                                           int64_t &lo, int64_t &hi,
                                           int64_t &c, int64_t &hi_nominal)
{
    c = t / G.P;
    int64_t j = t - c * G.P;
    int64_t cend = c * G.cs + G.cs;
    lo = c * G.cs + j * FC_TILE;
    hi_nominal = lo + FC_TILE < cend ? lo + FC_TILE : cend;
    hi = hi_nominal < G.N ? hi_nominal : G.N;
    return lo < hi;
}

struct UnitGeom {
    int64_t N;      // elements
    int64_t cs;     // chunk size
    int64_t U;      // units per (full) chunk
    int64_t C;      // chunks
    int64_t units;  // total units: (C-1)*U + units of the last chunk
};

__device__ __forceinline__ void unit_range(const UnitGeom &G, int64_t u,
                                           int64_t &c, int64_t &lo,
                                           int64_t &hi)
{
    c = u / G.U;
    const int64_t j = u - c * G.U;
    const int64_t cend = c * G.cs + G.cs < G.N ? c * G.cs + G.cs : G.N;
    lo = c * G.cs + j * FC_UNIT;
    hi = lo + FC_UNIT < cend ? lo + FC_UNIT : cend;
}

// Number of units of chunk c.
__device__ __forceinline__ int64_t units_of_chunk(const UnitGeom &G, int64_t c)
{
    return c + 1 < G.C ? G.U : G.units - c * G.U;
}

// Smallest l with off[l+1] > f (skips empty layers).
template <class Tab>
__device__ __forceinline__ int find_layer(const Tab &t, int64_t f)
{
    int lo = 0, hi = t.L - 1;
    while (lo < hi) {
        int mid = (lo + hi) >> 1;
        if (t.off[mid + 1] > f)
            hi = mid;
        else
            lo = mid + 1;
    }
    return lo;
}

// ---- programmatic dependent launch ---------------------------------------------
//
// The selection and update kernels are launched with programmatic stream
// serialisation: the GPU may start them before the kernel ahead of them in
// the stream has finished, and their first action is to wait (in hardware,
// no polling) until that kernel has completed and its writes are visible.
// The kernel ahead signals early that its dependents may be scheduled.

__device__ __forceinline__ void wait_for_prior_grid()
{
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

__device__ __forceinline__ void allow_dependent_launch()
{
    asm volatile("griddepcontrol.launch_dependents;" :::);
}

// ---- cache-hinted memory access ---------------------------------------------

__device__ __forceinline__ uint64_t policy_evict_first()
{
    uint64_t p;
    asm("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// 16-byte streaming load of read-only data (the worker gradients).
__device__ __forceinline__ uint4 ld_stream16(const void *ptr, uint64_t pol)
{
    uint4 v;
    asm("ld.global.nc.L1::no_allocate.L2::cache_hint.v4.u32 {%0,%1,%2,%3}, [%4], %5;"
        : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
        : "l"(ptr), "l"(pol));
    return v;
}

__device__ __forceinline__ float ld_half_as_float(const __half *p)
{
    unsigned short b = __ldg(reinterpret_cast<const unsigned short *>(p));
    return __half2float(__ushort_as_half(b));
}

__device__ __forceinline__ void unpack8(const uint4 &q, float (&x)[8])
{
    const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        __half2 h = *reinterpret_cast<const __half2 *>(&w[i]);
        float2 f = __half22float2(h);
        x[2 * i] = f.x;
        x[2 * i + 1] = f.y;
    }
}

// 8 fp16 values starting `d` halves (0..7) into the 16 halves a:b.
__device__ __forceinline__ uint4 funnel8(const uint4 &a, const uint4 &b, int d)
{
    uint32_t w0 = a.x, w1 = a.y, w2 = a.z, w3 = a.w, w4 = b.x, w5 = b.y, w6 = b.z, w7 = b.w;
    if (d & 4) { w0 = w2; w1 = w3; w2 = w4; w3 = w5; w4 = w6; w5 = w7; }
    if (d & 2) { w0 = w1; w1 = w2; w2 = w3; w3 = w4; w4 = w5; }
    if (d & 1) {
        w0 = __funnelshift_r(w0, w1, 16);
        w1 = __funnelshift_r(w1, w2, 16);
        w2 = __funnelshift_r(w2, w3, 16);
        w3 = __funnelshift_r(w3, w4, 16);
    }
    return make_uint4(w0, w1, w2, w3);
}

// ---- the binary reduction tree over the workers ------------------------------
//
// Level-order adjacent pairing with an odd element carried up equals the
// binary-counter form used here: complete subtrees of 2^h leaves are merged
// into slot h as they arrive (older partial on the left), and the leftover
// slots are folded from the lowest height up at the end.  Leaves arrive in
// batches of 8 (one subtree of height 3) so that eight 16-byte loads are in
// flight at once; the W % 8 remainder arrives as subtrees of 4, 2 and 1.

template <int H0, int MAXH, int V>
__device__ __forceinline__ void tree_push(float (&acc)[MAXH][V], int cnt,
                                          float (&x)[V])
{
    bool carry = true;
#pragma unroll
    for (int h = H0; h < MAXH; ++h) {
        if (carry) {
            if ((cnt >> h) & 1) {
#pragma unroll
                for (int e = 0; e < V; ++e) x[e] = __fadd_rn(acc[h][e], x[e]);
            } else {
#pragma unroll
                for (int e = 0; e < V; ++e) acc[h][e] = x[e];
                carry = false;
            }
        }
    }
}

// Load(w, float (&x)[V]) fills the V values of worker w.
template <int WT, int MAXH, int V, class Load>
__device__ __forceinline__ void tree_sum(int Wrt, Load &&load, float (&out)[V])
{
    const int W = WT > 0 ? WT : Wrt;
    float acc[MAXH][V];
    int done = 0;
#pragma unroll
    for (; done + 8 <= W; done += 8) {
        float x[8][V];
#pragma unroll
        for (int u = 0; u < 8; ++u) load(done + u, x[u]);
#pragma unroll
        for (int e = 0; e < V; ++e) {
            float p0 = __fadd_rn(x[0][e], x[1][e]);
            float p1 = __fadd_rn(x[2][e], x[3][e]);
            float p2 = __fadd_rn(x[4][e], x[5][e]);
            float p3 = __fadd_rn(x[6][e], x[7][e]);
            x[0][e] = __fadd_rn(__fadd_rn(p0, p1), __fadd_rn(p2, p3));
        }
        tree_push<3>(acc, done, x[0]);
    }
    if (W - done >= 4) {
        float x[4][V];
#pragma unroll
        for (int u = 0; u < 4; ++u) load(done + u, x[u]);
#pragma unroll
        for (int e = 0; e < V; ++e)
            x[0][e] = __fadd_rn(__fadd_rn(x[0][e], x[1][e]),
                                __fadd_rn(x[2][e], x[3][e]));
        tree_push<2>(acc, done, x[0]);
        done += 4;
    }
    if (W - done >= 2) {
        float x[2][V];
        load(done, x[0]);
        load(done + 1, x[1]);
#pragma unroll
        for (int e = 0; e < V; ++e) x[0][e] = __fadd_rn(x[0][e], x[1][e]);
        tree_push<1>(acc, done, x[0]);
        done += 2;
    }
    if (W - done >= 1) {
        float x[V];
        load(done, x);
        tree_push<0>(acc, done, x);
        done += 1;
    }
    bool have = false;
#pragma unroll
    for (int h = 0; h < MAXH; ++h) {
        if ((W >> h) & 1) {
            if (!have) {
#pragma unroll
                for (int e = 0; e < V; ++e) out[e] = acc[h][e];
                have = true;
            } else {
#pragma unroll
                for (int e = 0; e < V; ++e) out[e] = __fadd_rn(acc[h][e], out[e]);
            }
        }
    }
}

// ---- other summation orders -------------------------------------------------------
//
// Left-to-right sum over the workers start, start+1, ..., start-1 (indices
// modulo W): the parameter-server order (start = 0) and the ring
// reduce-scatter order (start = the element's ring segment).  Loads are
// issued eight at a time; the additions stay in order.

__device__ __forceinline__ int ring_next(int w, int W) { return w + 1 == W ? 0 : w + 1; }

template <int V, class Load>
__device__ __forceinline__ void seq_sum(int W, int start, Load &&load,
                                        float (&out)[V])
{
    int w = start;
    load(w, out);
    w = ring_next(w, W);
    int t = 1;
    for (; t + 8 <= W; t += 8) {
        float x[8][V];
        int ws[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            ws[u] = w;
            w = ring_next(w, W);
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) load(ws[u], x[u]);
#pragma unroll
        for (int u = 0; u < 8; ++u)
#pragma unroll
            for (int e = 0; e < V; ++e) out[e] = __fadd_rn(out[e], x[u][e]);
    }
    for (; t < W; ++t) {
        float x[V];
        load(w, x);
#pragma unroll
        for (int e = 0; e < V; ++e) out[e] = __fadd_rn(out[e], x[e]);
        w = ring_next(w, W);
    }
}

// Ring segment of fused index f: the s in [0, W) with
// floor(s*N/W) <= f < floor((s+1)*N/W), i.e. floor(((f+1)*W - 1) / N).
__device__ __forceinline__ int ring_segment(int64_t f, int64_t N, int W)
{
    return (int)(((f + 1) * (int64_t)W - 1) / N);
}

// ---- sums of squares ------------------------------------------------------------

// Pairwise sum of squares of 8 values; v[e] must be 0 for masked elements.
__device__ __forceinline__ float group_sumsq(const float (&v)[8])
{
    float q[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) q[e] = __fmul_rn(v[e], v[e]);
    return __fadd_rn(__fadd_rn(__fadd_rn(q[0], q[1]), __fadd_rn(q[2], q[3])),
                     __fadd_rn(__fadd_rn(q[4], q[5]), __fadd_rn(q[6], q[7])));
}

// Butterfly sums over the 32 lanes: every lane ends with the same value.
__device__ __forceinline__ float warp_sum_f32(float x)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        x = __fadd_rn(x, __shfl_xor_sync(0xffffffffu, x, o));
    return x;
}

// Float-float (hi + lo) running sums: each addition keeps its exact rounding
// error (Knuth's two-sum) in lo, so a sum of n fp32 terms is exact to about
// n * 2^-48 relative, with fp32 instructions only (this GPU's fp64 rate is a
// small fraction of its fp32 rate).
struct FF {
    float hi, lo;
};

__device__ __forceinline__ FF ff_add(FF a, float x)
{
    const float s = __fadd_rn(a.hi, x);
    const float bb = __fsub_rn(s, a.hi);
    const float err = __fadd_rn(__fsub_rn(a.hi, __fsub_rn(s, bb)), __fsub_rn(x, bb));
    return FF{s, __fadd_rn(a.lo, err)};
}

__device__ __forceinline__ FF ff_add(FF a, FF b)
{
    FF r = ff_add(a, b.hi);
    r.lo = __fadd_rn(r.lo, b.lo);
    return r;
}

// Butterfly over the 32 lanes; lane 0's result is the defined one.
__device__ __forceinline__ FF warp_sum_ff(FF x)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        FF y;
        y.hi = __shfl_xor_sync(0xffffffffu, x.hi, o);
        y.lo = __shfl_xor_sync(0xffffffffu, x.lo, o);
        x = ff_add(x, y);
    }
    return x;
}

// Norm of a chunk from its float-float sum of squares: hi + lo rounded to
// fp32, then the correctly rounded fp32 square root.
__device__ __forceinline__ float norm_from_sumsq(FF ss)
{
    return __fsqrt_rn(__fadd_rn(ss.hi, ss.lo));
}

// Chunk norm from the unit sums, in the fixed order (see the top of this file):
// lane t adds units t, t+32, ... in float-float arithmetic, then the
// butterfly.  Called by a whole warp; the result is valid in lane 0.
// The unit sums are loaded eight per lane at a time, all eight loads in
// flight before the first addition, so a chunk of up to 256 units costs one
// memory round trip; the additions keep the order above.
__device__ __forceinline__ float chunk_norm_from_units(const UnitGeom &G,
                                                       const float *partials,
                                                       int64_t c, int lane)
{
    const int64_t Uc = units_of_chunk(G, c);
    const float *p = partials + c * G.U;
    FF ss = {0.f, 0.f};
    for (int64_t j0 = lane; j0 < Uc; j0 += 8 * 32) {
        float x[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            const int64_t j = j0 + 32 * q;
            x[q] = j < Uc ? __ldcg(p + j) : 0.f;
        }
#pragma unroll
        for (int q = 0; q < 8; ++q)
            if (j0 + 32 * q < Uc) ss = ff_add(ss, x[q]);
    }
    return norm_from_sumsq(warp_sum_ff(ss));
}

// ---- the update -------------------------------------------------------------------

// One element of a5: g = kept ? a : 0, r = kept ? 0 : a, v = mu*v + lr*g as
// two products and their sum, w = w - v; every operation one rounding.
__device__ __forceinline__ void sgd1(float a, bool kept, float lr, float mu,
                                     float &r, float &v, float &w)
{
    const float g = kept ? a : 0.f;
    r = kept ? 0.f : a;
    const float t1 = __fmul_rn(mu, v);
    const float t2 = __fmul_rn(lr, g);
    v = __fadd_rn(t1, t2);
    w = __fsub_rn(w, v);
}

}  // namespace fc
