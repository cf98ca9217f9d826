// a1 + a2 (+ the partial sums of a3): fuse and tree-reduce the workers'
// gradients.
//
// FireCaffe (arXiv 1511.00175), §6: the workers' gradient vectors are summed
// element-wise, through a binary reduction tree whose depth is the base-2
// log of the worker count.  GradientFlow (arXiv 1902.06855), abstract: mixed precision
// (fp16 gradients, fp32 sums here) and lazy allreduce, which fuses the
// per-layer operations into one; here the fusion is a layout (offsets) that
// the reduction reads through, so the fused copy need not be materialised.
//
// GB300 mapping: one pass over HBM, each element of each worker read exactly
// once with 16-byte streaming loads (L1 bypass, L2 evict-first); eight
// workers' loads in flight per thread before their subtree is formed in
// registers; fp32 results written once; the chunk sums of squares formed from
// the registers, so the norms cost no extra pass.
#include "fc_internal.h"

namespace fc {

// ---- a2 kernel ------------------------------------------------------------------
//
// One warp per unit of 256 fused elements (see fc_common.cuh), no block-wide
// synchronisation and no fences, so every warp streams independently.  With
// `partials` given, the warp also writes the unit's sum of squares, which
// the selection kernel turns into chunk norms.

// Resident blocks per SM the register allocation aims at for W <= 16.
#ifndef FC_REDUCE_MIN_BLOCKS_SMALL_W
#define FC_REDUCE_MIN_BLOCKS_SMALL_W 3
#endif

// ORDER: 0 the binary tree, 1 parameter server (workers in index order),
// 2 ring reduce-scatter (see fc_common.cuh).
template <class Tab, int WT, int MAXH, int ORDER>
__global__ void __launch_bounds__(FC_BLOCK, (WT == 0 && MAXH > 7) ? 1
                                            : ((WT > 0 && WT <= 16) ? FC_REDUCE_MIN_BLOCKS_SMALL_W : 2))
    k_reduce(const __grid_constant__ Tab tab, const UnitGeom G, const float u,
             const float *resid, float *out, float *partials, const int64_t u_begin,
             const int64_t u_end)
{
    const uint64_t pol = policy_evict_first();
    const int W = WT > 0 ? WT : tab.W;
    const int L = tab.L;
    const int lane = threadIdx.x & 31;
    // Launched after whatever the stream ran before (programmatic serialisation):
    // nothing is read before that work is complete.
    wait_for_prior_grid();
    allow_dependent_launch();  // the selection may be scheduled; it waits for us
    const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;

    for (int64_t un = u_begin + (((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5);
         un < u_end; un += nwarps) {
        int64_t c, lo, hi;
        unit_range(G, un, c, lo, hi);
        float tss = 0.f;
        const int64_t g1 = (hi + 7) >> 3;
        for (int64_t g = (lo >> 3) + lane; g < g1; g += 32) {
            const int64_t f0 = g << 3;
            float a[8];
            const bool full = (f0 >= lo) && (f0 + 8 <= hi);
            int l = find_layer(tab, f0 > lo ? f0 : lo);
            // ring order: one start worker for the whole group, if the group
            // lies in one ring segment
            const int start = ORDER == 2 ? ring_segment(f0 > lo ? f0 : lo, G.N, W) : 0;
            const bool one_start =
                ORDER != 2 || ring_segment(f0 + 7 < hi ? f0 + 7 : hi - 1, G.N, W) == start;
            if (full && one_start && f0 + 8 <= tab.off[l + 1] &&
                ((tab.vec[l >> 5] >> (l & 31)) & 1u)) {
                // vector path: 8 consecutive elements of one layer
                const int64_t j = f0 - tab.off[l];
                auto ld8 = [&](int w, float(&x)[8]) {
                    unpack8(ld_stream16(tab.ptr[w * L + l] + j, pol), x);
                };
                if constexpr (ORDER == 0)
                    tree_sum<WT, MAXH, 8>(W, ld8, a);
                else
                    seq_sum<8>(W, start, ld8, a);
                float r[8];
                if (resid) {
                    const float4 r0 = __ldcs(reinterpret_cast<const float4 *>(resid + f0));
                    const float4 r1 = __ldcs(reinterpret_cast<const float4 *>(resid + f0 + 4));
                    r[0] = r0.x; r[1] = r0.y; r[2] = r0.z; r[3] = r0.w;
                    r[4] = r1.x; r[5] = r1.y; r[6] = r1.z; r[7] = r1.w;
                }
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    a[e] = __fmul_rn(a[e], u);
                    if (resid) a[e] = __fadd_rn(a[e], r[e]);
                }
                reinterpret_cast<float4 *>(out + f0)[0] = make_float4(a[0], a[1], a[2], a[3]);
                reinterpret_cast<float4 *>(out + f0)[1] = make_float4(a[4], a[5], a[6], a[7]);
            } else {
                // element path: group clipped by the unit, crossing a layer
                // or ring-segment boundary, or a layer whose workers are not
                // 16-byte aligned
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const int64_t f = f0 + e;
                    if (f < lo || f >= hi) {
                        a[e] = 0.f;
                        continue;
                    }
                    while (tab.off[l + 1] <= f) ++l;
                    const int64_t j = f - tab.off[l];
                    float s1[1];
                    auto ld1 = [&](int w, float(&x)[1]) {
                        x[0] = ld_half_as_float(tab.ptr[w * L + l] + j);
                    };
                    if constexpr (ORDER == 0)
                        tree_sum<WT, MAXH, 1>(W, ld1, s1);
                    else
                        seq_sum<1>(W, ORDER == 2 ? ring_segment(f, G.N, W) : 0, ld1, s1);
                    float v = __fmul_rn(s1[0], u);
                    if (resid) v = __fadd_rn(v, __ldcs(resid + f));
                    out[f] = v;
                    a[e] = v;
                }
            }
            tss = __fadd_rn(tss, group_sumsq(a));
        }
        if (partials) {
            tss = warp_sum_f32(tss);
            if (lane == 0) partials[un] = tss;
        }
    }
}

template <class Tab, int WT, int MAXH, int ORDER = 0>
static cudaError_t launch_reduce_w(const Tab &tab, const UnitGeom &G, float u,
                                   const float *resid, float *out,
                                   float *partials, cudaStream_t s, int64_t ub,
                                   int64_t ue)
{
    auto kern = k_reduce<Tab, WT, MAXH, ORDER>;
    const int64_t blocks_needed = (ue - ub + FC_BLOCK / 32 - 1) / (FC_BLOCK / 32);
    const int grid = grid_for((const void *)kern, FC_BLOCK, 0, blocks_needed);
    return launch_after_prior(kern, (unsigned)grid, FC_BLOCK, 0, s, tab, G, u, resid,
                              out, partials, ub, ue);
}

template <class Tab>
cudaError_t launch_reduce(const Tab &tab, const UnitGeom &G, float u,
                          const float *resid, float *out, float *partials,
                          cudaStream_t s, int order, int64_t ub, int64_t ue)
{
    if (ue < 0) ue = G.units;
    if (ub >= ue) return cudaSuccess;
#define FC_R(WT, MAXH, ORDER) \
    launch_reduce_w<Tab, WT, MAXH, ORDER>(tab, G, u, resid, out, partials, s, ub, ue)
    if (order == 1) return FC_R(0, 1, 1);
    if (order == 2) return FC_R(0, 1, 2);
    switch (tab.W) {
    case 1: return FC_R(1, 1, 0);
    case 2: return FC_R(2, 2, 0);
    case 4: return FC_R(4, 3, 0);
    case 8: return FC_R(8, 4, 0);
    case 16: return FC_R(16, 5, 0);
    case 32: return FC_R(32, 6, 0);
    case 64: return FC_R(64, 7, 0);
    default: break;
    }
    if (tab.W < 32) return FC_R(0, 5, 0);
    if (tab.W < 128) return FC_R(0, 7, 0);
    return FC_R(0, 12, 0);
#undef FC_R
}

template cudaError_t launch_reduce<TableS>(const TableS &, const UnitGeom &,
                                           float, const float *, float *,
                                           float *, cudaStream_t, int, int64_t,
                                           int64_t);
template cudaError_t launch_reduce<TableL>(const TableL &, const UnitGeom &,
                                           float, const float *, float *,
                                           float *, cudaStream_t, int, int64_t,
                                           int64_t);

}  // namespace fc
