// a5: residual fold and momentum-SGD update of the fp32 master weights.
//
// FireCaffe (arXiv 1511.00175), §3: training is batched SGD; §6: every worker
// applies the summed gradient to its copy of the model.  The pages give no
// optimiser formula; the engine uses Caffe's momentum form (FireCaffe is
// Caffe-compatible, appendix): v = momentum*v + lr*g, w = w - v.  Values of
// chunks that were not sent (GradientFlow, arXiv 1902.06855, abstract:
// coarse-grained sparse communication) are carried to the next step in an
// fp32 residual instead of being dropped.  The kept chunks are also written
// to the send buffers: fp32, and/or fp16 (mixed-precision communication,
// GradientFlow abstract) as binary16(a * send_scale).
//
// GB300 mapping: one streaming pass over the chunk-aligned tiles, so every
// tile has a single kept/unkept decision (no per-element division); 16-byte
// loads and stores with evict-first hints; when the reduced gradient sits in
// the residual buffer (in place), unkept tiles neither read it nor rewrite
// it, which leaves 16 bytes per element (velocity and weights) for the
// common unkept case.
#include "fc_internal.h"

namespace fc {

// Threads per block of the update (each tile of 2048 elements is 512
// 16-byte groups, spread over the block's threads).
#ifndef FC_UPDATE_BLOCK
#define FC_UPDATE_BLOCK 128
#endif

__global__ void __launch_bounds__(FC_UPDATE_BLOCK)
    k_update(const TileGeom G, const int64_t tiles, const float *a,
             const uint8_t *__restrict__ mask, const int32_t *__restrict__ slot,
             float *__restrict__ packed, __half *__restrict__ packed16,
             const float send_scale, const float lr, const float mu,
             float *r, float *__restrict__ v, float *__restrict__ w,
             __half *__restrict__ w16, const int inplace,
             const unsigned *__restrict__ status)
{
    const int64_t cs = G.cs;
    const bool pvec = (cs & 3) == 0;
    wait_for_prior_grid();
    allow_dependent_launch();  // the next step's reduction waits for us
    // the selection marked the step as not applied: change nothing
    if (status && __ldcg(status) != 0u) return;
    for (int64_t t = blockIdx.x; t < tiles; t += gridDim.x) {
        int64_t lo, hi, c, hin;
        const bool any = tile_range(G, t, lo, hi, c, hin);
        const bool kept = __ldg(mask + c) != 0;
        const bool need_a = kept || !inplace;
        const bool write_r = kept || !inplace;
        // packed index of element i of a kept chunk: pbase + i
        const int32_t sl = ((packed != nullptr || packed16 != nullptr) && kept)
                               ? __ldg(slot + c) : -1;
        const bool pk = sl >= 0;  // the slot map comes from the same selection
        const int64_t pbase = pk ? (int64_t)sl * cs - c * cs : 0;
        if (any) {
            const int64_t q1 = (hi + 3) >> 2;
#pragma unroll 4
            for (int64_t q = (lo >> 2) + threadIdx.x; q < q1; q += FC_UPDATE_BLOCK) {
                const int64_t i0 = q << 2;
                if (i0 >= lo && i0 + 4 <= hi) {
                    float4 av = make_float4(0.f, 0.f, 0.f, 0.f);
                    if (need_a) av = __ldcs(reinterpret_cast<const float4 *>(a + i0));
                    float4 vv = __ldcs(reinterpret_cast<const float4 *>(v + i0));
                    float4 ww = __ldcs(reinterpret_cast<const float4 *>(w + i0));
                    float4 rr;
                    sgd1(av.x, kept, lr, mu, rr.x, vv.x, ww.x);
                    sgd1(av.y, kept, lr, mu, rr.y, vv.y, ww.y);
                    sgd1(av.z, kept, lr, mu, rr.z, vv.z, ww.z);
                    sgd1(av.w, kept, lr, mu, rr.w, vv.w, ww.w);
                    __stcs(reinterpret_cast<float4 *>(v + i0), vv);
                    __stcs(reinterpret_cast<float4 *>(w + i0), ww);
                    if (write_r) __stcs(reinterpret_cast<float4 *>(r + i0), rr);
                    if (w16) {
                        __half2 h0 = __floats2half2_rn(ww.x, ww.y);
                        __half2 h1 = __floats2half2_rn(ww.z, ww.w);
                        uint2 hv;
                        hv.x = *reinterpret_cast<uint32_t *>(&h0);
                        hv.y = *reinterpret_cast<uint32_t *>(&h1);
                        __stcs(reinterpret_cast<uint2 *>(w16 + i0), hv);
                    }
                    if (pk && packed) {
                        if (pvec) {
                            __stcs(reinterpret_cast<float4 *>(packed + pbase + i0), av);
                        } else {
                            packed[pbase + i0] = av.x;
                            packed[pbase + i0 + 1] = av.y;
                            packed[pbase + i0 + 2] = av.z;
                            packed[pbase + i0 + 3] = av.w;
                        }
                    }
                    if (pk && packed16) {
                        const __half2 s0 = __floats2half2_rn(__fmul_rn(av.x, send_scale),
                                                             __fmul_rn(av.y, send_scale));
                        const __half2 s1 = __floats2half2_rn(__fmul_rn(av.z, send_scale),
                                                             __fmul_rn(av.w, send_scale));
                        if (pvec) {
                            uint2 hv;
                            hv.x = *reinterpret_cast<const uint32_t *>(&s0);
                            hv.y = *reinterpret_cast<const uint32_t *>(&s1);
                            __stcs(reinterpret_cast<uint2 *>(packed16 + pbase + i0), hv);
                        } else {
                            packed16[pbase + i0] = __low2half(s0);
                            packed16[pbase + i0 + 1] = __high2half(s0);
                            packed16[pbase + i0 + 2] = __low2half(s1);
                            packed16[pbase + i0 + 3] = __high2half(s1);
                        }
                    }
                } else {
                    for (int e = 0; e < 4; ++e) {
                        const int64_t i = i0 + e;
                        if (i < lo || i >= hi) continue;
                        const float ai = need_a ? __ldcs(a + i) : 0.f;
                        float vi = v[i], wi = w[i], ri;
                        sgd1(ai, kept, lr, mu, ri, vi, wi);
                        v[i] = vi;
                        w[i] = wi;
                        if (write_r) r[i] = ri;
                        if (w16) w16[i] = __float2half_rn(wi);
                        if (pk && packed) packed[pbase + i] = ai;
                        if (pk && packed16)
                            packed16[pbase + i] = __float2half_rn(__fmul_rn(ai, send_scale));
                    }
                }
            }
        }
        // zero the packed slot beyond N (short last chunk)
        if (pk && hin > hi) {
            const int64_t p0 = lo > G.N ? lo : G.N;
            for (int64_t i = p0 + threadIdx.x; i < hin; i += FC_UPDATE_BLOCK) {
                if (packed) packed[pbase + i] = 0.f;
                if (packed16) packed16[pbase + i] = __float2half_rn(0.f);
            }
        }
    }
}

cudaError_t launch_update(const TileGeom &G, int64_t tiles, const float *a,
                          const uint8_t *mask, const int32_t *slot,
                          float *packed, __half *packed16, float send_scale,
                          float lr, float mu, float *r, float *v, float *w,
                          __half *w16, bool inplace, cudaStream_t s,
                          const unsigned *status)
{
    int grid = grid_for((const void *)k_update, FC_UPDATE_BLOCK, 0, tiles);
    // as many rounds of tiles as the resident blocks need, dealt out evenly
    // (the last round as full as the others)
    if (tiles > grid) {
        const int64_t rounds = (tiles + grid - 1) / grid;
        grid = (int)((tiles + rounds - 1) / rounds);
    }
    return launch_after_prior(k_update, (unsigned)grid, FC_UPDATE_BLOCK, 0, s, G, tiles,
                              a, mask, slot, packed, packed16, send_scale, lr,
                              mu, r, v, w, w16, inplace ? 1 : 0, status);
}

}  // namespace fc
