// a1 as a materialised copy: the fused [W][N] fp16 buffer.
//
// GradientFlow (arXiv 1902.06855), abstract: lazy allreduce fuses many
// per-layer communication operations into a single one.  Row w of the fused
// buffer is worker w's layers concatenated in order (no padding).
//
// GB300 mapping: one grid row (blockIdx.y) per worker; each thread writes one
// 16-byte-aligned group of 8 destination elements with a single 16-byte store.
// A group whose 8 source elements lie in one layer is read with one 16-byte
// streaming load when the source is 16-byte aligned, else with the two
// aligned 16-byte words that hold it and a funnel shift (both words hold at
// least one byte of the layer, so neither leaves the layer's pages; the
// neighbouring thread reads the same words, so the second one mostly hits in
// L1).  Only groups that straddle a layer boundary are read element by
// element.  Groups at the ends of a row (when N is not a multiple of 8) are
// stored element by element so that two rows never write the same 16 bytes.
#include "fc_internal.h"

namespace fc {

template <class Tab>
__global__ void __launch_bounds__(FC_BLOCK)
    k_pack(const __grid_constant__ Tab tab, const int64_t N, __half *fused)
{
    const uint64_t pol = policy_evict_first();
    const int w = blockIdx.y;
    const int L = tab.L;
    const int64_t rb = (int64_t)w * N, re = rb + N;
    const int64_t q1 = (re + 7) >> 3;
    unsigned short *dst = reinterpret_cast<unsigned short *>(fused);
    for (int64_t q = (rb >> 3) + (int64_t)blockIdx.x * FC_BLOCK + threadIdx.x;
         q < q1; q += (int64_t)gridDim.x * FC_BLOCK) {
        const int64_t D0 = q << 3;
        if (D0 >= rb && D0 + 8 <= re) {
            const int64_t f0 = D0 - rb;
            int l = find_layer(tab, f0);
            const __half *src = tab.ptr[w * L + l] + (f0 - tab.off[l]);
            uint4 val;
            if (f0 + 8 <= tab.off[l + 1] && (((uintptr_t)src & 15u) == 0)) {
                val = ld_stream16(src, pol);
            } else if (f0 + 8 <= tab.off[l + 1]) {
                const uintptr_t at = (uintptr_t)src;
                const uint4 *q = reinterpret_cast<const uint4 *>(at & ~(uintptr_t)15);
                val = funnel8(__ldg(q), __ldg(q + 1), (int)((at & 15u) >> 1));
            } else {
                unsigned short h[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const int64_t f = f0 + e;
                    while (tab.off[l + 1] <= f) ++l;
                    h[e] = __ldg(reinterpret_cast<const unsigned short *>(
                        tab.ptr[w * L + l] + (f - tab.off[l])));
                }
                val.x = h[0] | ((uint32_t)h[1] << 16);
                val.y = h[2] | ((uint32_t)h[3] << 16);
                val.z = h[4] | ((uint32_t)h[5] << 16);
                val.w = h[6] | ((uint32_t)h[7] << 16);
            }
            __stcs(reinterpret_cast<uint4 *>(dst + D0), val);
        } else {
            for (int e = 0; e < 8; ++e) {
                const int64_t D = D0 + e;
                if (D < rb || D >= re) continue;
                const int64_t f = D - rb;
                const int l = find_layer(tab, f);
                dst[D] = __ldg(reinterpret_cast<const unsigned short *>(
                    tab.ptr[w * L + l] + (f - tab.off[l])));
            }
        }
    }
}

template <class Tab>
cudaError_t launch_pack(const Tab &tab, int64_t N, __half *fused,
                        cudaStream_t s)
{
    auto kern = k_pack<Tab>;
    const int64_t groups = N / 8 + 2;
    int gx = grid_for((const void *)kern, FC_BLOCK, 0,
                      (groups + FC_BLOCK - 1) / FC_BLOCK * tab.W);
    gx = (gx + tab.W - 1) / tab.W;
    const int64_t need = (groups + FC_BLOCK - 1) / FC_BLOCK;
    if (gx > need) gx = (int)need;
    if (gx < 1) gx = 1;
    dim3 grid(gx, tab.W);
    kern<<<grid, FC_BLOCK, 0, s>>>(tab, N, fused);
    return cudaGetLastError();
}

template cudaError_t launch_pack<TableS>(const TableS &, int64_t, __half *,
                                         cudaStream_t);
template cudaError_t launch_pack<TableL>(const TableL &, int64_t, __half *,
                                         cudaStream_t);

}  // namespace fc
