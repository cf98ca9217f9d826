// Host-side helpers of the kernels' launchers: the layer table and the
// launch-size cache.
#include <mutex>

#include "fc_internal.h"

namespace fc {

// Builds the kernels' layer table.  Consecutive layers that lie back to
// back in memory for every worker (a gradient bucket) are merged into one
// segment: the layout of the fused vector is the same, the kernels just see
// fewer, longer layers (and a bucketed layout with odd layer sizes becomes
// one aligned segment per worker).  Empty layers contribute nothing and are
// dropped.
template <class Tab>
bool fill_table(Tab &t, const void *const *grads, int32_t W, int32_t L,
                const int64_t *sizes)
{
    const int maxp = (int)(sizeof(t.ptr) / sizeof(t.ptr[0]));
    const int maxl = (int)(sizeof(t.off) / sizeof(t.off[0])) - 1;
    if (L > maxl || (int64_t)W * L > maxp) return false;
    // first pass: segment boundaries
    static thread_local int seg_first[FC_MAX_TABLE_LAYERS + 1];
    int nseg = 0;
    int64_t seg_len = 0;
    int prev = -1;
    for (int l = 0; l < L; ++l) {
        if (sizes[l] == 0) continue;
        bool extend = prev >= 0;
        for (int w = 0; extend && w < W; ++w) {
            const char *end = (const char *)grads[(int64_t)w * L + prev] + 2 * seg_len;
            if ((const char *)grads[(int64_t)w * L + l] != end) extend = false;
        }
        if (extend) {
            seg_len += sizes[l];
        } else {
            seg_first[nseg++] = l;
            prev = l;
            seg_len = sizes[l];
        }
    }
    t.W = W;
    t.L = nseg;
    // fused offsets of the segments
    int64_t acc = 0;
    int seg = 0;
    for (int l = 0; l < L; ++l) {
        if (seg < nseg && seg_first[seg] == l) t.off[seg++] = acc;
        acc += sizes[l];
    }
    t.off[nseg] = acc;
    for (int i = 0; i < (maxl + 31) / 32; ++i) t.vec[i] = 0;
    for (int sg = 0; sg < nseg; ++sg) {
        bool ok = true;
        for (int w = 0; w < W; ++w) {
            uintptr_t p = (uintptr_t)grads[(int64_t)w * L + seg_first[sg]];
            if ((p - 2u * (uintptr_t)t.off[sg]) & 15u) ok = false;
            t.ptr[w * nseg + sg] = static_cast<const __half *>(grads[(int64_t)w * L + seg_first[sg]]);
        }
        if (ok) t.vec[sg >> 5] |= 1u << (sg & 31);
    }
    return true;
}

template bool fill_table<TableS>(TableS &, const void *const *, int32_t,
                                 int32_t, const int64_t *);
template bool fill_table<TableL>(TableL &, const void *const *, int32_t,
                                 int32_t, const int64_t *);

// Shared-memory carveout (percent of the largest) preferred for every kernel
// sized by grid_for.  A kernel that needs more (the staged reduction) still
// gets what it needs.  Measured on the pipeline: with no preference set,
// the 62M-element step took 550 us; an explicit 25, 50 or 75 % on the
// selection and update kernels took it to 527 us, and the 7M-element steps
// gained 1.5 us, with each kernel's own time unchanged.  At 100 % the update
// kernel ran 15 % slower.
#ifndef FC_CARVEOUT
#define FC_CARVEOUT 50
#endif

// SM count and resident blocks per SM are looked up once per (kernel,
// device) and cached, so that later calls (for instance while a stream is
// being captured into a CUDA graph) make no further runtime queries.  The
// carveout preference is set at the same first lookup.
int grid_for(const void *kernel, int block, size_t smem, int64_t work)
{
    struct Entry {
        const void *kernel;
        int dev, block, blocks;
        size_t smem;
    };
    static std::mutex mu;
    static Entry cache[256];
    static int used = 0;
    int dev = 0;
    cudaGetDevice(&dev);
    int blocks = 0;
    {
        std::lock_guard<std::mutex> lock(mu);
        for (int i = 0; i < used; ++i)
            if (cache[i].kernel == kernel && cache[i].dev == dev &&
                cache[i].block == block && cache[i].smem == smem) {
                blocks = cache[i].blocks;
                break;
            }
    }
    if (blocks == 0) {
        int sms = 0, per_sm = 0;
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
#if FC_CARVEOUT >= 0
        cudaFuncSetAttribute(kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                             FC_CARVEOUT);
#endif
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, block,
                                                          smem) != cudaSuccess ||
            per_sm < 1)
            per_sm = 1;
        if (sms < 1) sms = 1;
        blocks = sms * per_sm;
        std::lock_guard<std::mutex> lock(mu);
        if (used < 256) cache[used++] = Entry{kernel, dev, block, blocks, smem};
    }
    int64_t g = blocks;
    if (work < g) g = work;
    return g < 1 ? 1 : (int)g;
}

}  // namespace fc
