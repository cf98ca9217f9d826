// The C ABI of libfc: argument checks, layout/tiling arithmetic on the host,
// and kernel launches.  Declarations and the contract of every entry point
// are in include/fc.h.
#include <math.h>
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include <nvtx3/nvToolsExt.h>

#include "fc.h"
#include "fc_internal.h"

using namespace fc;

namespace {

// NVTX range around every entry point (a no-op unless a profiler such as
// Nsight Systems or Nsight Compute is attached), so that traces show the
// engine's calls by name.
struct TraceRange {
    explicit TraceRange(const char *name) { nvtxRangePushA(name); }
    ~TraceRange() { nvtxRangePop(); }
};

thread_local char g_err[512] = "";

fc_status fail(fc_status st, const char *fmt, ...)
{
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_err, sizeof(g_err), fmt, ap);
    va_end(ap);
    return st;
}

fc_status ok()
{
    g_err[0] = '\0';
    return FC_OK;
}

fc_status cuda_fail(cudaError_t e, const char *what)
{
    return fail(FC_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e),
                cudaGetErrorString(e));
}

bool aligned(const void *p, uintptr_t a) { return ((uintptr_t)p & (a - 1)) == 0; }

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

TileGeom geom(int64_t N, int64_t cs)
{
    TileGeom G;
    G.N = N;
    G.cs = cs;
    G.P = ceil_div(cs, FC_TILE);
    return G;
}

UnitGeom ugeom(int64_t N, int64_t cs)
{
    UnitGeom G;
    G.N = N;
    G.cs = cs;
    G.C = ceil_div(N, cs);
    G.U = ceil_div(cs, FC_UNIT);
    const int64_t last = N - (G.C - 1) * cs;
    G.units = (G.C - 1) * G.U + ceil_div(last, FC_UNIT);
    return G;
}

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

// Workspace of the pipeline: unit sums (float [units]), a 256-byte block of
// 32-bit words (0: the selection's count of finished blocks; 1: the staged
// reduction's failure word; 2: the last step's outcome, 0 = applied; 4-5:
// the staged reduction's 64-bit counter of dynamically handed-out tiles; 6:
// its count of finished producers; all but word 2 zero between calls;
// 8-12: the one-launch grid step's 64-bit barrier count and its hand-off
// of the k-th chunk) and the kept-slot map (int32 [C]).
struct WsLayout {
    size_t partials, counters, slot, total;
};

WsLayout ws_layout(int64_t N, int64_t cs)
{
    const UnitGeom G = ugeom(N, cs);
    WsLayout l;
    l.partials = 0;
    l.counters = align256((size_t)G.units * sizeof(float));
    l.slot = l.counters + 256;
    l.total = l.slot + align256((size_t)G.C * sizeof(int32_t));
    return l;
}

fc_status check_sizes(int32_t L, const int64_t *sizes, int64_t *N_out)
{
    if (L < 1) return fail(FC_ERR_INVALID_ARG, "L = %d must be >= 1", L);
    if (!sizes) return fail(FC_ERR_INVALID_ARG, "sizes is NULL");
    int64_t N = 0;
    for (int32_t l = 0; l < L; ++l) {
        if (sizes[l] < 0) return fail(FC_ERR_INVALID_ARG, "sizes[%d] = %lld < 0", l, (long long)sizes[l]);
        if (sizes[l] > ((int64_t)1 << 48) || N > ((int64_t)1 << 48))
            return fail(FC_ERR_INVALID_ARG, "sizes too large");
        N += sizes[l];
    }
    if (N < 1) return fail(FC_ERR_INVALID_ARG, "the sizes sum to 0");
    *N_out = N;
    return FC_OK;
}

fc_status check_table(const void *const *grads, int32_t W, int32_t L,
                      const int64_t *sizes)
{
    if (!grads) return fail(FC_ERR_INVALID_ARG, "grads is NULL");
    if (W < 1) return fail(FC_ERR_INVALID_ARG, "W = %d must be >= 1", W);
    if (L > FC_MAX_TABLE_LAYERS)
        return fail(FC_ERR_LIMIT, "L = %d exceeds FC_MAX_TABLE_LAYERS = %d", L, FC_MAX_TABLE_LAYERS);
    if ((int64_t)W * L > FC_MAX_TABLE_PTRS)
        return fail(FC_ERR_LIMIT, "W*L = %lld exceeds FC_MAX_TABLE_PTRS = %d",
                    (long long)W * L, FC_MAX_TABLE_PTRS);
    for (int64_t i = 0; i < (int64_t)W * L; ++i) {
        if (sizes[i % L] == 0) continue;
        if (!grads[i]) return fail(FC_ERR_INVALID_ARG, "grads[%lld] is NULL", (long long)i);
        if (!aligned(grads[i], 2))
            return fail(FC_ERR_ALIGNMENT, "grads[%lld] is not 2-byte aligned", (long long)i);
    }
    return FC_OK;
}

bool fits_small(int32_t W, int32_t L)
{
    return L <= 64 && (int64_t)W * L <= 256;
}

fc_status check_f32(const void *p, const char *name, bool may_be_null)
{
    if (!p) return may_be_null ? FC_OK : fail(FC_ERR_INVALID_ARG, "%s is NULL", name);
    if (!aligned(p, 16)) return fail(FC_ERR_ALIGNMENT, "%s is not 16-byte aligned", name);
    return FC_OK;
}

// The TMA-staged phase 1 serves the tree order for 4, 8 or 16 workers, when
// every layer has one address shift for all workers.  Returns the layout
// (tma_layout) or 0 for the register kernel.
template <class Tab>
int use_tma(const Tab &tab, const UnitGeom &G, const float *partials, int order)
{
#ifdef FC_DISABLE_TMA
    (void)tab; (void)G; (void)partials; (void)order;
    return 0;
#else
    // With more than 16 workers a 64 KB stage holds fewer than eight units,
    // which leaves consumer warps idle; the register kernel streams those
    // layouts at the copy rate already.
    const int W = tab.W;
    if (order != FC_ORDER_TREE) return 0;
    if (W != 4 && W != 8 && W != 16) return 0;
    return tma_layout(tab, G, partials);
#endif
}

#define TRY(x)                         \
    do {                               \
        fc_status _st = (x);           \
        if (_st != FC_OK) return _st;  \
    } while (0)

}  // namespace

extern "C" {

const char *fc_last_error(void) { return g_err; }

int32_t fc_version(void) { return 200; }

int64_t fc_num_chunks(int64_t N, int64_t chunk)
{
    if (N < 0 || chunk < 1) return -1;
    return ceil_div(N, chunk);
}

int64_t fc_keep_count(int64_t C, int64_t keep_num, int64_t keep_den)
{
    if (C < 1 || keep_num < 0 || keep_den < 1) return -1;
    if (keep_num > keep_den) keep_num = keep_den;
    // C * keep_num may not fit in 64 bits for large denominators
    const __int128 prod = (__int128)C * keep_num;
    int64_t k = (int64_t)((prod + keep_den - 1) / keep_den);
    if (k < 1) k = 1;
    if (k > C) k = C;
    return k;
}

fc_status fc_layout(int32_t L, const int64_t *sizes, int64_t *offsets,
                    int64_t *N_out)
{
    int64_t N = 0;
    TRY(check_sizes(L, sizes, &N));
    if (offsets) {
        int64_t acc = 0;
        for (int32_t l = 0; l < L; ++l) {
            offsets[l] = acc;
            acc += sizes[l];
        }
    }
    if (N_out) *N_out = N;
    return ok();
}

fc_status fc_fuse_pack(const void *const *grads, int32_t W, int32_t L,
                       const int64_t *sizes, int64_t *offsets, void *fused,
                       void *stream)
{
    TraceRange trace("fc_fuse_pack");
    int64_t N = 0;
    TRY(check_sizes(L, sizes, &N));
    TRY(check_table(grads, W, L, sizes));
    if (!fused) return fail(FC_ERR_INVALID_ARG, "fused is NULL");
    if (!aligned(fused, 16)) return fail(FC_ERR_ALIGNMENT, "fused is not 16-byte aligned");
    if (offsets) TRY(fc_layout(L, sizes, offsets, nullptr));
    DeviceScope scope;
    TRY(scope.bind(fused));
    cudaError_t e;
    if (fits_small(W, L)) {
        TableS tab;
        fill_table(tab, grads, W, L, sizes);
        e = launch_pack(tab, N, (__half *)fused, (cudaStream_t)stream);
    } else {
        static thread_local TableL tab;
        fill_table(tab, grads, W, L, sizes);
        e = launch_pack(tab, N, (__half *)fused, (cudaStream_t)stream);
    }
    if (e != cudaSuccess) return cuda_fail(e, "fuse_pack launch");
    return ok();
}

fc_status fc_reduce_ordered(const void *fused, int32_t W, int64_t N,
                            float loss_scale, const float *residual_in,
                            float *out, int32_t order, void *stream)
{
    TraceRange trace("fc_reduce_ordered");
    if (order < FC_ORDER_TREE || order > FC_ORDER_RING)
        return fail(FC_ERR_INVALID_ARG, "order = %d is not an FC_ORDER_* value", order);
    if (!fused) return fail(FC_ERR_INVALID_ARG, "fused is NULL");
    if (W < 1 || W > FC_MAX_TABLE_PTRS)
        return fail(FC_ERR_INVALID_ARG, "W = %d out of [1, %d]", W, FC_MAX_TABLE_PTRS);
    if (N < 1) return fail(FC_ERR_INVALID_ARG, "N = %lld must be >= 1", (long long)N);
    if (!(loss_scale > 0.f) || !isfinite(loss_scale))
        return fail(FC_ERR_INVALID_ARG, "loss_scale must be finite and > 0");
    if (!aligned(fused, 2)) return fail(FC_ERR_ALIGNMENT, "fused is not 2-byte aligned");
    TRY(check_f32(residual_in, "residual_in", true));
    TRY(check_f32(out, "out", false));
    DeviceScope scope;
    TRY(scope.bind(out));
    const float u = (float)(1.0 / ((double)loss_scale * (double)W));
    const UnitGeom G = ugeom(N, N);  // one chunk: no norms here
    const int64_t sizes[1] = {N};
    cudaError_t e;
    // one "layer" per worker: row w of the fused buffer
    if (W <= 256) {
        TableS tab;
        const void *rows[256];
        for (int w = 0; w < W; ++w) rows[w] = (const __half *)fused + (int64_t)w * N;
        fill_table(tab, rows, W, 1, sizes);
        e = launch_reduce(tab, G, u, residual_in, out, nullptr, (cudaStream_t)stream, order);
    } else {
        static thread_local TableL tab;
        static thread_local const void *rows[FC_MAX_TABLE_PTRS];
        for (int w = 0; w < W; ++w) rows[w] = (const __half *)fused + (int64_t)w * N;
        fill_table(tab, rows, W, 1, sizes);
        e = launch_reduce(tab, G, u, residual_in, out, nullptr, (cudaStream_t)stream, order);
    }
    if (e != cudaSuccess) return cuda_fail(e, "reduce launch");
    return ok();
}

fc_status fc_tree_reduce(const void *fused, int32_t W, int64_t N,
                         float loss_scale, const float *residual_in,
                         float *out, void *stream)
{
    return fc_reduce_ordered(fused, W, N, loss_scale, residual_in, out,
                             FC_ORDER_TREE, stream);
}

fc_status fc_chunk_norms(const float *a, int64_t N, int64_t chunk,
                         float *norms, void *stream)
{
    TraceRange trace("fc_chunk_norms");
    if (N < 1) return fail(FC_ERR_INVALID_ARG, "N must be >= 1");
    if (chunk < 1) return fail(FC_ERR_INVALID_ARG, "chunk must be >= 1");
    TRY(check_f32(a, "a", false));
    TRY(check_f32(norms, "norms", false));
    DeviceScope scope;
    TRY(scope.bind(a));
    cudaError_t e = launch_norms(a, ugeom(N, chunk), norms, (cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(e, "chunk_norms launch");
    return ok();
}

size_t fc_chunk_select_workspace(int64_t C)
{
    (void)C;  // the selection's scratch lives in one block's shared memory
    return 0;
}

static fc_status check_select_args(int64_t C, int64_t k, const int32_t *idx,
                                   const uint8_t *mask, const float *threshold)
{
    if (C < 1 || C > 0x7fffffffLL) return fail(FC_ERR_INVALID_ARG, "C = %lld out of range", (long long)C);
    if (k < 1 || k > C) return fail(FC_ERR_INVALID_ARG, "k = %lld must be in [1, C = %lld]", (long long)k, (long long)C);
    if (!idx) return fail(FC_ERR_INVALID_ARG, "idx is NULL");
    if (!mask) return fail(FC_ERR_INVALID_ARG, "mask is NULL");
    if (!threshold) return fail(FC_ERR_INVALID_ARG, "threshold is NULL");
    if (!aligned(idx, 4) || !aligned(threshold, 4))
        return fail(FC_ERR_ALIGNMENT, "idx/threshold are not 4-byte aligned");
    return FC_OK;
}

fc_status fc_chunk_select(const float *norms, int64_t C, int64_t k,
                          const float *a, int64_t N, int64_t chunk,
                          int32_t *idx, uint8_t *mask, float *packed,
                          void *packed_fp16, float send_scale,
                          float *threshold, void *stream)
{
    TraceRange trace("fc_chunk_select");
    TRY(check_select_args(C, k, idx, mask, threshold));
    TRY(check_f32(norms, "norms", false));
    if (packed || packed_fp16) {
        TRY(check_f32(a, "a", false));
        TRY(check_f32(packed, "packed", true));
        TRY(check_f32(packed_fp16, "packed_fp16", true));
        if (!isfinite(send_scale))
            return fail(FC_ERR_INVALID_ARG, "send_scale must be finite");
        if (chunk < 1 || N < 1 || ceil_div(N, chunk) != C)
            return fail(FC_ERR_INVALID_ARG, "N and chunk do not give C chunks");
    }
    DeviceScope scope;
    TRY(scope.bind(norms));
    UnitGeom G;
    G.N = N;
    G.cs = chunk;
    G.C = C;
    G.U = 1;
    G.units = C;
    cudaError_t e = launch_select(G, nullptr, nullptr, const_cast<float *>(norms), k,
                                  idx, mask, nullptr, threshold, (cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(e, "chunk_select launch");
    if (packed || packed_fp16) {
        e = launch_gather(a, N, chunk, ceil_div(chunk, FC_TILE), idx, k, packed,
                          (__half *)packed_fp16, send_scale, (cudaStream_t)stream);
        if (e != cudaSuccess) return cuda_fail(e, "gather launch");
    }
    return ok();
}

static fc_status check_update_args(const float *a, const uint8_t *mask,
                                   int64_t N, int64_t chunk, float lr,
                                   float momentum, float *residual,
                                   float *velocity, float *weights,
                                   void *weights_fp16)
{
    if (N < 1) return fail(FC_ERR_INVALID_ARG, "N must be >= 1");
    if (chunk < 1) return fail(FC_ERR_INVALID_ARG, "chunk must be >= 1");
    if (!isfinite(lr) || !isfinite(momentum))
        return fail(FC_ERR_INVALID_ARG, "lr and momentum must be finite");
    if (!mask) return fail(FC_ERR_INVALID_ARG, "mask is NULL");
    TRY(check_f32(a, "a", false));
    TRY(check_f32(residual, "residual", false));
    TRY(check_f32(velocity, "velocity", false));
    TRY(check_f32(weights, "weights", false));
    TRY(check_f32(weights_fp16, "weights_fp16", true));
    return FC_OK;
}

fc_status fc_residual_sgd_update(const float *a, const uint8_t *mask,
                                 int64_t N, int64_t chunk, float lr,
                                 float momentum, float *residual,
                                 float *velocity, float *weights,
                                 void *weights_fp16, void *stream)
{
    TraceRange trace("fc_residual_sgd_update");
    TRY(check_update_args(a, mask, N, chunk, lr, momentum, residual, velocity,
                          weights, weights_fp16));
    DeviceScope scope;
    TRY(scope.bind(a));
    const TileGeom G = geom(N, chunk);
    const int64_t tiles = ceil_div(N, chunk) * G.P;
    cudaError_t e = launch_update(G, tiles, a, mask, nullptr, nullptr, nullptr, 1.f, lr,
                                  momentum, residual, velocity, weights,
                                  (__half *)weights_fp16, a == residual,
                                  (cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(e, "update launch");
    return ok();
}

size_t fc_step_workspace_size(int64_t N, int64_t chunk)
{
    if (N < 1 || chunk < 1) return 0;
    return ws_layout(N, chunk).total;
}

static fc_status check_ws(int64_t N, int64_t chunk, void *ws, size_t bytes)
{
    if (!ws) return fail(FC_ERR_WORKSPACE, "workspace is NULL");
    if (!aligned(ws, 256)) return fail(FC_ERR_ALIGNMENT, "workspace is not 256-byte aligned");
    const size_t need = fc_step_workspace_size(N, chunk);
    if (bytes < need)
        return fail(FC_ERR_WORKSPACE, "workspace has %zu bytes, %zu needed", bytes, need);
    return FC_OK;
}

// First unit (in the order of the unit index) whose first element is at or
// after fused index f; G.units if none.
static int64_t first_unit_at(const UnitGeom &G, int64_t f)
{
    if (f <= 0) return 0;
    if (f >= G.N) return G.units;
    const int64_t c = f / G.cs;
    const int64_t j = ceil_div(f - c * G.cs, FC_UNIT);
    const int64_t in_c = c + 1 < G.C ? G.U : G.units - c * G.U;
    return j < in_c ? c * G.U + j : (c + 1) * G.U;
}

// Phase 1 over the units whose first element lies in [f_begin, f_end).
static fc_status reduce_span(const char *name, const void *const *grads, int32_t W,
                             int32_t L, const int64_t *sizes, float loss_scale,
                             int64_t chunk, const float *residual, float *a, int32_t order,
                             int64_t f_begin, int64_t f_end, bool whole, void *workspace,
                             size_t workspace_bytes, void *stream)
{
    TraceRange trace(name);
    if (order < FC_ORDER_TREE || order > FC_ORDER_RING)
        return fail(FC_ERR_INVALID_ARG, "order = %d is not an FC_ORDER_* value", order);
    int64_t N = 0;
    TRY(check_sizes(L, sizes, &N));
    TRY(check_table(grads, W, L, sizes));
    if (chunk < 1) return fail(FC_ERR_INVALID_ARG, "chunk must be >= 1");
    if (!(loss_scale > 0.f) || !isfinite(loss_scale))
        return fail(FC_ERR_INVALID_ARG, "loss_scale must be finite and > 0");
    if (whole) {
        f_begin = 0;
        f_end = N;
    } else if (f_begin < 0 || f_end < f_begin || f_end > N) {
        return fail(FC_ERR_INVALID_ARG, "span [%lld, %lld) is not inside [0, N = %lld]",
                    (long long)f_begin, (long long)f_end, (long long)N);
    }
    TRY(check_f32(residual, "residual", true));
    TRY(check_f32(a, "a", false));
    TRY(check_ws(N, chunk, workspace, workspace_bytes));
    DeviceScope scope;
    TRY(scope.bind(a));
    const float u = (float)(1.0 / ((double)loss_scale * (double)W));
    const UnitGeom G = ugeom(N, chunk);
    const WsLayout wl = ws_layout(N, chunk);
    float *partials = (float *)((char *)workspace + wl.partials);
    unsigned *ctr = (unsigned *)((char *)workspace + wl.counters);
    const int64_t ub = first_unit_at(G, f_begin), ue = first_unit_at(G, f_end);
    if (ub >= ue) return ok();
    cudaError_t e;
    auto run = [&](const auto &tab) {
        if (const int lay = use_tma(tab, G, partials, order)) {
            // chunk % 256 == 0 here: unit j starts at 256 j
            const int64_t fb = ub * FC_UNIT;
            const int64_t fe = ue * FC_UNIT < N ? ue * FC_UNIT : N;
            return launch_reduce_tma(tab, G, u, residual, a, partials, ctr,
                                     (cudaStream_t)stream, lay, fb, fe);
        }
        return launch_reduce(tab, G, u, residual, a, partials, (cudaStream_t)stream, order,
                             ub, ue);
    };
    if (fits_small(W, L)) {
        TableS tab;
        fill_table(tab, grads, W, L, sizes);
        e = run(tab);
    } else {
        static thread_local TableL tab;
        fill_table(tab, grads, W, L, sizes);
        e = run(tab);
    }
    if (e != cudaSuccess) return cuda_fail(e, "step_reduce launch");
    return ok();
}

fc_status fc_step_reduce_ordered(const void *const *grads, int32_t W,
                                 int32_t L, const int64_t *sizes,
                                 float loss_scale, int64_t chunk,
                                 const float *residual, float *a,
                                 int32_t order, void *workspace,
                                 size_t workspace_bytes, void *stream)
{
    return reduce_span("fc_step_reduce_ordered", grads, W, L, sizes, loss_scale, chunk,
                       residual, a, order, 0, 0, true, workspace, workspace_bytes, stream);
}

fc_status fc_step_reduce_span(const void *const *grads, int32_t W, int32_t L,
                              const int64_t *sizes, float loss_scale, int64_t chunk,
                              const float *residual, float *a, int64_t f_begin,
                              int64_t f_end, void *workspace, size_t workspace_bytes,
                              void *stream)
{
    return reduce_span("fc_step_reduce_span", grads, W, L, sizes, loss_scale, chunk, residual,
                       a, FC_ORDER_TREE, f_begin, f_end, false, workspace, workspace_bytes,
                       stream);
}

int64_t fc_unit_start(int64_t N, int64_t chunk, int64_t f)
{
    if (N < 1 || chunk < 1 || f < 0 || f > N) return -1;
    if (f == N) return N;
    const int64_t c = f / chunk;
    return c * chunk + (f - c * chunk) / FC_UNIT * FC_UNIT;
}

int32_t fc_step_reduce_kernel(const void *const *grads, int32_t W, int32_t L,
                              const int64_t *sizes, int64_t chunk, int32_t order)
{
    if (order < FC_ORDER_TREE || order > FC_ORDER_RING) {
        fail(FC_ERR_INVALID_ARG, "order = %d is not an FC_ORDER_* value", order);
        return -1;
    }
    int64_t N = 0;
    if (check_sizes(L, sizes, &N) != FC_OK || check_table(grads, W, L, sizes) != FC_OK)
        return -1;
    if (chunk < 1) {
        fail(FC_ERR_INVALID_ARG, "chunk must be >= 1");
        return -1;
    }
    const UnitGeom G = ugeom(N, chunk);
    // phase 1 always writes unit sums in the pipeline: any non-null marker
    const float *partials = reinterpret_cast<const float *>(sizeof(float));
    int lay;
    if (fits_small(W, L)) {
        TableS tab;
        fill_table(tab, grads, W, L, sizes);
        lay = use_tma(tab, G, partials, order);
    } else {
        static thread_local TableL tab;
        fill_table(tab, grads, W, L, sizes);
        lay = use_tma(tab, G, partials, order);
    }
    ok();
    return lay == 1 ? FC_REDUCE_STAGED : lay == 2 ? FC_REDUCE_STAGED_SHIFTED : FC_REDUCE_REGISTER;
}

fc_status fc_step_reduce(const void *const *grads, int32_t W, int32_t L,
                         const int64_t *sizes, float loss_scale,
                         int64_t chunk, const float *residual, float *a,
                         void *workspace, size_t workspace_bytes,
                         void *stream)
{
    return fc_step_reduce_ordered(grads, W, L, sizes, loss_scale, chunk,
                                  residual, a, FC_ORDER_TREE, workspace,
                                  workspace_bytes, stream);
}

fc_status fc_step_select(int64_t N, int64_t chunk, int64_t k, float *norms,
                         int32_t *idx, uint8_t *mask, float *threshold,
                         void *workspace, size_t workspace_bytes,
                         void *stream)
{
    TraceRange trace("fc_step_select");
    if (N < 1 || chunk < 1) return fail(FC_ERR_INVALID_ARG, "N and chunk must be >= 1");
    const int64_t C = ceil_div(N, chunk);
    TRY(check_select_args(C, k, idx, mask, threshold));
    TRY(check_f32(norms, "norms", false));
    TRY(check_ws(N, chunk, workspace, workspace_bytes));
    DeviceScope scope;
    TRY(scope.bind(norms));
    const WsLayout wl = ws_layout(N, chunk);
    const float *partials = (const float *)((const char *)workspace + wl.partials);
    unsigned *done = (unsigned *)((char *)workspace + wl.counters);
    int32_t *slot = (int32_t *)((char *)workspace + wl.slot);
    cudaError_t e = launch_select(ugeom(N, chunk), partials, done, norms, k, idx,
                                  mask, slot, threshold, (cudaStream_t)stream, done + 1,
                                  done + 2);
    if (e != cudaSuccess) return cuda_fail(e, "step_select launch");
    return ok();
}

fc_status fc_step_update(const float *a, int64_t N, int64_t chunk, float lr,
                         float momentum, float *residual, float *velocity,
                         float *weights, void *weights_fp16,
                         const uint8_t *mask, float *packed,
                         void *packed_fp16, float send_scale, void *workspace,
                         size_t workspace_bytes, void *stream)
{
    TraceRange trace("fc_step_update");
    TRY(check_update_args(a, mask, N, chunk, lr, momentum, residual, velocity,
                          weights, weights_fp16));
    TRY(check_f32(packed, "packed", true));
    TRY(check_f32(packed_fp16, "packed_fp16", true));
    if (!isfinite(send_scale)) return fail(FC_ERR_INVALID_ARG, "send_scale must be finite");
    TRY(check_ws(N, chunk, workspace, workspace_bytes));
    DeviceScope scope;
    TRY(scope.bind(a));
    const TileGeom G = geom(N, chunk);
    const int64_t C = ceil_div(N, chunk);
    const WsLayout wl = ws_layout(N, chunk);
    const int32_t *slot = (const int32_t *)((char *)workspace + wl.slot);
    const unsigned *status = (const unsigned *)((char *)workspace + wl.counters) + 2;
    cudaError_t e = launch_update(G, C * G.P, a, mask, slot, packed,
                                  (__half *)packed_fp16, send_scale, lr,
                                  momentum, residual, velocity, weights,
                                  (__half *)weights_fp16, a == residual,
                                  (cudaStream_t)stream, status);
    if (e != cudaSuccess) return cuda_fail(e, "step_update launch");
    return ok();
}

fc_status fc_step(const void *const *grads, int32_t W, int32_t L,
                  const int64_t *sizes, float loss_scale, int64_t chunk,
                  int64_t k, float lr, float momentum, float *residual,
                  float *a, float *velocity, float *weights,
                  void *weights_fp16, float *norms, int32_t *idx,
                  uint8_t *mask, float *packed, void *packed_fp16,
                  float send_scale, float *threshold, void *workspace,
                  size_t workspace_bytes, void *stream)
{
    TraceRange trace("fc_step");
    int64_t N = 0;
    // check everything before the first launch so that an error launches
    // nothing
    TRY(check_step_args(grads, W, L, sizes, loss_scale, chunk, k, lr, momentum, residual, a,
                        velocity, weights, weights_fp16, norms, idx, mask, packed,
                        packed_fp16, send_scale, threshold, &N));
    TRY(check_ws(N, chunk, workspace, workspace_bytes));
    // small problems: the whole step in one launch
    if (!stage_loss_armed()) {
        DeviceScope scope;
        TRY(scope.bind(a));
        const WsLayout wl = ws_layout(N, chunk);
        SmallStep st;
        st.G = ugeom(N, chunk);
        st.u = (float)(1.0 / ((double)loss_scale * (double)W));
        st.resid = residual;
        st.a = a;
        st.partials = (float *)((char *)workspace + wl.partials);
        st.norms = norms;
        st.k = k;
        st.idx = idx;
        st.mask = mask;
        st.threshold = threshold;
        st.status = (unsigned *)((char *)workspace + wl.counters) + 2;
        st.bar = (unsigned *)((char *)workspace + wl.counters) + 8;
        st.lr = lr;
        st.mu = momentum;
        st.r = residual;
        st.v = velocity;
        st.w = weights;
        st.w16 = (__half *)weights_fp16;
        st.packed = packed;
        st.packed16 = (__half *)packed_fp16;
        st.send_scale = send_scale;
        int launched = FC_STEP_THREE_KERNELS;
        cudaError_t e;
        if (fits_small(W, L)) {
            TableS tab;
            fill_table(tab, grads, W, L, sizes);
            e = launch_step_small(tab, st, (cudaStream_t)stream, false, &launched);
        } else {
            static thread_local TableL tab;
            fill_table(tab, grads, W, L, sizes);
            e = launch_step_small(tab, st, (cudaStream_t)stream, false, &launched);
        }
        if (e == cudaErrorCooperativeLaunchTooLarge || e == cudaErrorInvalidClusterSize) {
            // the device cannot hold the launch at all (for instance a
            // context limited to a share of the SMs): the three kernels
            // instead
            (void)cudaGetLastError();
            launched = FC_STEP_THREE_KERNELS;
        } else if (e != cudaSuccess) {
            return cuda_fail(e, "step_small launch");
        }
        if (launched != FC_STEP_THREE_KERNELS) return ok();
    }
    TRY(fc_step_reduce(grads, W, L, sizes, loss_scale, chunk, residual, a,
                       workspace, workspace_bytes, stream));
    TRY(fc_step_select(N, chunk, k, norms, idx, mask, threshold, workspace,
                       workspace_bytes, stream));
    TRY(fc_step_update(a, N, chunk, lr, momentum, residual, velocity, weights,
                       weights_fp16, mask, packed, packed_fp16, send_scale,
                       workspace, workspace_bytes, stream));
    return ok();
}

int32_t fc_step_path(const void *const *grads, int32_t W, int32_t L, const int64_t *sizes,
                     int64_t chunk)
{
    int64_t N = 0;
    if (check_sizes(L, sizes, &N) != FC_OK || check_table(grads, W, L, sizes) != FC_OK)
        return -1;
    if (chunk < 1) {
        fail(FC_ERR_INVALID_ARG, "chunk must be >= 1");
        return -1;
    }
    SmallStep st = {};
    st.G = ugeom(N, chunk);
    static unsigned probe_bar[5];  // never touched: the probe launches nothing
    st.bar = probe_bar;
    int small = FC_STEP_THREE_KERNELS;
    cudaError_t e;
    if (fits_small(W, L)) {
        TableS tab;
        fill_table(tab, grads, W, L, sizes);
        e = launch_step_small(tab, st, nullptr, true, &small);
    } else {
        static thread_local TableL tab;
        fill_table(tab, grads, W, L, sizes);
        e = launch_step_small(tab, st, nullptr, true, &small);
    }
    (void)e;
    (void)cudaGetLastError();
    ok();
    return small;
}

fc_status fc_step_status(const void *workspace, size_t workspace_bytes, int64_t N,
                         int64_t chunk, void *stream)
{
    TraceRange trace("fc_step_status");
    if (N < 1 || chunk < 1) return fail(FC_ERR_INVALID_ARG, "N and chunk must be >= 1");
    TRY(check_ws(N, chunk, const_cast<void *>(workspace), workspace_bytes));
    DeviceScope scope;
    TRY(scope.bind(workspace));
    const unsigned *word =
        (const unsigned *)((const char *)workspace + ws_layout(N, chunk).counters) + 2;
    unsigned h = 0;
    cudaError_t e = cudaMemcpyAsync(&h, word, sizeof(h), cudaMemcpyDeviceToHost,
                                    (cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemcpyAsync of the step status");
    e = cudaStreamSynchronize((cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
    if (h != 0u)
        return fail(FC_ERR_TIMEOUT, "the last step was not applied: a bounded wait of its "
                                    "staged reduction ran out");
    return ok();
}

}  // extern "C"

// ---- helpers for other translation units of the library ----------------------

namespace fc {

fc_status set_error(fc_status st, const char *msg)
{
    snprintf(g_err, sizeof(g_err), "%s", msg);
    return st;
}

size_t step_ws_counter_offset(int64_t N, int64_t chunk)
{
    return ws_layout(N, chunk).counters;
}

fc_status DeviceScope::bind(const void *ptr)
{
    (void)cudaGetLastError();  // clear a stale error of this runtime
    cudaPointerAttributes at;
    cudaError_t e = cudaPointerGetAttributes(&at, ptr);
    if (e != cudaSuccess) return cuda_fail(e, "cudaPointerGetAttributes");
    if (at.type != cudaMemoryTypeDevice && at.type != cudaMemoryTypeManaged)
        return fail(FC_ERR_INVALID_ARG, "pointer %p is not device memory", ptr);
    int cur = -1;
    e = cudaGetDevice(&cur);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (cur != at.device) {
        e = cudaSetDevice(at.device);
        if (e != cudaSuccess) return cuda_fail(e, "cudaSetDevice");
        if (prev_ < 0) prev_ = cur;
    }
    dev_ = at.device;
    return FC_OK;
}

DeviceScope::~DeviceScope()
{
    if (prev_ >= 0) (void)cudaSetDevice(prev_);
}

fc_status check_step_args(const void *const *grads, int32_t W, int32_t L,
                          const int64_t *sizes, float loss_scale, int64_t chunk,
                          int64_t k, float lr, float momentum, const float *residual,
                          const float *a, const float *velocity, const float *weights,
                          const void *weights_fp16, const float *norms, const int32_t *idx,
                          const uint8_t *mask, const float *packed, const void *packed_fp16,
                          float send_scale, const float *threshold, int64_t *N_out)
{
    int64_t N = 0;
    TRY(check_sizes(L, sizes, &N));
    TRY(check_table(grads, W, L, sizes));
    if (chunk < 1) return fail(FC_ERR_INVALID_ARG, "chunk must be >= 1");
    if (!(loss_scale > 0.f) || !isfinite(loss_scale))
        return fail(FC_ERR_INVALID_ARG, "loss_scale must be finite and > 0");
    TRY(check_select_args(ceil_div(N, chunk), k, idx, mask, threshold));
    TRY(check_f32(norms, "norms", false));
    TRY(check_f32(residual, "residual", true));
    TRY(check_update_args(a, mask, N, chunk, lr, momentum, const_cast<float *>(residual),
                          const_cast<float *>(velocity), const_cast<float *>(weights),
                          const_cast<void *>(weights_fp16)));
    TRY(check_f32(packed, "packed", true));
    TRY(check_f32(packed_fp16, "packed_fp16", true));
    if (!isfinite(send_scale)) return fail(FC_ERR_INVALID_ARG, "send_scale must be finite");
    *N_out = N;
    return FC_OK;
}

}  // namespace fc
