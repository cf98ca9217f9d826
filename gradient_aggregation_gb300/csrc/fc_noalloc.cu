// fc_step_noalloc: the fused pipeline with its scratch in a fixed device
// array that ships inside libfc, for callers that cannot allocate device
// memory when they step.
//
// The array below is a file-scope __device__ variable: every GPU that loads
// the library holds FC_NOALLOC_WORKSPACE_BYTES of it until the process exits.
// In host code the name `g_noalloc_ws` is only a host-side stand-in, not a
// device address, so the device address is looked up with
// cudaGetSymbolAddress while the device is current, checked, and cached.
// The cache entry of a device remembers the identity of the CUDA context it
// was looked up in: cudaDeviceReset destroys that context (and with it the
// array's mapping), and the next call, seeing another context, looks the
// address up again instead of handing the kernels a stale one.
#include <stdio.h>

#include <mutex>

#include "fc.h"
#include "fc_internal.h"

namespace {

__device__ __align__(256) unsigned char g_noalloc_ws[FC_NOALLOC_WORKSPACE_BYTES];

constexpr int kMaxDevices = 64;

struct CacheEntry {
    void *addr;
    unsigned long long ctx_id;  // 0: unknown, look the address up every call
};

std::mutex g_mu;
CacheEntry g_cache[kMaxDevices];

// Driver calls reached through the runtime's entry-point query, so that the
// library needs no link against the driver library.  Both are plain queries
// (legal while a stream is being captured).
using CtxGetCurrentFn = int (*)(void **ctx);
using CtxGetIdFn = int (*)(void *ctx, unsigned long long *id);

struct DriverQueries {
    CtxGetCurrentFn get_current = nullptr;
    CtxGetIdFn get_id = nullptr;
};

const DriverQueries &driver_queries()
{
    static DriverQueries q = [] {
        DriverQueries d;
        void *fn = nullptr;
        cudaDriverEntryPointQueryResult res;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &fn, 4000, cudaEnableDefault,
                                             &res) == cudaSuccess &&
            res == cudaDriverEntryPointSuccess)
            d.get_current = reinterpret_cast<CtxGetCurrentFn>(fn);
        fn = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &fn, 12000, cudaEnableDefault,
                                             &res) == cudaSuccess &&
            res == cudaDriverEntryPointSuccess)
            d.get_id = reinterpret_cast<CtxGetIdFn>(fn);
        return d;
    }();
    return q;
}

// Identity of the calling thread's current CUDA context (unique for the life
// of the process), or 0 if the driver cannot say.
unsigned long long current_context_id()
{
    const DriverQueries &q = driver_queries();
    if (!q.get_current || !q.get_id) return 0;
    void *ctx = nullptr;
    if (q.get_current(&ctx) != 0 || !ctx) return 0;
    unsigned long long id = 0;
    if (q.get_id(ctx, &id) != 0) return 0;
    return id;
}

// Device address of the array on device `dev`, which must be current.
// Looked up on the first call for that device (and again whenever the
// device's context has changed since), cached otherwise.
fc_status noalloc_workspace(int dev, void **out)
{
    char msg[256];
    if (dev < 0 || dev >= kMaxDevices) {
        snprintf(msg, sizeof(msg), "device %d is out of range", dev);
        return fc::set_error(FC_ERR_CUDA, msg);
    }
    const unsigned long long ctx = current_context_id();
    std::lock_guard<std::mutex> lock(g_mu);
    CacheEntry &e = g_cache[dev];
    if (!e.addr || ctx == 0 || e.ctx_id != ctx) {
        void *p = nullptr;
        const cudaError_t err = cudaGetSymbolAddress(&p, g_noalloc_ws);
        if (err != cudaSuccess || !p) {
            e.addr = nullptr;
            snprintf(msg, sizeof(msg), "cudaGetSymbolAddress of the built-in scratch: %s",
                     cudaGetErrorString(err));
            return fc::set_error(FC_ERR_CUDA, msg);
        }
        e.addr = p;
        // the lookup may have created the context: ask again
        e.ctx_id = ctx != 0 ? ctx : current_context_id();
    }
    *out = e.addr;
    return FC_OK;
}

}  // namespace

extern "C" {

fc_status fc_step_noalloc(const void *const *grads, int32_t W, int32_t L,
                          const int64_t *sizes, float loss_scale,
                          int64_t chunk, int64_t k, float lr, float momentum,
                          float *residual, float *a, float *velocity,
                          float *weights, void *weights_fp16, float *norms,
                          int32_t *idx, uint8_t *mask, float *packed,
                          void *packed_fp16, float send_scale,
                          float *threshold, void *stream)
{
    char msg[256];
    int64_t N = 0;
    // every argument first, so that an invalid call queues nothing
    fc_status st = fc::check_step_args(grads, W, L, sizes, loss_scale, chunk, k, lr, momentum,
                                       residual, a, velocity, weights, weights_fp16, norms, idx,
                                       mask, packed, packed_fp16, send_scale, threshold, &N);
    if (st != FC_OK) return st;
    const size_t need = fc_step_workspace_size(N, chunk);
    if (need > (size_t)FC_NOALLOC_WORKSPACE_BYTES) {
        snprintf(msg, sizeof(msg),
                 "N = %lld in chunks of %lld needs %zu bytes of scratch; the built-in "
                 "array holds %zu (use fc_step with a workspace)",
                 (long long)N, (long long)chunk, need, (size_t)FC_NOALLOC_WORKSPACE_BYTES);
        return fc::set_error(FC_ERR_LIMIT, msg);
    }
    // the device that owns the output is the one whose copy of the array is
    // used; the caller's device is current again when this call returns
    fc::DeviceScope scope;
    st = scope.bind(a);
    if (st != FC_OK) return st;
    void *ws = nullptr;
    st = noalloc_workspace(scope.device(), &ws);
    if (st != FC_OK) return st;
    // The array keeps whatever the previous call left; the one part that must
    // start at zero (the selection's count of finished blocks and the staged
    // reduction's failure word) is cleared on the stream, ahead of this
    // step's kernels.
    cudaError_t e = cudaMemsetAsync((char *)ws + fc::step_ws_counter_offset(N, chunk), 0, 256,
                                    (cudaStream_t)stream);
    if (e != cudaSuccess) {
        snprintf(msg, sizeof(msg), "cudaMemsetAsync: %s", cudaGetErrorString(e));
        return fc::set_error(FC_ERR_CUDA, msg);
    }
    return fc_step(grads, W, L, sizes, loss_scale, chunk, k, lr, momentum,
                   residual, a, velocity, weights, weights_fp16, norms, idx,
                   mask, packed, packed_fp16, send_scale, threshold, ws, need,
                   stream);
}

}  // extern "C"
