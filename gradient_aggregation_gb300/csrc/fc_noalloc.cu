// fc_step_noalloc: the fused pipeline with its scratch in a fixed device
// array that ships inside libfc, for callers that cannot allocate device
// memory when they step.
//
// The array below is a file-scope __device__ variable: every GPU that loads
// the library holds FC_NOALLOC_WORKSPACE_BYTES of it until the process exits.
// In host code the name `g_noalloc_ws` is only a host-side stand-in, not a
// device address, so the device address is looked up once per device with
// cudaGetSymbolAddress while that device is current, checked, and cached.
#include <stdio.h>

#include <mutex>

#include "fc.h"
#include "fc_internal.h"

namespace {

__device__ __align__(256) unsigned char g_noalloc_ws[FC_NOALLOC_WORKSPACE_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void *g_addr[kMaxDevices];

// Device address of the array on device `dev`, which must be current.
// Looked up on the first call for that device and cached afterwards.
fc_status noalloc_workspace(int dev, void **out)
{
    char msg[256];
    if (dev < 0 || dev >= kMaxDevices) {
        snprintf(msg, sizeof(msg), "device %d is out of range", dev);
        return fc::set_error(FC_ERR_CUDA, msg);
    }
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_addr[dev]) {
        void *p = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_ws);
        if (e != cudaSuccess || !p) {
            snprintf(msg, sizeof(msg), "cudaGetSymbolAddress of the built-in scratch: %s",
                     cudaGetErrorString(e));
            return fc::set_error(FC_ERR_CUDA, msg);
        }
        g_addr[dev] = p;
    }
    *out = g_addr[dev];
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
    fc_status st = fc_layout(L, sizes, nullptr, &N);
    if (st != FC_OK) return st;
    if (chunk < 1) return fc::set_error(FC_ERR_INVALID_ARG, "chunk must be >= 1");
    const size_t need = fc_step_workspace_size(N, chunk);
    if (need > (size_t)FC_NOALLOC_WORKSPACE_BYTES) {
        snprintf(msg, sizeof(msg),
                 "N = %lld in chunks of %lld needs %zu bytes of scratch; the built-in "
                 "array holds %zu (use fc_step with a workspace)",
                 (long long)N, (long long)chunk, need, (size_t)FC_NOALLOC_WORKSPACE_BYTES);
        return fc::set_error(FC_ERR_LIMIT, msg);
    }
    if (!a) return fc::set_error(FC_ERR_INVALID_ARG, "a is NULL");
    // the device that owns the output is the one whose copy of the array is used
    cudaPointerAttributes at;
    cudaError_t e = cudaPointerGetAttributes(&at, a);
    if (e != cudaSuccess) {
        snprintf(msg, sizeof(msg), "cudaPointerGetAttributes: %s", cudaGetErrorString(e));
        return fc::set_error(FC_ERR_CUDA, msg);
    }
    if (at.type != cudaMemoryTypeDevice && at.type != cudaMemoryTypeManaged)
        return fc::set_error(FC_ERR_INVALID_ARG, "a is not device memory");
    e = cudaSetDevice(at.device);
    if (e != cudaSuccess) {
        snprintf(msg, sizeof(msg), "cudaSetDevice: %s", cudaGetErrorString(e));
        return fc::set_error(FC_ERR_CUDA, msg);
    }
    void *ws = nullptr;
    st = noalloc_workspace(at.device, &ws);
    if (st != FC_OK) return st;
    // The array keeps whatever the previous call left; the one part that must
    // start at zero (the selection's count of finished blocks) is cleared on
    // the stream, ahead of this step's kernels.
    e = cudaMemsetAsync((char *)ws + fc::step_ws_counter_offset(N, chunk), 0, 256,
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
