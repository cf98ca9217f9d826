// Launchers shared between the engine's translation units (not exported).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "fc.h"
#include "fc_common.cuh"

namespace fc {

// Builds a table; returns false if it does not fit the given tier.
template <class Tab>
bool fill_table(Tab &t, const void *const *grads, int32_t W, int32_t L,
                const int64_t *sizes);

// Phase-1 / fc_tree_reduce kernel launch over units [ub, ue) (ue < 0: all).
// With partials != NULL the unit sums of squares go to partials [G.units].
// order: FC_ORDER_* of fc.h.
template <class Tab>
cudaError_t launch_reduce(const Tab &tab, const UnitGeom &G, float u,
                          const float *resid, float *out, float *partials,
                          cudaStream_t s, int order = 0, int64_t ub = 0,
                          int64_t ue = -1);

// TMA-staged phase 1 (tree order only).  tma_layout: 0 if the layout does
// not allow it, 1 for the aligned layout, 2 for the shifted one (layers at
// any offset, one address shift per layer for all workers).  ctr: the
// pipeline workspace's 256-byte block of counter words (zero on entry and
// on exit but for word 1, which is set if a wait inside the kernel gave up).
template <class Tab>
int tma_layout(const Tab &tab, const UnitGeom &G, const float *partials);
// The staged kernel works on whole 256-element units: fused elements
// [fb, fe) with fb a multiple of 256 and fe a multiple of 256 or N (fe < 0:
// N).
template <class Tab>
cudaError_t launch_reduce_tma(const Tab &tab, const UnitGeom &G, float u,
                              const float *resid, float *out, float *partials,
                              unsigned *ctr, cudaStream_t s, int layout, int64_t fb = 0,
                              int64_t fe = -1);

template <class Tab>
cudaError_t launch_pack(const Tab &tab, int64_t N, __half *fused,
                        cudaStream_t s);

cudaError_t launch_norms(const float *a, const UnitGeom &G, float *norms,
                         cudaStream_t s);

// With partials == NULL, norms [C] is the input.  Otherwise the chunk
// norms are first formed from the unit sums (partials [G.units]) by many
// blocks and written to norms; `done` (zero on entry, zero on exit) counts
// finished blocks and the last one selects.  slot may be NULL.  err: the
// staged reduction's failure word (read and cleared); status: the step's
// outcome word, written with 0 (applied) or 1 (not applied: a wait ran out).
cudaError_t launch_select(const UnitGeom &G, const float *partials,
                          unsigned *done, float *norms, int64_t k,
                          int32_t *idx, uint8_t *mask, int32_t *slot,
                          float *threshold, cudaStream_t s,
                          unsigned *err = nullptr, unsigned *status = nullptr);

cudaError_t launch_gather(const float *a, int64_t N, int64_t cs, int64_t P,
                          const int32_t *idx, int64_t k, float *packed,
                          __half *packed16, float send_scale, cudaStream_t s);

// status (may be NULL): the step's outcome word written by the selection;
// when it is non-zero the update writes nothing.
cudaError_t launch_update(const TileGeom &G, int64_t tiles, const float *a,
                          const uint8_t *mask, const int32_t *slot,
                          float *packed, __half *packed16, float send_scale,
                          float lr, float mu, float *r, float *v, float *w,
                          __half *w16, bool inplace, cudaStream_t s,
                          const unsigned *status = nullptr);

// ---- fc_step in one launch (small problems) ------------------------------------

// The one-launch path serves chunk sizes that are multiples of 8, at most
// FC_SMALL_MAX_CHUNKS chunks, at most FC_SMALL_MAX_N elements, at most 64
// workers, and at most FC_SMALL_UNITS_PER_WARP 256-element units per warp of
// the cluster.
#define FC_SMALL_MAX_CHUNKS 1024
#define FC_SMALL_MAX_N (1 << 19)
#define FC_SMALL_UNITS_PER_WARP 8

struct SmallStep {
    UnitGeom G;
    float u;                 // binary32 nearest 1/(S*W)
    const float *resid;      // may be NULL
    float *a, *partials, *norms;
    int64_t k;
    int32_t *idx;
    uint8_t *mask;
    float *threshold;
    unsigned *status;        // the workspace's step-outcome word
    float lr, mu;
    float *r, *v, *w;
    __half *w16;
    float *packed;
    __half *packed16;
    float send_scale;
    unsigned *bar;           // five workspace words for the grid kernel (64-bit
                             // barrier count, the k-th chunk and its tag),
                             // 8-byte aligned; NULL: cluster kernel only
};

// Launches the whole step as one kernel when the problem and the device
// allow it: a cooperative launch over every SM when st.bar is set and the
// device runs cooperative launches (*kind = FC_STEP_ONE_LAUNCH), else one
// thread-block cluster (FC_STEP_ONE_CLUSTER); otherwise launches nothing
// (FC_STEP_THREE_KERNELS).  With probe_only, only decides.
template <class Tab>
cudaError_t launch_step_small(const Tab &tab, const SmallStep &st, cudaStream_t s,
                              bool probe_only, int *kind);

// True while fc_test_stage_loss has armed the next staged launch (fc_step
// then takes the three-kernel path, whose phase 1 is that launch).
bool stage_loss_armed();

// Sets the calling thread's fc_last_error() message; returns st.
fc_status set_error(fc_status st, const char *msg);

// Makes the device that owns a pointer argument current for the rest of an
// entry point, and makes the caller's device current again when the scope
// ends.  Uses only queries that are legal while a stream is captured.
class DeviceScope {
public:
    DeviceScope() = default;
    DeviceScope(const DeviceScope &) = delete;
    DeviceScope &operator=(const DeviceScope &) = delete;
    ~DeviceScope();
    // FC_OK, or an error status with fc_last_error() set.
    fc_status bind(const void *device_ptr);
    int device() const { return dev_; }

private:
    int prev_ = -1;  // the caller's device, if it was changed
    int dev_ = -1;
};

// Every argument check of fc_step except the workspace; the fused length
// goes to *N_out.  Queues nothing.
fc_status check_step_args(const void *const *grads, int32_t W, int32_t L,
                          const int64_t *sizes, float loss_scale, int64_t chunk,
                          int64_t k, float lr, float momentum, const float *residual,
                          const float *a, const float *velocity, const float *weights,
                          const void *weights_fp16, const float *norms, const int32_t *idx,
                          const uint8_t *mask, const float *packed, const void *packed_fp16,
                          float send_scale, const float *threshold, int64_t *N_out);

// Byte offset, inside the pipeline workspace for (N, chunk), of the 256-byte
// word block that must be zero before a step.
size_t step_ws_counter_offset(int64_t N, int64_t chunk);

// Launches kernel<<<grid, block, smem, s>>>(args...) with programmatic
// stream serialisation allowed (the kernel must begin with
// wait_for_prior_grid()).
template <typename... KArgs, typename... Args>
cudaError_t launch_after_prior(void (*kernel)(KArgs...), unsigned grid,
                               unsigned block, size_t smem, cudaStream_t s,
                               Args... args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(block);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// Blocks to launch for a grid-stride kernel: min(work, SMs * resident).
int grid_for(const void *kernel, int block, size_t smem, int64_t work);

}  // namespace fc
