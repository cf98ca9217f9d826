/*
 * fc.h — C ABI of the GB300 gradient-aggregation engine (libfc.so).
 *
 * One data-parallel step as FireCaffe and GradientFlow describe it, run on
 * one GPU where W simulated workers' gradients already sit in HBM:
 *
 *   a1 fuse     concatenate each worker's per-layer fp16 gradients into one
 *               buffer (GradientFlow, "Optimizing Network Performance for
 *               Distributed DNN Training on GPU Clusters", arXiv 1902.06855,
 *               abstract: lazy allreduce fuses many communication operations
 *               into a single one)
 *   a2 reduce   element-wise sum over the workers (FireCaffe, "near-linear
 *               acceleration of deep neural network training on compute
 *               clusters", arXiv 1511.00175, §6: allreduce of vectors of
 *               length |dW|) in a binary reduction tree (same §6: its depth
 *               is the base-2 log of the worker count), accumulated in fp32
 *               (mixed precision, GradientFlow abstract) and unscaled by
 *               1/(loss scale * W)
 *   a3 norms    L2 norm of every fixed-size chunk of the fused vector
 *   a4 select   keep the k highest-norm chunks and compact them (GradientFlow
 *               abstract: coarse-grained sparse communication sends only the
 *               chunks that matter)
 *   a5 update   carry unkept values in an fp32 residual; momentum SGD on the
 *               fp32 master weights (FireCaffe §3 batched SGD, §6 each worker
 *               applies the summed update)
 *
 * Readings of points the pages leave open (each implemented exactly):
 *  - tree pairing: adjacent pairs (0,1),(2,3),... level by level; an odd last
 *    element moves up unchanged;
 *  - a[i] = tree_sum[i] * u + r[i] with u = binary32 nearest 1/(S*W), the
 *    residual r added after the unscale (so it can promote a chunk);
 *  - chunks run over the fused vector across layer boundaries; the last
 *    chunk may be short; its score is its plain L2 norm;
 *  - k chunks are kept; the order is larger norm first, equal norms lower
 *    index first; k = ceil(C * num / den), at least 1;
 *  - update (per element, kept = chunk of i is kept; every operation one
 *    binary32 rounding, no FMA):
 *        g = kept ? a : 0;  r = kept ? 0 : a;
 *        v = momentum*v + lr*g;  w = w - v;  w16 = fp16_rne(w) (optional).
 *
 * Conventions for every call:
 *  - Device pointers are CUDA device (or managed) memory owned by the caller;
 *    host pointers are marked "host".  The library allocates nothing at run
 *    time.  Its state between calls is the thread-local error message,
 *    launch sizes cached per kernel and device, and the scratch array built
 *    into the library for fc_step_noalloc (with its address per device).
 *  - `stream` is a cudaStream_t (NULL = the legacy default stream).  Calls
 *    are asynchronous and stream-ordered; a returned FC_OK means the
 *    arguments were valid and the kernels were launched, not that they
 *    finished.  No call except fc_step_status synchronises or queries the
 *    stream, so sequences can be captured in a CUDA graph (after one call
 *    outside capture has cached the launch configuration).  Kernels run on
 *    the device that owns the call's main device buffer (the output for
 *    most calls); the caller's current device is the same after the call as
 *    before it.
 *  - fp32 arrays and fp16 outputs must be 16-byte aligned; fp16 gradient
 *    inputs must be 2-byte aligned.  Otherwise FC_ERR_ALIGNMENT.  Which
 *    phase-1 kernel a layout of gradients gets (and so its speed, never its
 *    result) depends on their alignment: fc_step_reduce_kernel says which.
 *  - Aliasing: only the pairs stated per call may alias.
 *  - Inputs are assumed finite (no inf/NaN in the gradients).
 *  - On error nothing is launched and fc_last_error() describes the cause.
 *  - No kernel waits on the host.  Only the cooperative one-launch step's
 *    CTAs wait on one another (all resident by the cooperative launch), and
 *    every wait on the device is bounded (2 s), so no call can hang.
 */
#ifndef FC_H_
#define FC_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define FC_API __attribute__((visibility("default")))
#else
#define FC_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum fc_status {
    FC_OK = 0,
    FC_ERR_INVALID_ARG = -1, /* null pointer, size or count out of range */
    FC_ERR_ALIGNMENT = -2,   /* a pointer breaks the alignment rule above */
    FC_ERR_WORKSPACE = -3,   /* workspace missing or smaller than required */
    FC_ERR_CUDA = -4,        /* a CUDA runtime call or launch failed */
    FC_ERR_TIMEOUT = -5,     /* a bounded wait on the device ran out: the
                                step was not applied (fc_step_status) */
    FC_ERR_LIMIT = -6        /* a table or size exceeds a fixed capacity */
} fc_status;

/* Largest W*L and L that fc_fuse_pack / fc_step_reduce / fc_step accept in
 * one call (the worker-layer pointer table travels as a kernel parameter). */
#define FC_MAX_TABLE_PTRS 3072
#define FC_MAX_TABLE_LAYERS 512

/* Message for the last error on the calling thread ("" if none).  The string
 * is owned by the library and valid until the next call on this thread. */
FC_API const char *fc_last_error(void);

/* Library ABI version (100 * major + minor). */
FC_API int32_t fc_version(void);

/* ---- host-only helpers (no GPU needed) ---------------------------------- */

/* C = ceil(N / chunk): number of chunks of `chunk` elements over a fused
 * vector of N elements (the last one may be short).  Returns -1 if N < 0 or
 * chunk < 1. */
FC_API int64_t fc_num_chunks(int64_t N, int64_t chunk);

/* k = ceil(C * keep_num / keep_den) in integers, clamped to [1, C]: how many
 * chunks the top fraction keep_num/keep_den keeps.  Returns -1 if C < 1,
 * keep_num < 0 or keep_den < 1. */
FC_API int64_t fc_keep_count(int64_t C, int64_t keep_num, int64_t keep_den);

/* Layout of the fused buffer (a1): offsets[l] = sizes[0] + ... + sizes[l-1]
 * (host arrays of L entries), layers in the given order with no padding;
 * *N_out (host) = sum of the sizes.  Sizes must be >= 0 with a positive
 * sum. */
FC_API fc_status fc_layout(int32_t L, const int64_t *sizes, int64_t *offsets,
                           int64_t *N_out);

/* ---- a1: fuse --------------------------------------------------------------- */

/* Copies W workers' L per-layer fp16 gradients into the fused buffer:
 *   fused[w*N + offsets[l] + j] = grads[w*L + l][j],  0 <= j < sizes[l].
 *  grads    host array of W*L device pointers to fp16, worker-major
 *           (grads[w*L + l] is worker w's layer l); 2-byte aligned.
 *  sizes    host [L] element counts (>= 0, sum N >= 1).
 *  offsets  host [L] output (may be NULL): the layout as in fc_layout.
 *  fused    device fp16 [W*N] output, 16-byte aligned; must not overlap the
 *           gradients.
 * W >= 1, L >= 1, W*L <= FC_MAX_TABLE_PTRS, L <= FC_MAX_TABLE_LAYERS. */
FC_API fc_status fc_fuse_pack(const void *const *grads, int32_t W, int32_t L,
                              const int64_t *sizes, int64_t *offsets, void *fused,
                              void *stream);

/* ---- a2: binary-tree reduction ---------------------------------------------- */

/* out[i] = tree_{w=0..W-1}(fp32(fused[w*N + i])) * u  (+ residual_in[i]),
 * u = binary32 nearest 1/(loss_scale*W), the tree as in the readings above.
 *  fused        device fp16 [W*N] (row w = worker w), 2-byte aligned
 *               (16-byte aligned with N % 8 == 0 takes the vector path).
 *  residual_in  device fp32 [N] or NULL (then nothing is added).
 *  out          device fp32 [N]; may alias residual_in (in place).
 * 1 <= W <= FC_MAX_TABLE_PTRS, N >= 1, loss_scale finite and > 0. */
FC_API fc_status fc_tree_reduce(const void *fused, int32_t W, int64_t N,
                                float loss_scale, const float *residual_in,
                                float *out, void *stream);

/* Summation orders over the workers.  The engine's method is the binary
 * tree; the other two are the aggregation schemes the pages set the tree
 * against, with the same operations in another order (results differ from
 * the tree's by fp32 rounding only):
 *  FC_ORDER_TREE        FireCaffe §6 reduction tree (as above);
 *  FC_ORDER_SEQUENTIAL  parameter server (FireCaffe §6: one node receives
 *                       and sums every worker's gradient): ((x0+x1)+x2)+...;
 *  FC_ORDER_RING        ring reduce-scatter (GradientFlow abstract, ring-
 *                       based allreduce): the fused vector is cut into W
 *                       segments [floor(s*N/W), floor((s+1)*N/W)); the sum of
 *                       segment s starts at worker s and goes round the ring:
 *                       ((x_s + x_{s+1}) + ...) + x_{s-1}, indices mod W. */
#define FC_ORDER_TREE 0
#define FC_ORDER_SEQUENTIAL 1
#define FC_ORDER_RING 2

/* fc_tree_reduce with a selectable summation order (FC_ORDER_*); the
 * FC_ORDER_TREE result is bit-identical to fc_tree_reduce. */
FC_API fc_status fc_reduce_ordered(const void *fused, int32_t W, int64_t N,
                                   float loss_scale, const float *residual_in,
                                   float *out, int32_t order, void *stream);

/* ---- a3: chunk norms ---------------------------------------------------------- */

/* norms[c] = sqrt(sum_{i in chunk c} a[i]^2), c < C = fc_num_chunks(N, chunk).
 * Squares and partial sums in fp32 over units of at most 256 elements
 * (pairs of 8, then a warp butterfly), the unit sums added in float-float
 * (compensated fp32) arithmetic in a fixed order, then a correctly rounded
 * fp32 square root; the relative error is below 6e-7.  Deterministic: the
 * same inputs give the same bits, and the same bits as the pipeline's
 * fc_step_select.
 *  a      device fp32 [N].
 *  norms  device fp32 [C] output. */
FC_API fc_status fc_chunk_norms(const float *a, int64_t N, int64_t chunk,
                                float *norms, void *stream);

/* ---- a4: top-k selection and compaction -------------------------------------- */

/* Bytes of caller workspace fc_chunk_select needs for C chunks: always 0.
 * The selection keeps its histogram and scan state in shared memory of one
 * block (the norms too, up to 11264 chunks; more are re-read from `norms`),
 * so the call takes no workspace argument.  Returns 0 for any C. */
FC_API size_t fc_chunk_select_workspace(int64_t C);

/* Keeps the k chunks that come first in (norm descending, index ascending)
 * order, found by a radix select on the norms' bit patterns.
 *  norms      device fp32 [C], finite and >= 0.
 *  a, N, chunk  the reduced gradient the norms were taken over (a device fp32
 *             [N]); only read when a send buffer is asked for.
 *  idx        device int32 [k] output: kept chunk indices, ascending.
 *  mask       device uint8 [C] output: 1 = kept.
 *  packed     device fp32 [k*chunk] output or NULL: the send buffer, kept
 *             chunks' values of a in idx order, one `chunk`-float slot each,
 *             the short last chunk zero-padded.
 *  packed_fp16  device fp16 [k*chunk] output or NULL: the same send buffer
 *             in fp16 (GradientFlow abstract: mixed-precision communication),
 *             fp16_rne(value * send_scale); send_scale (finite) typically
 *             puts the values back in fp16 range, e.g. the loss scale.
 *  threshold  device fp32 [1] output: the norm of the k-th kept chunk.
 * 1 <= k <= C. */
FC_API fc_status fc_chunk_select(const float *norms, int64_t C, int64_t k,
                                 const float *a, int64_t N, int64_t chunk,
                                 int32_t *idx, uint8_t *mask, float *packed,
                                 void *packed_fp16, float send_scale,
                                 float *threshold, void *stream);

/* ---- a5: residual fold and momentum SGD ---------------------------------------- */

/* Per element i (kept = mask[i / chunk] != 0), as in the readings above:
 *   residual = kept ? 0 : a;  velocity = momentum*velocity + lr*(kept ? a : 0);
 *   weights -= velocity;      weights_fp16 = fp16_rne(weights) if not NULL.
 *  a             device fp32 [N]; may alias residual.
 *  mask          device uint8 [C].
 *  residual, velocity, weights  device fp32 [N], updated in place.
 *  weights_fp16  device fp16 [N] output or NULL. */
FC_API fc_status fc_residual_sgd_update(const float *a, const uint8_t *mask,
                                        int64_t N, int64_t chunk, float lr,
                                        float momentum, float *residual,
                                        float *velocity, float *weights,
                                        void *weights_fp16, void *stream);

/* ---- the fused pipeline (a1..a5 without materialising the fused buffer) ---- */

/* Bytes of scratch the pipeline needs for N elements in chunks of `chunk`
 * (per-unit sums of squares, a count of finished selection blocks and the
 * kept-slot map); 0 on bad arguments.  The workspace must be zero-filled
 * before its first use with a given (N, chunk), e.g. by cudaMemsetAsync;
 * every pipeline step leaves the count at zero again. */
FC_API size_t fc_step_workspace_size(int64_t N, int64_t chunk);

/* Phase 1 of the pipeline: a2 and the per-unit sums of squares of a3,
 * reading every worker's layer tensors in place through the layout of a1
 * (the fused buffer itself is never written):
 *   a[f] = tree_w(grads[w*L + l][f - offsets[l]]) * u + residual[f]
 * for every fused index f in layer l.  `a` is bit-identical to
 * fc_fuse_pack + fc_tree_reduce.
 *  grads, W, L, sizes  as for fc_fuse_pack.
 *  residual  device fp32 [N] or NULL.
 *  a         device fp32 [N] output; may alias residual (in place).
 *  workspace device, fc_step_workspace_size(N, chunk) bytes, 256-aligned,
 *            zero-filled before first use. */
FC_API fc_status fc_step_reduce(const void *const *grads, int32_t W, int32_t L,
                                const int64_t *sizes, float loss_scale,
                                int64_t chunk, const float *residual, float *a,
                                void *workspace, size_t workspace_bytes,
                                void *stream);

/* fc_step_reduce with a selectable summation order (FC_ORDER_*); the
 * FC_ORDER_TREE call is fc_step_reduce. */
FC_API fc_status fc_step_reduce_ordered(const void *const *grads, int32_t W,
                                        int32_t L, const int64_t *sizes,
                                        float loss_scale, int64_t chunk,
                                        const float *residual, float *a,
                                        int32_t order, void *workspace,
                                        size_t workspace_bytes, void *stream);

/* Phase 1 on a span of the fused vector, so that the reduction of early
 * layer groups overlaps the arrival of later ones (GradientFlow abstract:
 * computation/communication overlap; backprop hands the layers over last
 * layer first).  Reduces exactly the 256-element units (unit = up to 256
 * elements of one chunk, the j-th starting at chunk start + 256 j) whose
 * first element lies in [f_begin, f_end): `a` for every element of those
 * units and their sums of squares in the workspace, as fc_step_reduce
 * does.  Calls whose spans partition [0, N) leave `a` and the workspace
 * exactly as one fc_step_reduce call does (same bits, any call order);
 * fc_step_select and fc_step_update then finish the step.
 *  A unit that starts in the span may end up to 255 elements after f_end
 *  (never past its chunk), so every layer overlapping
 *  [f_begin, fc_unit_start of the span's last unit + 256) must hold its
 *  gradients when the call runs on the stream.  For layer groups arriving
 *  last layer first, [group start, group end) is such a span; for groups
 *  arriving first layer first, [fc_unit_start(group start),
 *  fc_unit_start(group end)) is.
 *  Tree order only.  0 <= f_begin <= f_end <= N, else FC_ERR_INVALID_ARG;
 *  an empty span launches nothing.  Other arguments as fc_step_reduce. */
FC_API fc_status fc_step_reduce_span(const void *const *grads, int32_t W,
                                     int32_t L, const int64_t *sizes,
                                     float loss_scale, int64_t chunk,
                                     const float *residual, float *a,
                                     int64_t f_begin, int64_t f_end,
                                     void *workspace, size_t workspace_bytes,
                                     void *stream);

/* First element of the unit (see fc_step_reduce_span) that holds fused
 * element f: chunk start + 256 * floor(offset in chunk / 256), for
 * 0 <= f < N; N for f == N; -1 for any other argument. */
FC_API int64_t fc_unit_start(int64_t N, int64_t chunk, int64_t f);

/* Which phase-1 kernel fc_step_reduce_ordered (and so fc_step) launches for
 * this layout of gradients (arguments as there; chunk > 0, order an
 * FC_ORDER_* value).  Host only: the pointers are compared, never read, and
 * no device work is done.  Returns FC_REDUCE_* below, or -1 (message in
 * fc_last_error) for arguments the reduction would reject.  The kernels
 * produce the same bits; the choice only changes speed.
 *  FC_REDUCE_REGISTER        register streaming, one warp per 256-element unit;
 *  FC_REDUCE_STAGED          bulk copies staged in shared memory, every layer
 *                            at a multiple of 8 elements and 16-byte aligned
 *                            for every worker (4, 8 or 16 workers), fewer
 *                            than 1536 tiles of 2048 elements;
 *  FC_REDUCE_STAGED_SHIFTED  the same for layers at any offset whose address
 *                            modulo 16 bytes, at a given fused index, is the
 *                            same for every worker; also taken by aligned
 *                            layouts of at least 8192 tiles.
 * Aligned layouts from 1536 to 8191 tiles take FC_REDUCE_REGISTER: there it
 * measured faster than either staged variant. */
#define FC_REDUCE_REGISTER 0
#define FC_REDUCE_STAGED 1
#define FC_REDUCE_STAGED_SHIFTED 2
FC_API int32_t fc_step_reduce_kernel(const void *const *grads, int32_t W,
                                     int32_t L, const int64_t *sizes,
                                     int64_t chunk, int32_t order);

/* Phase 2: finishes the chunk norms from phase 1's unit sums (norms [C],
 * device output, bitwise the same as fc_chunk_norms on a) and selects the
 * top k chunks exactly as fc_chunk_select does (idx [k], mask [C],
 * threshold [1] are device outputs); each kept chunk's slot in the packed
 * output goes to the workspace for phase 3. */
FC_API fc_status fc_step_select(int64_t N, int64_t chunk, int64_t k,
                                float *norms, int32_t *idx, uint8_t *mask,
                                float *threshold, void *workspace,
                                size_t workspace_bytes, void *stream);

/* Phase 3: the a5 update of fc_residual_sgd_update, which also writes the
 * kept chunks into the send buffers `packed` (device fp32 [k*chunk] or NULL)
 * and `packed_fp16` (device fp16 [k*chunk] or NULL, values times
 * send_scale), laid out as in fc_chunk_select.  `mask` must be the one
 * phase 2 wrote.  When a == residual (in place), unkept elements already
 * hold their new residual and are neither read nor rewritten. */
FC_API fc_status fc_step_update(const float *a, int64_t N, int64_t chunk,
                                float lr, float momentum, float *residual,
                                float *velocity, float *weights,
                                void *weights_fp16, const uint8_t *mask,
                                float *packed, void *packed_fp16,
                                float send_scale, void *workspace,
                                size_t workspace_bytes, void *stream);

/* Outcome of the last pipeline step (fc_step, or fc_step_select and
 * fc_step_update after phase 1) that used this workspace, read after
 * `stream` has finished: the call copies one word back and synchronises
 * the stream, so it is not for use while the stream is being captured.
 *  FC_OK           the step was applied;
 *  FC_ERR_TIMEOUT  a bounded wait inside the staged phase 1 ran out (not
 *                  expected in normal operation: each wait allows 2 s).
 *                  The step was then not applied: phase 2 reported a NaN
 *                  threshold, an empty mask and idx = -1, and phase 3 left
 *                  velocity, weights, the fp16 weights and the send buffers
 *                  as they were.  With a separate `a` buffer the residual is
 *                  unchanged too, so the step can simply be run again; in
 *                  place (a == residual) phase 1 had already overwritten the
 *                  residual with a for the tiles it reduced, so restore the
 *                  residual before running the step again.  The same status
 *                  comes from a one-launch step (FC_STEP_ONE_LAUNCH) whose
 *                  grid barrier wait ran out: nothing but `a`, the norms and
 *                  the unit sums was written, and the barrier's arrival
 *                  count is left part-way, so zero the workspace again (as
 *                  before its first use) before the next step.
 * Other statuses: bad arguments or a failed CUDA call. */
FC_API fc_status fc_step_status(const void *workspace, size_t workspace_bytes,
                                int64_t N, int64_t chunk, void *stream);

/* Phases 1-3 in one call on one stream.  Small problems run as one launch
 * (see fc_step_path); all others as the three kernels of fc_step_reduce,
 * fc_step_select and fc_step_update.  All give the same bits.  If the
 * device refuses the one launch as too large for it (for instance a context
 * limited to a share of the SMs), the call takes the three kernels
 * instead. */
FC_API fc_status fc_step(const void *const *grads, int32_t W, int32_t L,
                         const int64_t *sizes, float loss_scale, int64_t chunk,
                         int64_t k, float lr, float momentum, float *residual,
                         float *a, float *velocity, float *weights,
                         void *weights_fp16, float *norms, int32_t *idx,
                         uint8_t *mask, float *packed, void *packed_fp16,
                         float send_scale, float *threshold, void *workspace,
                         size_t workspace_bytes, void *stream);

/* How fc_step runs a problem of this layout on the current device:
 *  FC_STEP_THREE_KERNELS  the three kernels of fc_step_reduce,
 *                         fc_step_select and fc_step_update;
 *  FC_STEP_ONE_LAUNCH     one cooperative launch with one CTA per SM that
 *                         runs all three phases, with a grid barrier in the
 *                         workspace after the norms (bounded waits) and the
 *                         k-th chunk handed to every CTA through one word;
 *  FC_STEP_ONE_CLUSTER    where the device runs no cooperative launch: one
 *                         launch of one thread-block cluster (16 CTAs where
 *                         the GPU can schedule them, else 8) with hardware
 *                         cluster barriers between the phases.
 * The one-launch forms serve chunk sizes that are multiples of 8, up to
 * 1024 chunks, up to 2^19 elements, up to 64 workers, and up to 8
 * 256-element units per warp.  Returns -1 for arguments fc_step would
 * reject.  Queries the device (occupancy, cooperative launch) on its first
 * call per device; without a device the answer is FC_STEP_THREE_KERNELS.
 * While fc_test_stage_loss is armed, fc_step takes the three kernels
 * whatever this returns. */
#define FC_STEP_THREE_KERNELS 0
#define FC_STEP_ONE_LAUNCH 1
#define FC_STEP_ONE_CLUSTER 2
FC_API int32_t fc_step_path(const void *const *grads, int32_t W, int32_t L,
                            const int64_t *sizes, int64_t chunk);

/* ---- the pipeline without a caller workspace ---------------------------------- */

/* Size of the scratch array built into the library for fc_step_noalloc. */
#define FC_NOALLOC_WORKSPACE_BYTES (4u << 20)

/* fc_step for callers that cannot allocate device memory when they step:
 * code running while a stream is captured into a CUDA graph (cudaMalloc is
 * not allowed then), frameworks whose pool allocator owns every device byte,
 * and latency-critical loops that forbid allocation after start-up.  The
 * pages have no counterpart to this call: it only changes where the scratch
 * lives.
 *
 * Arguments and results are those of fc_step without the workspace.  The
 * scratch is a FC_NOALLOC_WORKSPACE_BYTES (4 MiB) array inside the library,
 * which every GPU that loads libfc holds until the process exits; a problem
 * whose fc_step_workspace_size(N, chunk) exceeds it gets FC_ERR_LIMIT and
 * nothing runs (4 MiB covers about 260 million elements in chunks that are
 * multiples of 256).  The call allocates nothing: no cudaMalloc, no
 * cudaFree, no allocating library routine.
 *
 * Every argument is checked before anything is queued on `stream`, so an
 * invalid call queues nothing.
 *
 * The array's device address is looked up (cudaGetSymbolAddress) with the
 * output's device current, and cached together with the identity of that
 * device's current CUDA context.  The first call on a device, and the first
 * call after cudaDeviceReset (which destroys the context and so moves the
 * array), do the lookup: make those calls before capturing a stream.  Every
 * call shares the one array per device and finds it as the last call left
 * it: it clears the part that must start at zero on `stream` before its
 * kernels, but two calls whose work overlaps on the GPU (different streams
 * without ordering between them) race on the array and give wrong results.
 * A failed step (FC_ERR_TIMEOUT in fc_step_status) shows here as a NaN
 * threshold with idx = -1. */
FC_API fc_status fc_step_noalloc(const void *const *grads, int32_t W,
                                 int32_t L, const int64_t *sizes,
                                 float loss_scale, int64_t chunk, int64_t k,
                                 float lr, float momentum, float *residual,
                                 float *a, float *velocity, float *weights,
                                 void *weights_fp16, float *norms,
                                 int32_t *idx, uint8_t *mask, float *packed,
                                 void *packed_fp16, float send_scale,
                                 float *threshold, void *stream);

/* ---- test hook ------------------------------------------------------------------- */

/* Exercises the failure path of the TMA-staged phase 1 (not part of the
 * method).  Arms the next TMA-staged launch (4, 8 or 16 workers, aligned or
 * shifted layout) to issue no copies for fused tile `tile` (2048 elements),
 * with every wait of that launch bounded by wait_limit_ns (1 ms .. 2 s)
 * instead of 2 s.  The waits on that tile then run out, the kernel records
 * the failure in the workspace and returns, and phase 2 reports it: the
 * threshold is NaN, no chunk is kept and idx is -1; the record is cleared,
 * so the following steps run normally.  tile < 0 disarms the hook.  Host
 * only; the next launch from any thread consumes it. */
FC_API fc_status fc_test_stage_loss(int64_t tile, uint64_t wait_limit_ns);

/* Test hooks for the one-launch step (not part of the method).
 * fc_test_one_launch_kind(FC_STEP_ONE_CLUSTER) makes fc_step and
 * fc_step_path use the cluster form even where the cooperative one runs;
 * FC_STEP_ONE_LAUNCH restores the default.  Other values:
 * FC_ERR_INVALID_ARG.  Process-wide, host only. */
FC_API fc_status fc_test_one_launch_kind(int32_t kind);

/* Arms the next cooperative one-launch step: CTA `cta` (clamped to the
 * last) gives up before the grid barrier, and the other CTAs wait for it at
 * most wait_limit_ns (0 < limit <= 10 s) instead of 2 s.  Their waits then
 * run out and the step is not applied: fc_step_status reports
 * FC_ERR_TIMEOUT, and the workspace must be zeroed again before the next
 * step.  cta < 0 disarms.  Host only; the next such launch from any thread
 * consumes it. */
FC_API fc_status fc_test_barrier_loss(int32_t cta, uint64_t wait_limit_ns);

#ifdef __cplusplus
}
#endif

#endif /* FC_H_ */
