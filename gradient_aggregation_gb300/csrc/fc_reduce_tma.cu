// Phase 1 (a2 + unit sums of squares) with TMA staging, for 4, 8 or 16
// workers, N a multiple of 8 and a chunk size that is a multiple of 256.
//
// One CTA per SM (two in the cases below): a producer warp streams tiles
// of TT fused elements of all W workers (and the residual) from HBM into a
// ring of S shared-memory stages with bulk copies (cp.async.bulk, completion
// counted on an mbarrier); eight consumer warps take one 256-element unit
// each per tile, add the workers in the same binary tree as the register
// kernel (k_reduce) from shared memory, and write `a` and the unit sums of
// squares exactly as k_reduce does, so the results are bit-identical.  The
// copies keep S-1 tiles of every worker in flight per SM regardless of
// register pressure.
//
// Two layouts:
//  * aligned (MIS = false): every layer starts at a multiple of 8 fused
//    elements and every worker's copy of it is 16-byte aligned there.  Each
//    worker row of a stage holds the tile's TT elements in fused order.
//  * shifted (MIS = true): layers may start anywhere, as long as each layer's
//    address, taken modulo 16 bytes at a given fused index, is the same for
//    every worker (true for separately allocated tensors and for buckets).
//    A bulk copy must start and end on 16-byte boundaries, so each layer
//    piece of a tile lands in shared memory at the same position modulo 16
//    bytes as in global memory: element u of the tile sits at u + sh, sh =
//    the layer's shift (0..7 elements) plus a gap (a multiple of 8) that
//    keeps the pieces apart.  The producer copies the 16-byte-aligned part
//    of every piece (running past the tile's ends where the layer goes on)
//    and records the pieces in a small table in the stage.  A consumer reads
//    its 8 elements with two 16-byte shared-memory loads and a funnel shift;
//    a group across a layer boundary takes each part from its own staged
//    piece, and only groups in unstaged pieces (past the table or the row's
//    slack) or across three or more layers read their elements from global
//    memory.  Aligned layouts long enough (FC_TMA_SHIFTED_MIN_TILES) also
//    take this variant, with every shift 0: it measured faster on long
//    runs.  Aligned mid-size runs go to the register kernel instead (see
//    tma_layout).
//
// Worker halves (shifted layout, 16 workers): each tile goes through the
// ring as two stages, the first holding workers 0..7 and the second workers
// 8..15, with two CTAs per SM (each about 100 KB of stages; the residual is
// prefetched into L2 at the first stage and read by the consumers from
// there at the second).  A consumer warp keeps the first half's subtree in
// registers and adds the second's to it: in the binary tree of 16 leaves
// those two subtrees are joined last, so the bits do not change.  Two
// producers and sixteen consumer warps per SM: the GoogLeNet-shaped phase 1
// (many short layers, so many short copies per tile) went from 55.0 to
// 51.7 us; the AlexNet-shaped one was unchanged (350 us).  With 8 workers
// the halves gained nothing in phase 1 and lost 3 us in the step; there two
// CTAs per SM keep whole stages instead (two 42 KB stages each, 75 %
// carveout), which took the NiN-shaped phase 1 from 37.7 to 34.1 us and its
// step from 68.7 to 66.8 us.
//
// Tile order: CTA b takes tiles b, b + grid, b + 2 grid, ...  In long
// launches (kDynMinRounds rounds or more) that holds for all but the last
// kDynRounds rounds; the tiles after those are handed out one at a time from
// a counter in the workspace, each producer fetching its next index while it
// issues the copies of the current tile.  CTAs that stream faster (SMs
// differ in how fast their memory requests are served) then take more of
// the tail, instead of idling while the slowest CTA finishes.  Each stage
// carries the index of its tile, and a stage with index -1 tells the
// consumers that their CTA is done.  The last producer to finish leaves the
// counters at zero for the next launch.
//
// Every wait on an mbarrier gives up after a time limit (read from the
// global timer); the kernel then records the failure in the error word and
// returns, the producer first waiting (again with a limit) for the copies it
// issued.
#include <atomic>
#include <mutex>

#include "fc_internal.h"

namespace fc {

namespace {

__device__ __forceinline__ uint32_t smem_u32(const void *p)
{
    return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_test(uint32_t bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ uint64_t global_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Waits until the phase of the given parity has completed; false if that
// takes longer than limit_ns.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, uint64_t limit_ns)
{
    if (mbar_test(bar, parity)) return true;
    const uint64_t t0 = global_ns();
    while (!mbar_test(bar, parity))
        if (global_ns() - t0 > limit_ns) return false;
    return true;
}

__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void *src, uint32_t bytes,
                                         uint32_t bar)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
        "l"(src), "r"(bytes), "r"(bar)
        : "memory");
}

// Test hook (fc_test_stage_loss): a one-shot tile to drop and the wait limit
// that goes with it.
std::atomic<int64_t> g_drop_tile{-1};
std::atomic<uint64_t> g_drop_limit_ns{0};

constexpr int kConsumerWarps = 8;
constexpr int kThreads = 32 * (kConsumerWarps + 1);
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s: far beyond any tile

// Shifted layout: extra elements per worker row (room for the shifts and
// gaps of the pieces), and entries of a stage's piece table.  A tile whose
// pieces need more room, or more entries, leaves the rest unstaged (read
// from global memory by the consumers).
constexpr int kSlack = 64;

// Aligned layouts of at least FC_TMA_SHIFTED_MIN_TILES tiles take the
// shifted variant; from FC_TMA_REGISTER_MIN_TILES up to that, the register
// kernel; shorter ones the aligned variant.
#ifndef FC_TMA_SHIFTED_MIN_TILES
#define FC_TMA_SHIFTED_MIN_TILES 8192
#endif
#ifndef FC_TMA_REGISTER_MIN_TILES
#define FC_TMA_REGISTER_MIN_TILES 1536
#endif
constexpr int kMaxPieces = 32;

// Launches of at least kDynMinRounds rounds of tiles (one tile per CTA a
// round) hand out the tiles of their last kDynRounds rounds dynamically.
// Shorter launches stay cyclic to the end: measured, the dynamic tail cost
// them more than it saved (7M elements x 16 workers: 55.1 -> 56.2 us with
// two rounds; no gain with 2 to 6 rounds once the first index is fetched
// early), while a 62M-element step gained 525 -> 518 us going from two
// dynamic rounds to eight.
constexpr int64_t kDynRounds = 8;
constexpr int64_t kDynMinRounds = 64;

// Bytes at the end of each stage that carry the stage's tile index (a whole
// 128-byte line, so that every stage starts 128-byte aligned).
constexpr int kStageHead = 128;

__device__ __forceinline__ int64_t round_down8(int64_t x) { return x & ~(int64_t)7; }
__device__ __forceinline__ int64_t round_up8(int64_t x) { return (x + 7) & ~(int64_t)7; }

// Shift, in elements (0..7), of layer l: its worker-0 address at fused
// index 0 modulo 16 bytes, halved.
template <class Tab>
__device__ __forceinline__ int layer_shift(const Tab &tab, int l)
{
    return (int)((((uintptr_t)tab.ptr[l]) - 2u * (uintptr_t)tab.off[l]) >> 1) & 7;
}

}  // namespace

// ctr: the workspace's 256-byte block of counter words: [1] the error word,
// [4..5] the 64-bit counter of dynamically handed-out tiles, [6] the count
// of producers that have finished with it (all zero between launches).
// drop_tile >= 0 (test hook only, see fc_test_stage_loss): the producer
// issues no copies for that tile, so the bounded waits on it run out.
template <class Tab, int WT, int MAXH, bool MIS, int NH, int CPS>
__global__ void __launch_bounds__(kThreads, CPS)
    k_reduce_tma(const __grid_constant__ Tab tab, const UnitGeom G, const int TT,
                 const int S, const float u, const float *resid, float *out,
                 float *partials, unsigned *ctr, const int64_t drop_tile,
                 const uint64_t limit_ns, const int64_t f_begin, const int64_t f_end)
{
    static_assert(NH == 1 || (MIS && WT == 16 && CPS == 2),
                  "worker halves: shifted layout, 16 workers, two CTAs per SM");
    extern __shared__ __align__(128) unsigned char smem[];
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem);  // full[S], empty[S]
    unsigned char *stages = smem + 128;
    unsigned *err = ctr + 1;
    unsigned long long *dyn_next = reinterpret_cast<unsigned long long *>(ctr + 4);
    unsigned *dyn_done = ctr + 6;
    const int W = WT > 0 ? WT : tab.W;
    const int WH = W / NH;  // worker rows per stage
    const int L = tab.L;
    const int ROW = TT + (MIS ? kSlack : 0);  // elements per worker row
    const size_t gbytes = (size_t)WH * ROW * 2;
    // with one stage per tile the residual is staged too; with halves the
    // consumers read it from global memory (prefetched into L2)
    const size_t rreg = NH == 1 ? (size_t)TT * 4 : 0;
    const size_t sbytes = gbytes + rreg + (MIS ? kMaxPieces * sizeof(int4) : 0) + kStageHead;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // tiles of TT fused elements from f_begin (a multiple of 256) to f_end
    const int64_t ntiles = (f_end - f_begin + TT - 1) / TT;
    const int64_t G_ = gridDim.x;
    const bool dyn = ntiles / G_ >= kDynMinRounds;
    const int64_t rounds_static = dyn ? ntiles / G_ - kDynRounds : (ntiles + G_ - 1) / G_;

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(smem_u32(&bars[s]), 1);
            mbar_init(smem_u32(&bars[S + s]), kConsumerWarps);
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    // Launched after whatever the stream ran before (programmatic
    // serialisation): no global memory is touched before that work is done.
    wait_for_prior_grid();
    allow_dependent_launch();
    __syncthreads();

    if (warp == kConsumerWarps) {
        // producer
        if (lane != 0) return;
        // Plans stage s for worker half h of tile t: the tile's index and half
        // (for the consumers) and, in the shifted layout, the piece table, with
        // its length and the bytes it copies per worker row.
        //
        // Piece table: {end of the piece (tile-relative), sh (or -1 if
        // unstaged), layer, copied range [lo, hi) of the row as lo | hi << 16}.
        // The last entry always ends at the tile's end.  The second half of a
        // tile copies the first half's table (the stage planned just before).
        auto plan = [&](int s, int64_t t, int h) {
            unsigned char *st = stages + (size_t)s * sbytes;
            volatile int64_t *head = reinterpret_cast<volatile int64_t *>(st + sbytes - kStageHead);
            head[0] = t * NH + h;
            if constexpr (MIS) {
                volatile int32_t *hh = reinterpret_cast<volatile int32_t *>(head);
                int4 *pieces = reinterpret_cast<int4 *>(st + gbytes + rreg);
                if (h > 0) {
                    const unsigned char *pst = stages + (size_t)((s + S - 1) % S) * sbytes;
                    const volatile int32_t *ph =
                        reinterpret_cast<const volatile int32_t *>(pst + sbytes - kStageHead);
                    const int n = ph[2];
                    const int4 *pp = reinterpret_cast<const int4 *>(pst + gbytes + rreg);
                    for (int i = 0; i < n; ++i) pieces[i] = pp[i];
                    hh[2] = n;
                    hh[3] = ph[3];
                    return;
                }
                const int64_t f0 = f_begin + t * TT;
                const int64_t f1 = f0 + TT < f_end ? f0 + TT : f_end;
                int n = 0;
                uint32_t row_bytes = 0;
                int64_t prev_phi = 0;  // end of the last staged piece's frames
                int l = find_layer(tab, f0);
                for (int64_t fa = f0; fa < f1;) {
                    while (tab.off[l + 1] <= fa) ++l;
                    const int64_t fb = tab.off[l + 1] < f1 ? tab.off[l + 1] : f1;
                    if (n == kMaxPieces - 1) {
                        pieces[n++] = make_int4((int)(f1 - f0), -1, l, 0);
                        break;
                    }
                    // The piece is copied as the whole 16-byte frames that hold
                    // it, including the partial frames at a layer's ends (every
                    // frame holds at least one element of the layer, so no copy
                    // reaches a page the layer does not touch).  Its gap is the
                    // smallest multiple of 8 that puts its first frame after the
                    // last frame of the piece before.
                    const int d = layer_shift(tab, l);
                    const int64_t x = fa - f0;
                    int64_t g = prev_phi - round_down8(x + d);
                    g = g > 0 ? round_up8(g) : 0;
                    const int64_t sh = g + d;
                    const int64_t plo = round_down8(x + sh);
                    const int64_t phi = round_up8(fb - f0 + sh);
                    if (phi > ROW) {
                        pieces[n++] = make_int4((int)(fb - f0), -1, l, 0);
                    } else {
                        pieces[n++] = make_int4((int)(fb - f0), (int)sh, l, (int)(plo | (phi << 16)));
                        row_bytes += (uint32_t)(phi - plo) * 2;
                        prev_phi = phi;
                    }
                    fa = fb;
                }
                hh[2] = n;
                hh[3] = (int32_t)row_bytes;
            }
        };
        // Issues the copies of stage s, planned for worker half h of tile t;
        // the expect-tx arrive (a release) also publishes the plan.
        auto issue = [&](int s, int64_t t, int h) {
            const uint32_t full = smem_u32(&bars[s]);
            unsigned char *st = stages + (size_t)s * sbytes;
            if (t == drop_tile) return;
            const int64_t f0 = f_begin + t * TT;
            const int64_t f1 = f0 + TT < f_end ? f0 + TT : f_end;
            const uint32_t rbytes = NH == 1 && resid ? (uint32_t)((f1 - f0) * 4) : 0u;
            // The copies' sources are read from the parameter bank into
            // registers before the first copy of a piece is issued: a copy
            // (an asm with a memory clobber) would otherwise hold each
            // pointer's read back until the copy before it has gone out.
            constexpr int WHc = WT / NH;
            if constexpr (!MIS) {
                mbar_expect_tx(full, (uint32_t)((f1 - f0) * 2 * W) + rbytes);
                int l = find_layer(tab, f0);
                for (int64_t fa = f0; fa < f1;) {
                    while (tab.off[l + 1] <= fa) ++l;
                    const int64_t fb = tab.off[l + 1] < f1 ? tab.off[l + 1] : f1;
                    const int64_t j = fa - tab.off[l];
                    const __half *src[WHc];
#pragma unroll
                    for (int w = 0; w < WHc; ++w) src[w] = tab.ptr[w * L + l];
#pragma unroll
                    for (int w = 0; w < WHc; ++w)
                        bulk_g2s(smem_u32(st + ((size_t)w * ROW + (size_t)(fa - f0)) * 2),
                                 src[w] + j, (uint32_t)((fb - fa) * 2), full);
                    fa = fb;
                }
            } else {
                const volatile int32_t *hh =
                    reinterpret_cast<const volatile int32_t *>(st + sbytes - kStageHead);
                const int n = hh[2];
                const uint32_t row_bytes = (uint32_t)hh[3];
                const int4 *pieces = reinterpret_cast<const int4 *>(st + gbytes + rreg);
                const int w0 = h * WH;
                mbar_expect_tx(full, row_bytes * (uint32_t)WH + rbytes);
                for (int i = 0; i < n; ++i) {
                    const int4 pc = pieces[i];
                    const int plo = pc.w & 0xffff, phi = pc.w >> 16;
                    if (pc.y < 0 || phi <= plo) continue;
                    const int64_t j = f0 + plo - pc.y - tab.off[pc.z];  // layer element at row plo
                    const __half *src[WHc];
#pragma unroll
                    for (int w = 0; w < WHc; ++w) src[w] = tab.ptr[(w0 + w) * L + pc.z];
#pragma unroll
                    for (int w = 0; w < WHc; ++w)
                        bulk_g2s(smem_u32(st + ((size_t)w * ROW + (size_t)plo) * 2), src[w] + j,
                                 (uint32_t)(phi - plo) * 2, full);
                }
            }
            if (rbytes) bulk_g2s(smem_u32(st + gbytes), resid + f0, rbytes, full);
            // with halves the consumers read the residual themselves, at the
            // tile's second stage: warm L2 with it at the first
            if (NH > 1 && h == 0 && resid)
                asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(resid + f0),
                             "r"((uint32_t)((f1 - f0) * 4))
                             : "memory");
        };
        // Waits until the consumers have released the slot of iteration it.
        auto slot_free = [&](int it) {
            const int s = it % S;
            if (it >= S && !mbar_wait(smem_u32(&bars[S + s]), ((it / S) - 1) & 1, limit_ns)) {
                atomicOr(err, 1u);
                return false;
            }
            return true;
        };
        int it = 0;  // stage iterations: NH per tile
        bool ok = true;
        unsigned long long q = 0;
        // the cyclic rounds: kept free of any other work, since the
        // producer's issue rate bounds the kernel's
        for (int64_t r = 0; r < rounds_static && ok; ++r) {
            const int64_t t = blockIdx.x + r * G_;
            if (t >= ntiles) break;
            for (int h = 0; h < NH; ++h, ++it) {
                if (!slot_free(it)) {
                    ok = false;
                    break;
                }
                plan(it % S, t, h);
                // the first tail index travels while the last cyclic tile's
                // copies go out
                if (dyn && r == rounds_static - 1 && h == NH - 1) q = atomicAdd(dyn_next, 1ull);
                issue(it % S, t, h);
            }
        }
        // the tail, handed out one tile at a time; the next index travels
        // while this tile's copies go out
        if (ok && dyn) {
            for (;;) {
                const int64_t t = rounds_static * G_ + (int64_t)q;
                if (t >= ntiles) break;
                for (int h = 0; h < NH; ++h, ++it) {
                    if (!slot_free(it)) {
                        ok = false;
                        break;
                    }
                    plan(it % S, t, h);
                    if (h == NH - 1) q = atomicAdd(dyn_next, 1ull);
                    issue(it % S, t, h);
                }
                if (!ok) break;
            }
        }
        // no tile left: the consumers stop at this stage
        if (ok && slot_free(it)) {
            unsigned char *st = stages + (size_t)(it % S) * sbytes;
            *reinterpret_cast<volatile int64_t *>(st + sbytes - kStageHead) = -1;
            mbar_arrive(smem_u32(&bars[it % S]));
            ++it;
        }
        // No copy may still be landing in shared memory when the CTA exits:
        // wait for every stage still in flight (each wait bounded; a stage
        // that gives up does not stop the waits for the others).
        for (int j = it > S ? it - S : 0; j < it; ++j)
            if (!mbar_wait(smem_u32(&bars[j % S]), (j / S) & 1, limit_ns))
                atomicOr(err, 2u);
        // Every index this producer fetched has come back (the fence waits
        // for its atomics); the last producer to get here resets the counters.
        if (dyn) {
            __threadfence();
            if (atomicAdd(dyn_done, 1u) == gridDim.x - 1) {
                atomicExch(dyn_next, 0ull);
                atomicExch(dyn_done, 0u);
            }
        }
        return;
    }

    // consumers
    // With worker halves (NH == 2) a warp sums the first half's workers of
    // its group into part[] and adds the second half's subtree to it: for
    // W = 16 that is the tree of all W (the binary-counter form joins the two
    // subtrees of 8 leaves last), so the bits are unchanged.  TT = 2048 gives
    // each warp one unit per tile, so one part[] per warp suffices.
    constexpr int WTH = WT > 0 ? WT / NH : 0;
    constexpr int MAXHH = NH == 1 ? MAXH : MAXH - 1;
    float part[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) part[e] = 0.f;
    for (int it = 0;; ++it) {
        const int s = it % S;
        if (!mbar_wait(smem_u32(&bars[s]), (it / S) & 1, limit_ns)) {
            if (lane == 0) atomicOr(err, 4u);
            return;
        }
        const unsigned char *st = stages + (size_t)s * sbytes;
        const int64_t hdr = *reinterpret_cast<const volatile int64_t *>(st + sbytes - kStageHead);
        if (hdr < 0) break;
        const int64_t t = hdr / NH;
        const int h = (int)(hdr - t * NH);
        const bool last = h == NH - 1;  // the tile's last stage: finish the groups
        const int64_t f0 = f_begin + t * TT;
        const int64_t f1 = f0 + TT < f_end ? f0 + TT : f_end;
        for (int64_t lo = f0 + (int64_t)warp * FC_UNIT; lo < f1;
             lo += (int64_t)kConsumerWarps * FC_UNIT) {
            const int64_t hi = lo + FC_UNIT < f1 ? lo + FC_UNIT : f1;
            const int64_t f = lo + 8 * lane;
            float tss = 0.f;
            if (f < hi) {  // f + 8 <= hi: N and every unit start are multiples of 8
                const size_t off = (size_t)(f - f0);
                // with halves the residual comes from global memory: its load
                // is issued before the tree, so that the two overlap
                float4 g0 = make_float4(0.f, 0.f, 0.f, 0.f), g1 = g0;
                if (NH > 1 && last && resid) {
                    g0 = __ldcs(reinterpret_cast<const float4 *>(resid + f));
                    g1 = __ldcs(reinterpret_cast<const float4 *>(resid + f + 4));
                }
                float a[8];
                bool whole = false;  // a holds the tree of all W workers
                if constexpr (!MIS) {
                    tree_sum<WT, MAXH, 8>(
                        W,
                        [&](int w, float(&x)[8]) {
                            unpack8(*reinterpret_cast<const uint4 *>(st + ((size_t)w * ROW + off) * 2), x);
                        },
                        a);
                    whole = true;
                } else {
                    const int uu = (int)off;
                    const int4 *pieces = reinterpret_cast<const int4 *>(st + gbytes + rreg);
                    int i = 0;
                    int4 pc = pieces[0];
                    while (pc.x <= uu) pc = pieces[++i];
                    const int alo = pc.w & 0xffff, ahi = pc.w >> 16;
                    // a group that runs past its piece (a layer boundary) takes
                    // the next piece too; the last piece ends at the tile's end
                    const int split = uu + 8 <= pc.x ? 8 : pc.x - uu;
                    const int4 pn = pieces[split < 8 ? i + 1 : i];
                    const int blo = pn.w & 0xffff, bhi = pn.w >> 16;
                    if (split == 8 && pc.y >= 0 && uu + pc.y >= alo && uu + pc.y + 8 <= ahi) {
                        // all 8 in one copied piece: two aligned loads, shifted
                        const int p0 = uu + (pc.y & ~7), d = pc.y & 7;
                        tree_sum<WTH, MAXHH, 8>(
                            WH,
                            [&](int w, float(&x)[8]) {
                                const uint4 *q = reinterpret_cast<const uint4 *>(
                                    st + ((size_t)w * ROW + p0) * 2);
                                const uint4 qa = q[0];
                                unpack8(d ? funnel8(qa, q[1], d) : qa, x);
                            },
                            a);
                    } else if (split < 8 && pc.y >= 0 && pn.y >= 0 && uu + pc.y >= alo &&
                               uu + pc.y + split <= ahi && uu + split + pn.y >= blo &&
                               uu + 8 + pn.y <= bhi && uu + 8 <= pn.x) {
                        // at a layer boundary, both pieces staged: elements
                        // e < split from piece pc, the rest from piece pn, each
                        // read as two aligned 16-byte words and a funnel shift
                        const int pa = uu + (pc.y & ~7), da = pc.y & 7;
                        const int pb = uu + (pn.y & ~7), db = pn.y & 7;
                        // word j holds elements 2j, 2j+1: mask of the halves from pc
                        uint32_t m[4];
#pragma unroll
                        for (int j = 0; j < 4; ++j)
                            m[j] = 2 * j + 1 < split ? 0xffffffffu : (2 * j < split ? 0x0000ffffu : 0u);
                        tree_sum<WTH, MAXHH, 8>(
                            WH,
                            [&](int w, float(&x)[8]) {
                                const unsigned char *row = st + (size_t)w * ROW * 2;
                                const uint4 *qa = reinterpret_cast<const uint4 *>(row + (size_t)pa * 2);
                                const uint4 *qb = reinterpret_cast<const uint4 *>(row + (size_t)pb * 2);
                                uint4 v = qa[0], vb = qb[0];
                                if (da) v = funnel8(v, qa[1], da);
                                if (db) vb = funnel8(vb, qb[1], db);
                                v.x = (v.x & m[0]) | (vb.x & ~m[0]);
                                v.y = (v.y & m[1]) | (vb.y & ~m[1]);
                                v.z = (v.z & m[2]) | (vb.z & ~m[2]);
                                v.w = (v.w & m[3]) | (vb.w & ~m[3]);
                                unpack8(v, x);
                            },
                            a);
                    } else {
                        // unstaged pieces (a tile with more pieces than the
                        // table holds, or past the row's slack) or a group over
                        // three or more layers: element by element from
                        // global memory, all W workers at the tile's last stage
                        whole = true;
                        if (last) {
                            int l = pc.z;
#pragma unroll
                            for (int e = 0; e < 8; ++e) {
                                while (tab.off[l + 1] <= f + e) ++l;
                                const int64_t j = f + e - tab.off[l];
                                float s1[1];
                                tree_sum<WT, MAXH, 1>(
                                    W,
                                    [&](int w, float(&x)[1]) {
                                        x[0] = ld_half_as_float(tab.ptr[w * L + l] + j);
                                    },
                                    s1);
                                a[e] = s1[0];
                            }
                        }
                    }
                }
                if (NH > 1 && !whole) {
                    if (!last) {
#pragma unroll
                        for (int e = 0; e < 8; ++e) part[e] = a[e];
                    } else {
#pragma unroll
                        for (int e = 0; e < 8; ++e) a[e] = __fadd_rn(part[e], a[e]);
                    }
                }
                if (last) {
                    float r[8];
                    if (resid) {
                        float4 r0, r1;
                        if (NH == 1) {
                            const float4 *rr = reinterpret_cast<const float4 *>(st + gbytes + off * 4);
                            r0 = rr[0];
                            r1 = rr[1];
                        } else {
                            r0 = g0;
                            r1 = g1;
                        }
                        r[0] = r0.x; r[1] = r0.y; r[2] = r0.z; r[3] = r0.w;
                        r[4] = r1.x; r[5] = r1.y; r[6] = r1.z; r[7] = r1.w;
                    }
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        a[e] = __fmul_rn(a[e], u);
                        if (resid) a[e] = __fadd_rn(a[e], r[e]);
                    }
                    reinterpret_cast<float4 *>(out + f)[0] = make_float4(a[0], a[1], a[2], a[3]);
                    reinterpret_cast<float4 *>(out + f)[1] = make_float4(a[4], a[5], a[6], a[7]);
                    tss = __fadd_rn(tss, group_sumsq(a));
                }
            }
            if (last && partials) {
                tss = warp_sum_f32(tss);
                if (lane == 0) partials[lo / FC_UNIT] = tss;
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&bars[S + s]));
    }
}

// Tile size and stage count for W workers in NH stages per tile and CPS
// CTAs per SM: a stage holds W/NH rows of TT fp16 values (plus the slack
// of the shifted layout), with one stage per tile also the TT fp32
// residuals, and the piece table.
//  * one CTA per SM: about 64 KB of gradients a stage, as many stages as
//    fit (at most 4);
//  * worker halves (two CTAs per SM, full carveout): TT = 2048 (one unit per
//    consumer warp), as many stages as fit in 113 KB (at most 6);
//  * two CTAs per SM with whole stages (8 workers): TT = 2048, two stages,
//    85 KB per CTA, so that a 75 % carveout holds both.
static void tma_shape(int W, bool mis, int NH, int CPS, int &TT, int &S, size_t &smem)
{
    TT = 2048;
    if (CPS == 1)
        while (TT > FC_UNIT && (size_t)W * TT * 2 > 65536) TT /= 2;
    const size_t row = (size_t)TT + (mis ? kSlack : 0);
    const size_t sbytes = (size_t)(W / NH) * row * 2 + (NH == 1 ? (size_t)TT * 4 : 0) +
                          (mis ? kMaxPieces * sizeof(int4) : 0) + kStageHead;
    const size_t cap = CPS == 1 ? 227 * 1024 - 128 : NH > 1 ? 113 * 1024 - 128 : 86400 - 128;
    const int smax = CPS == 1 ? 4 : NH > 1 ? 6 : 2;
    S = (int)(cap / sbytes);
    if (S > smax) S = smax;
    smem = 128 + (size_t)S * sbytes;
}

template <class Tab>
int tma_layout(const Tab &tab, const UnitGeom &G, const float *partials)
{
    if (partials && G.cs % FC_UNIT != 0) return 0;
    if (G.N % 8 != 0) return 0;
    bool aligned = true;
    for (int l = 0; l < tab.L; ++l) {
        if (tab.off[l] % 8 != 0 || !((tab.vec[l >> 5] >> (l & 31)) & 1u)) aligned = false;
        // the shifted layout needs one shift per layer, the same for all workers
        const uintptr_t s0 = ((uintptr_t)tab.ptr[l] - 2u * (uintptr_t)tab.off[l]) & 15u;
        for (int w = 1; w < tab.W; ++w)
            if ((((uintptr_t)tab.ptr[w * tab.L + l] - 2u * (uintptr_t)tab.off[l]) & 15u) != s0)
                return 0;
    }
    int TT, S;
    size_t smem;
    tma_shape(tab.W, !aligned, 1, 1, TT, S, smem);
    if (S < 2) return 0;
    if (!aligned) return 2;
    // Aligned layouts, by length (tiles of TT elements), as measured in
    // isolation:
    //  * long runs take the shifted variant (every shift 0): AlexNet-sized
    //    352 against 361 us for the aligned variant;
    //  * mid-size runs the register kernel streams faster than either
    //    staged variant (7M elements x 16 workers: 43.5 against 48 us);
    //  * short runs keep the aligned variant (2M x 16: 11 against 13 us).
    const int64_t tiles = (G.N + TT - 1) / TT;
    if (tiles >= FC_TMA_SHIFTED_MIN_TILES) {
        tma_shape(tab.W, true, 1, 1, TT, S, smem);
        if (S >= 2) return 2;
    }
    return tiles >= FC_TMA_REGISTER_MIN_TILES ? 0 : 1;
}

// Worker halves (two stages per tile, two CTAs per SM) for the shifted
// layout with 16 workers; two CTAs per SM with whole stages for the shifted
// layout with 8 workers.
#ifndef FC_TMA_HALVES
#define FC_TMA_HALVES 1
#endif
#ifndef FC_TMA_W8_PAIRS
#define FC_TMA_W8_PAIRS 1
#endif

template <class Tab, int WT, int MAXH, bool MIS, int NH, int CPS>
static cudaError_t launch_tma_w(const Tab &tab, const UnitGeom &G, float u,
                                const float *resid, float *out, float *partials,
                                unsigned *ctr, cudaStream_t s, int64_t fb, int64_t fe)
{
    int TT, S;
    size_t smem;
    tma_shape(tab.W, MIS, NH, CPS, TT, S, smem);
    auto kern = k_reduce_tma<Tab, WT, MAXH, MIS, NH, CPS>;
    static std::mutex mu;
    static int blocks[64];  // resident CTAs on the device (set on first use)
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev >= 64) return cudaErrorInvalidDevice;
    int grid_cap = 0;
    {
        std::lock_guard<std::mutex> lock(mu);
        if (!blocks[dev]) {
            cudaError_t e = cudaFuncSetAttribute((const void *)kern,
                                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 CPS == 1 ? 227 * 1024 : (int)smem);
            if (e != cudaSuccess) return e;
            if (CPS > 1) {
                // two CTAs per SM: the carveout that holds both
                e = cudaFuncSetAttribute((const void *)kern,
                                         cudaFuncAttributePreferredSharedMemoryCarveout,
                                         NH > 1 ? 100 : 75);
                if (e != cudaSuccess) return e;
                int sms = 0, per_sm = 0;
                cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
                if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kThreads,
                                                                  smem) != cudaSuccess ||
                    per_sm < 1)
                    per_sm = 1;
                blocks[dev] = (sms < 1 ? 1 : sms) * per_sm;
            } else {
                blocks[dev] = -1;
            }
        }
        grid_cap = blocks[dev];
    }
    const int64_t tiles = (fe - fb + TT - 1) / TT;
    const int grid = grid_cap < 0 ? grid_for((const void *)kern, kThreads, smem, tiles)
                                  : (int)(tiles < grid_cap ? (tiles < 1 ? 1 : tiles) : grid_cap);
    const int64_t drop = g_drop_tile.exchange(-1);
    const uint64_t limit = drop >= 0 ? g_drop_limit_ns.load() : kWaitLimitNs;
    return launch_after_prior(kern, (unsigned)grid, kThreads, smem, s, tab, G, TT, S, u,
                              resid, out, partials, ctr, drop, limit, fb, fe);
}

template <class Tab, bool MIS>
static cudaError_t launch_tma_layout(const Tab &tab, const UnitGeom &G, float u,
                                     const float *resid, float *out, float *partials,
                                     unsigned *ctr, cudaStream_t s, int64_t fb, int64_t fe)
{
    constexpr int H = MIS && FC_TMA_HALVES ? 2 : 1;
    constexpr int P8 = MIS && FC_TMA_W8_PAIRS ? 2 : 1;
    switch (tab.W) {
    case 4: return launch_tma_w<Tab, 4, 3, MIS, 1, 1>(tab, G, u, resid, out, partials, ctr, s, fb, fe);
    case 8: return launch_tma_w<Tab, 8, 4, MIS, 1, P8>(tab, G, u, resid, out, partials, ctr, s, fb, fe);
    case 16: return launch_tma_w<Tab, 16, 5, MIS, H, H>(tab, G, u, resid, out, partials, ctr, s, fb, fe);
    default: break;
    }
    return cudaErrorNotSupported;
}

template <class Tab>
cudaError_t launch_reduce_tma(const Tab &tab, const UnitGeom &G, float u,
                              const float *resid, float *out, float *partials,
                              unsigned *ctr, cudaStream_t s, int layout, int64_t fb,
                              int64_t fe)
{
    if (fe < 0) fe = G.N;
    if (fb >= fe) return cudaSuccess;
    if (fb % FC_UNIT != 0) return cudaErrorInvalidValue;
    if (layout == 1)
        return launch_tma_layout<Tab, false>(tab, G, u, resid, out, partials, ctr, s, fb, fe);
    if (layout == 2)
        return launch_tma_layout<Tab, true>(tab, G, u, resid, out, partials, ctr, s, fb, fe);
    return cudaErrorNotSupported;
}

}  // namespace fc

extern "C" fc_status fc_test_stage_loss(int64_t tile, uint64_t wait_limit_ns)
{
    if (tile >= 0 && (wait_limit_ns < 1000000ull || wait_limit_ns > 2000000000ull))
        return fc::set_error(FC_ERR_INVALID_ARG, "wait_limit_ns must be in [1 ms, 2 s]");
    fc::g_drop_limit_ns.store(wait_limit_ns);
    fc::g_drop_tile.store(tile < 0 ? -1 : tile);
    return FC_OK;
}

namespace fc {

bool stage_loss_armed() { return g_drop_tile.load() >= 0; }

template int tma_layout<TableS>(const TableS &, const UnitGeom &, const float *);
template int tma_layout<TableL>(const TableL &, const UnitGeom &, const float *);
template cudaError_t launch_reduce_tma<TableS>(const TableS &, const UnitGeom &, float,
                                               const float *, float *, float *,
                                               unsigned *, cudaStream_t, int, int64_t,
                                               int64_t);
template cudaError_t launch_reduce_tma<TableL>(const TableL &, const UnitGeom &, float,
                                               const float *, float *, float *,
                                               unsigned *, cudaStream_t, int, int64_t,
                                               int64_t);

}  // namespace fc
