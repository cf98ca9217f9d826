/*
 * CPU oracle of the gradient-aggregation engine.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the plain, slow, single-threaded
 * statement of what the engine computes, used by the tests, by the smoke
 * check and by the benchmark's CPU-baseline leg.  The product path never
 * links, loads or calls it, and it shares no code with the CUDA library.
 *
 * Build: gcc -O2 -std=c11 -ffp-contract=off -fno-fast-math -shared -fPIC.
 * -ffp-contract=off matters: every float operation below is one IEEE-754
 * binary32 operation rounded to nearest-even, never fused into an FMA.
 *
 * Sources of the definitions (titles of the pages; no code is printed there):
 *  - FireCaffe: near-linear acceleration of deep neural network training on
 *    compute clusters (arXiv 1511.00175).
 *      §6: gradients of the workers are summed element-wise (allreduce over
 *          vectors of length |dW|) in a binary tree whose depth is the
 *          base-2 log of the worker count; the workers apply the sum.
 *      §3: batched SGD; Eq. 1 sizes the weight volume.
 *  - Optimizing Network Performance for Distributed DNN Training on GPU
 *    Clusters: ImageNet/AlexNet Training in 1.5 Minutes (GradientFlow,
 *    arXiv 1902.06855), abstract: mixed-precision training; lazy allreduce
 *    fuses many communication operations into one; coarse-grained sparse
 *    communication sends only the chunks that matter.
 *  The pages leave the score, the selection rule, the residual and the
 *  optimiser open; the readings taken here are: L2 norm of a chunk as its
 *  importance, top-k chunks with ties to the lower index, unkept values
 *  carried in an fp32 residual added after the unscale, and Caffe-form
 *  momentum SGD (v = mu v + lr g; w = w - v).
 *
 * Every function below has a pin in the CPU test suite except where its
 * header says otherwise.
 */
#include <math.h>
#include <stdatomic.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ---- binary16 <-> binary32, from the IEEE 754 format definition -------- */

/* Exact value of a binary16 bit pattern (finite values are exact in
 * binary32: 11 significant bits, exponents -24..15). */
float orc_half_to_float(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 31;
    int m = h & 1023;
    float v;
    if (e == 0)
        v = ldexpf((float)m, -24);            /* subnormal: m * 2^-24 */
    else if (e == 31)
        v = m ? NAN : INFINITY;
    else
        v = ldexpf((float)(m + 1024), e - 25); /* (1 + m/1024) * 2^(e-15) */
    return sign ? -v : v;
}

/* binary32 -> binary16, round to nearest, ties to even; overflow to inf. */
uint16_t orc_float_to_half(float x)
{
    uint16_t sign = signbit(x) ? 0x8000u : 0u;
    if (isnan(x)) return (uint16_t)(sign | 0x7e00u);
    double a = fabs((double)x);
    if (a == 0.0) return sign;
    /* largest finite is 65504 = (2 - 2^-10) 2^15; the rounding boundary to
     * infinity is 65504 + 16, where the tie goes to the even (overflowing)
     * neighbour. */
    if (a >= 65520.0) return (uint16_t)(sign | 0x7c00u);
    if (a < ldexp(1.0, -14)) {
        /* subnormal grid: multiples of 2^-24 */
        double q = nearbyint(a * ldexp(1.0, 24)); /* exact product; RNE */
        return (uint16_t)(sign | (uint16_t)q);   /* q == 1024 is 2^-14 */
    }
    int E;
    (void)frexp(a, &E);          /* a = f 2^E, f in [0.5, 1) */
    int ue = E - 1;              /* a in [2^ue, 2^(ue+1)) */
    double q = nearbyint(ldexp(a, 10 - ue)); /* significand in [1024, 2048] */
    if (q == 2048.0) { q = 1024.0; ue += 1; }
    if (ue > 15) return (uint16_t)(sign | 0x7c00u);
    return (uint16_t)(sign | (uint16_t)((ue + 15) << 10) | (uint16_t)(q - 1024.0));
}

/* ---- a1: fusion (lazy allreduce) --------------------------------------- */

/* offsets[l] = sizes[0] + ... + sizes[l-1]: the layers are concatenated in
 * their given order with no padding.  Returns N = the sum of all sizes. */
int64_t orc_layout(int32_t L, const int64_t *sizes, int64_t *offsets)
{
    int64_t acc = 0;
    for (int32_t l = 0; l < L; ++l) {
        offsets[l] = acc;
        acc += sizes[l];
    }
    return acc;
}

/* fused[w*N + offsets[l] + j] = grads[w*L + l][j], a bitwise copy.
 * grads is an array of W*L host pointers to binary16 data. */
void orc_fuse_pack(int32_t W, int32_t L, const int64_t *sizes,
                   const uint16_t *const *grads, uint16_t *fused)
{
    int64_t *off = (int64_t *)malloc(sizeof(int64_t) * (size_t)(L > 0 ? L : 1));
    int64_t N = orc_layout(L, sizes, off);
    for (int32_t w = 0; w < W; ++w)
        for (int32_t l = 0; l < L; ++l) {
            const uint16_t *src = grads[(int64_t)w * L + l];
            uint16_t *dst = fused + (int64_t)w * N + off[l];
            const int64_t n = sizes[l];
            for (int64_t j = 0; j < n; ++j) dst[j] = src[j];
        }
    free(off);
}

/* ---- a2: binary reduction tree over the workers ------------------------ */

/* Sum of x[0..m) by a binary tree in level order: at each level adjacent
 * pairs (0,1), (2,3), ... are added (binary32, round to nearest even); an
 * odd last element moves up unchanged.  Overwrites x. */
float orc_tree_sum(float *x, int32_t m)
{
    if (m <= 0) return 0.0f;
    while (m > 1) {
        int32_t half = m / 2;
        for (int32_t j = 0; j < half; ++j)
            x[j] = x[2 * j] + x[2 * j + 1];
        if (m & 1) {
            x[half] = x[m - 1];
            m = half + 1;
        } else {
            m = half;
        }
    }
    return x[0];
}

/* The multiplier that undoes the loss scale and averages over the workers:
 * the binary32 value nearest to 1 / (S * W). */
float orc_unscale_factor(float loss_scale, int32_t W)
{
    return (float)(1.0 / ((double)loss_scale * (double)W));
}

/* out[i] = tree_w(fp32(fused[w*N + i])) * (1/(S W)) [+ residual[i]].
 * residual may be NULL (treated as absent, not as zeros: x + 0 would turn
 * -0 into +0). */
void orc_tree_reduce(int32_t W, int64_t N, const uint16_t *fused,
                     float loss_scale, const float *residual, float *out)
{
    /* orc_half_to_float of every bit pattern, looked up instead of
     * recomputed per element (the values are identical).  The table is
     * filled once, by the first caller; a concurrent caller waits until it
     * is complete (state 0 empty, 1 being filled, 2 ready). */
    static float h2f[65536];
    static atomic_int h2f_state = 0;
    if (atomic_load_explicit(&h2f_state, memory_order_acquire) != 2) {
        int expected = 0;
        if (atomic_compare_exchange_strong(&h2f_state, &expected, 1)) {
            for (int b = 0; b < 65536; ++b) h2f[b] = orc_half_to_float((uint16_t)b);
            atomic_store_explicit(&h2f_state, 2, memory_order_release);
        } else {
            while (atomic_load_explicit(&h2f_state, memory_order_acquire) != 2) {
            }
        }
    }
    float *x = (float *)malloc(sizeof(float) * (size_t)W);
    float inv = orc_unscale_factor(loss_scale, W);
    for (int64_t i = 0; i < N; ++i) {
        for (int32_t w = 0; w < W; ++w)
            x[w] = h2f[fused[(int64_t)w * N + i]];
        float s = orc_tree_sum(x, W);
        float a = s * inv;
        if (residual) a = a + residual[i];
        out[i] = a;
    }
    free(x);
}

/* ---- a2 with other summation orders ------------------------------------ */
/* The pages contrast the tree with a parameter server (FireCaffe §6: one
 * node receives every worker's gradient and sums them) and name ring-based
 * allreduce (GradientFlow abstract).  Their fp32 results differ from the
 * tree's by rounding only; the engine offers them as selectable orders.
 *   order 0: the binary tree above;
 *   order 1: parameter server, workers added one after another in index
 *            order: ((x0 + x1) + x2) + ... ;
 *   order 2: ring reduce-scatter: the fused vector is cut into W segments,
 *            segment s = [floor(s*N/W), floor((s+1)*N/W)); the partial sum of
 *            segment s starts at worker s and travels around the ring, each
 *            worker adding its own value: ((x_s + x_{s+1}) + ...) + x_{s-1},
 *            indices modulo W. */

/* x[0] + x[1] + ... + x[m-1], added left to right. */
float orc_sequential_sum(const float *x, int32_t m)
{
    float acc = x[0];
    for (int32_t j = 1; j < m; ++j) acc = acc + x[j];
    return acc;
}

/* Segment of fused index i: the s with floor(s*N/W) <= i < floor((s+1)*N/W). */
int32_t orc_ring_segment(int64_t i, int64_t N, int32_t W)
{
    int32_t s = 0;
    while (s + 1 < W && ((int64_t)(s + 1) * N) / W <= i) ++s;
    return s;
}

void orc_reduce_ordered(int32_t W, int64_t N, const uint16_t *fused,
                        float loss_scale, const float *residual, float *out,
                        int32_t order)
{
    if (order == 0) {
        orc_tree_reduce(W, N, fused, loss_scale, residual, out);
        return;
    }
    float *x = (float *)malloc(sizeof(float) * (size_t)W);
    float inv = orc_unscale_factor(loss_scale, W);
    int32_t seg = 0;
    for (int64_t i = 0; i < N; ++i) {
        int32_t start = 0;
        if (order == 2) {
            while (seg + 1 < W && ((int64_t)(seg + 1) * N) / W <= i) ++seg;
            start = seg;
        }
        for (int32_t t = 0; t < W; ++t)
            x[t] = orc_half_to_float(fused[(int64_t)((start + t) % W) * N + i]);
        float s = orc_sequential_sum(x, W);
        float a = s * inv;
        if (residual) a = a + residual[i];
        out[i] = a;
    }
    free(x);
}

/* ---- a3: chunk L2 norms -------------------------------------------------- */

int64_t orc_num_chunks(int64_t N, int64_t chunk)
{
    return (N + chunk - 1) / chunk;
}

/* norms[c] = sqrt(sum of a[i]^2 over chunk c), chunks of `chunk` consecutive
 * elements of the concatenated vector (the last may be shorter).  The sum is
 * taken in binary64 in index order; the square of a binary32 value is exact
 * in binary64, so the only roundings are the additions and the final sqrt
 * and narrowing. */
void orc_chunk_norms(const float *a, int64_t N, int64_t chunk, float *norms)
{
    int64_t C = orc_num_chunks(N, chunk);
    for (int64_t c = 0; c < C; ++c) {
        int64_t lo = c * chunk, hi = lo + chunk < N ? lo + chunk : N;
        double ss = 0.0;
        for (int64_t i = lo; i < hi; ++i)
            ss += (double)a[i] * (double)a[i];
        norms[c] = (float)sqrt(ss);
    }
}

/* ---- a4: top-k chunk selection and compaction --------------------------- */

/* k = ceil(C * num / den) in integers, at least 1 and at most C. */
int64_t orc_keep_count(int64_t C, int64_t num, int64_t den)
{
    int64_t k = (C * num + den - 1) / den;
    if (k < 1) k = 1;
    if (k > C) k = C;
    return k;
}

static const float *g_sort_norms;

/* Order: larger norm first; equal norms, lower chunk index first. */
static int by_norm_desc_index_asc(const void *pa, const void *pb)
{
    int64_t a = *(const int64_t *)pa, b = *(const int64_t *)pb;
    float na = g_sort_norms[a], nb = g_sort_norms[b];
    if (na > nb) return -1;
    if (na < nb) return 1;
    return (a < b) ? -1 : (a > b) ? 1 : 0;
}

/* Keeps the k chunks that come first in the order above.  Outputs:
 *  idx[0..k)      kept chunk indices, ascending;
 *  mask[0..C)     1 for kept chunks, 0 otherwise;
 *  packed         (if not NULL) kept chunks' values of a, in idx order, each
 *                 in a slot of `chunk` floats, a short last chunk zero-padded;
 *  *threshold     the norm of the k-th chunk in the order. */
void orc_chunk_select(const float *norms, int64_t C, int64_t k,
                      const float *a, int64_t N, int64_t chunk,
                      int32_t *idx, uint8_t *mask, float *packed,
                      float *threshold)
{
    int64_t *order = (int64_t *)malloc(sizeof(int64_t) * (size_t)C);
    for (int64_t c = 0; c < C; ++c) order[c] = c;
    g_sort_norms = norms;
    qsort(order, (size_t)C, sizeof(int64_t), by_norm_desc_index_asc);
    memset(mask, 0, (size_t)C);
    for (int64_t q = 0; q < k; ++q) mask[order[q]] = 1;
    *threshold = norms[order[k - 1]];
    int64_t q = 0;
    for (int64_t c = 0; c < C; ++c) {
        if (!mask[c]) continue;
        idx[q] = (int32_t)c;
        if (packed) {
            for (int64_t j = 0; j < chunk; ++j) {
                int64_t i = c * chunk + j;
                packed[q * chunk + j] = (i < N) ? a[i] : 0.0f;
            }
        }
        ++q;
    }
    free(order);
}

/* fp16 send buffer of the kept chunks (mixed-precision communication,
 * GradientFlow abstract): out[j] = binary16(packed[j] * send_scale), each a
 * binary32 product rounded to nearest even, then rounded to binary16 (ties
 * to even, overflow to infinity).  The zero padding stays +0. */
void orc_pack_fp16(const float *packed, int64_t n, float send_scale,
                   uint16_t *out)
{
    for (int64_t j = 0; j < n; ++j)
        out[j] = orc_float_to_half(packed[j] * send_scale);
}

/* ---- a5: residual fold and momentum SGD ----------------------------------- */

/* For every element i, with kept = mask[i / chunk]:
 *   g = kept ? a : 0          (the aggregated gradient that is applied)
 *   r = kept ? 0 : a          (what was not sent is carried to the next step)
 *   v = mu * v + lr * g       (two products, then their sum)
 *   w = w - v
 *   w16 = binary16(w)         (if w16 is not NULL)
 * a and residual may be the same array. */
void orc_residual_sgd_update(const float *a, const uint8_t *mask, int64_t N,
                             int64_t chunk, float lr, float momentum,
                             float *residual, float *velocity, float *weights,
                             uint16_t *w16)
{
    for (int64_t i = 0; i < N; ++i) {
        int kept = mask[i / chunk] != 0;
        float ai = a[i];
        float g = kept ? ai : 0.0f;
        float r = kept ? 0.0f : ai;
        float t1 = momentum * velocity[i];
        float t2 = lr * g;
        float v = t1 + t2;
        float w = weights[i] - v;
        residual[i] = r;
        velocity[i] = v;
        weights[i] = w;
        if (w16) w16[i] = orc_float_to_half(w);
    }
}
