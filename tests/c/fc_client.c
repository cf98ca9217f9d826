/*
 * A plain C client of libfc: no Python, no torch.  It reads a problem and
 * its seeded gradients from a file, runs fc_step for the given number of
 * steps on the GPU through the C ABI of include/fc.h and the CUDA runtime,
 * and writes the engine's state and the last step's selection to a file.
 * The GPU tests compare that state with the oracle.
 *
 * Input (little-endian):  int32 W, L; int64 sizes[L]; int64 chunk;
 *   int64 keep_num, keep_den; float loss_scale, lr, momentum; int32 steps;
 *   float weights[N]; then per step the fp16 gradients, worker-major and in
 *   layer order (W * N halves).
 * Output: int64 k; int32 idx[k]; float threshold; float residual[N],
 *   velocity[N], weights[N].
 * Exit status 0 on success; otherwise a message on stderr.
 */
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>

#include <cuda_runtime_api.h>

#include "fc.h"

static int fail(const char *what, const char *detail)
{
    fprintf(stderr, "fc_client: %s: %s\n", what, detail ? detail : "");
    return 1;
}

#define CUDA(x)                                                        \
    do {                                                               \
        cudaError_t e_ = (x);                                          \
        if (e_ != cudaSuccess) return fail(#x, cudaGetErrorString(e_)); \
    } while (0)

#define FC(x)                                                          \
    do {                                                               \
        if ((x) != FC_OK) return fail(#x, fc_last_error());            \
    } while (0)

static int read_all(FILE *f, void *p, size_t n)
{
    return fread(p, 1, n, f) == n ? 0 : 1;
}

int main(int argc, char **argv)
{
    if (argc != 3) return fail("usage", "fc_client <input> <output>");
    FILE *in = fopen(argv[1], "rb");
    if (!in) return fail("cannot open", argv[1]);
    int32_t W, L, steps;
    int64_t chunk, keep_num, keep_den;
    float loss_scale, lr, momentum;
    if (read_all(in, &W, 4) || read_all(in, &L, 4)) return fail("read", "header");
    if (W < 1 || L < 1 || L > FC_MAX_TABLE_LAYERS) return fail("header", "W or L");
    int64_t *sizes = malloc(sizeof(int64_t) * (size_t)L);
    if (!sizes || read_all(in, sizes, sizeof(int64_t) * (size_t)L)) return fail("read", "sizes");
    if (read_all(in, &chunk, 8) || read_all(in, &keep_num, 8) || read_all(in, &keep_den, 8) ||
        read_all(in, &loss_scale, 4) || read_all(in, &lr, 4) || read_all(in, &momentum, 4) ||
        read_all(in, &steps, 4))
        return fail("read", "parameters");
    int64_t N = 0;
    for (int32_t l = 0; l < L; ++l) N += sizes[l];
    const int64_t C = fc_num_chunks(N, chunk);
    const int64_t k = fc_keep_count(C, keep_num, keep_den);
    if (N < 1 || C < 1 || k < 1) return fail("problem", "empty");

    float *host = malloc(sizeof(float) * (size_t)N);
    uint16_t *g_host = malloc(sizeof(uint16_t) * (size_t)(W * N));
    if (!host || !g_host) return fail("malloc", "host buffers");

    /* device state and outputs */
    float *residual, *velocity, *weights, *norms, *packed, *threshold;
    int32_t *idx;
    uint8_t *mask;
    void *ws, *grads_dev;
    const size_t ws_bytes = fc_step_workspace_size(N, chunk);
    CUDA(cudaMalloc((void **)&residual, sizeof(float) * (size_t)N));
    CUDA(cudaMalloc((void **)&velocity, sizeof(float) * (size_t)N));
    CUDA(cudaMalloc((void **)&weights, sizeof(float) * (size_t)N));
    CUDA(cudaMalloc((void **)&norms, sizeof(float) * (size_t)C));
    CUDA(cudaMalloc((void **)&packed, sizeof(float) * (size_t)(k * chunk)));
    CUDA(cudaMalloc((void **)&threshold, sizeof(float)));
    CUDA(cudaMalloc((void **)&idx, sizeof(int32_t) * (size_t)k));
    CUDA(cudaMalloc((void **)&mask, (size_t)C));
    CUDA(cudaMalloc(&ws, ws_bytes));
    CUDA(cudaMalloc(&grads_dev, sizeof(uint16_t) * (size_t)(W * N)));
    CUDA(cudaMemset(residual, 0, sizeof(float) * (size_t)N));
    CUDA(cudaMemset(velocity, 0, sizeof(float) * (size_t)N));
    CUDA(cudaMemset(ws, 0, ws_bytes));
    if (read_all(in, host, sizeof(float) * (size_t)N)) return fail("read", "weights");
    CUDA(cudaMemcpy(weights, host, sizeof(float) * (size_t)N, cudaMemcpyHostToDevice));

    /* every worker's layers back to back in one buffer, one pointer each */
    const void **table = malloc(sizeof(void *) * (size_t)W * (size_t)L);
    if (!table) return fail("malloc", "table");
    for (int32_t w = 0, p = 0; w < W; ++w) {
        int64_t off = (int64_t)w * N;
        for (int32_t l = 0; l < L; ++l, ++p) {
            table[p] = (const uint16_t *)grads_dev + off;
            off += sizes[l];
        }
    }
    cudaStream_t s;
    CUDA(cudaStreamCreate(&s));
    for (int32_t st = 0; st < steps; ++st) {
        if (read_all(in, g_host, sizeof(uint16_t) * (size_t)(W * N))) return fail("read", "grads");
        CUDA(cudaMemcpyAsync(grads_dev, g_host, sizeof(uint16_t) * (size_t)(W * N),
                             cudaMemcpyHostToDevice, s));
        FC(fc_step(table, W, L, sizes, loss_scale, chunk, k, lr, momentum, residual, residual,
                   velocity, weights, NULL, norms, idx, mask, packed, NULL, 1.0f, threshold, ws,
                   ws_bytes, (void *)s));
        CUDA(cudaStreamSynchronize(s));
    }
    fclose(in);

    FILE *out = fopen(argv[2], "wb");
    if (!out) return fail("cannot open", argv[2]);
    int32_t *idx_h = malloc(sizeof(int32_t) * (size_t)k);
    float thr;
    if (!idx_h) return fail("malloc", "idx");
    CUDA(cudaMemcpy(idx_h, idx, sizeof(int32_t) * (size_t)k, cudaMemcpyDeviceToHost));
    CUDA(cudaMemcpy(&thr, threshold, sizeof(float), cudaMemcpyDeviceToHost));
    fwrite(&k, 8, 1, out);
    fwrite(idx_h, sizeof(int32_t), (size_t)k, out);
    fwrite(&thr, 4, 1, out);
    float *arrays[3] = {residual, velocity, weights};
    for (int i = 0; i < 3; ++i) {
        CUDA(cudaMemcpy(host, arrays[i], sizeof(float) * (size_t)N, cudaMemcpyDeviceToHost));
        fwrite(host, sizeof(float), (size_t)N, out);
    }
    fclose(out);
    CUDA(cudaStreamDestroy(s));
    cudaFree(residual); cudaFree(velocity); cudaFree(weights); cudaFree(norms); cudaFree(packed);
    cudaFree(threshold); cudaFree(idx); cudaFree(mask); cudaFree(ws); cudaFree(grads_dev);
    free(sizes); free(host); free(g_host); free(table); free(idx_h);
    return 0;
}
