/*
 * A plain C program that uses libmoe_layout.so through include/moe_layout.h
 * alone (no Python, no C++), as any C caller of the library would.
 *
 *   moe_c_client host   checks the host-side parts of the ABI: status
 *                       strings, the workspace and launch-count queries, and
 *                       the synchronous rejection of bad arguments (no GPU
 *                       is touched);
 *   moe_c_client gpu    runs moe_layout_dispatch (bf16 and FP8) and
 *                       moe_combine on a decode-shaped and a prefill-shaped
 *                       batch and compares every output bit for bit with the
 *                       CPU oracle's C functions (test infrastructure,
 *                       linked in for the comparison only).
 *
 * Exit status 0 when every check passes.
 */
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime_api.h>

#include "moe_layout.h"

/* the oracle's C entry points (oracle/moe_oracle.c) */
uint16_t oracle_f32_to_bf16(float f);
uint32_t oracle_layout(const int32_t *topk_ids, int32_t T, int32_t K, int32_t E, int32_t R,
                       int32_t *counts, int32_t *offsets, int32_t *rank_offsets,
                       int32_t *src_token, int32_t *dst_row);
void oracle_dispatch_bf16(const uint16_t *tokens, int32_t T, int32_t H, int32_t K,
                          const int32_t *dst_row, uint16_t *packed);
void oracle_dispatch_fp8(const uint16_t *tokens, int32_t T, int32_t H, int32_t K,
                         const int32_t *dst_row, uint8_t *packed, float *scales);
void oracle_combine(const uint16_t *y, const float *topk_weights, const int32_t *dst_row,
                    int32_t T, int32_t H, int32_t K, uint16_t *out);

static int failures = 0;

#define CHECK(cond, ...)                                   \
    do {                                                   \
        if (!(cond)) {                                     \
            fprintf(stderr, "FAIL %s:%d: ", __FILE__, __LINE__); \
            fprintf(stderr, __VA_ARGS__);                  \
            fprintf(stderr, "\n");                         \
            ++failures;                                    \
        }                                                  \
    } while (0)

#define CUDA_OK(call)                                                         \
    do {                                                                      \
        cudaError_t e_ = (call);                                              \
        if (e_ != cudaSuccess) {                                              \
            fprintf(stderr, "CUDA error %s at %s:%d\n", cudaGetErrorString(e_), \
                    __FILE__, __LINE__);                                      \
            exit(2);                                                          \
        }                                                                     \
    } while (0)

/* xorshift64*: the client's own inputs, nothing the method computes */
static uint64_t rng_state = 0x9e3779b97f4a7c15ull;
static uint64_t rng_next(void)
{
    rng_state ^= rng_state >> 12;
    rng_state ^= rng_state << 25;
    rng_state ^= rng_state >> 27;
    return rng_state * 0x2545f4914f6cdd1dull;
}
static float rng_unit(void) { return (float)((rng_next() >> 40) * (1.0 / 16777216.0)); }

static int host_checks(void)
{
    CHECK(strcmp(moe_status_string(MOE_OK), "ok") == 0, "status string of MOE_OK");
    CHECK(moe_status_string((moe_status_t)99) != NULL, "unknown status has a string");
    CHECK(moe_layout_workspace_bytes(128, 8, 256) == 0, "decode needs no workspace");
    CHECK(moe_layout_workspace_bytes(16384, 8, 128) > 0, "prefill needs a workspace");
    CHECK(moe_layout_workspace_bytes(16, 8, 100000) == 0, "invalid E");
    CHECK(moe_layout_kernels(128, 8, 256) == 1, "decode layout is one launch");
    CHECK(moe_layout_dispatch_kernels(128, 7168, 8, 256, 0) == 1, "decode layout+dispatch");
    CHECK(moe_layout_dispatch_kernels(16384, 4096, 8, 128, 1) == 2, "prefill layout+dispatch");

    /* bad arguments are refused before anything is enqueued (no GPU needed):
     * fake, never-dereferenced device addresses */
    void *fake = (void *)(uintptr_t)0x10000;
    int32_t *fi = (int32_t *)fake;
    CHECK(moe_layout(fi, 4, 2, 8, 3, fi, fi, fi, fi, fi, NULL, NULL, 0, 0) ==
              MOE_ERR_INVALID_ARG, "E %% R != 0");
    CHECK(moe_layout(fi, 4, 9, 8, 2, fi, fi, fi, fi, fi, NULL, NULL, 0, 0) ==
              MOE_ERR_INVALID_ARG, "K > E");
    CHECK(moe_layout((const int32_t *)((char *)fake + 2), 4, 2, 8, 2, fi, fi, fi, fi, fi,
                     NULL, NULL, 0, 0) == MOE_ERR_ALIGNMENT, "misaligned ids");
    CHECK(moe_layout(fi, 16384, 8, 128, 16, fi, fi, fi, fi, fi, NULL, NULL, 0, 0) ==
              MOE_ERR_WORKSPACE, "missing workspace");
    CHECK(moe_dispatch(fake, 4, 100, 2, fi, 0, fake, NULL, 0) == MOE_ERR_INVALID_ARG,
          "H %% 8 != 0");
    CHECK(moe_dispatch(fake, 4, 136, 2, fi, 1, fake, (float *)fake, 0) == MOE_ERR_INVALID_ARG,
          "FP8 needs H %% 128 == 0");
    CHECK(moe_combine(NULL, NULL, NULL, 0, 128, 2, NULL, 0) == MOE_OK, "T = 0 is a no-op");
    CHECK(moe_layout_dispatch(fi, fake, 4, 128, 2, 8, 2, 2, fi, fi, fi, fi, fi, NULL, fake,
                              NULL, NULL, 0, 0) == MOE_ERR_INVALID_ARG, "fp8 flag not 0/1");
    return failures;
}

static void *dev_copy(const void *host, size_t bytes)
{
    void *d = NULL;
    CUDA_OK(cudaMalloc(&d, bytes > 0 ? bytes : 16));
    if (host && bytes) CUDA_OK(cudaMemcpy(d, host, bytes, cudaMemcpyHostToDevice));
    return d;
}

static int same(const void *a, const void *b, size_t bytes, const char *what, int T)
{
    if (memcmp(a, b, bytes) == 0) return 1;
    fprintf(stderr, "FAIL: %s differs from the oracle (T=%d)\n", what, T);
    ++failures;
    return 0;
}

static void gpu_case(int T, int H, int K, int E, int R, int fp8)
{
    const int64_t n = (int64_t)T * K, rows = n;
    uint16_t *tokens = malloc(sizeof(uint16_t) * (size_t)T * H);
    int32_t *ids = malloc(sizeof(int32_t) * (size_t)n);
    float *w = malloc(sizeof(float) * (size_t)n);
    int32_t *perm = malloc(sizeof(int32_t) * (size_t)E);
    for (int64_t i = 0; i < (int64_t)T * H; ++i)
        tokens[i] = oracle_f32_to_bf16(8.0f * rng_unit() - 4.0f);
    for (int t = 0; t < T; ++t) {              /* K distinct experts per token */
        for (int e = 0; e < E; ++e) perm[e] = e;
        for (int k = 0; k < K; ++k) {
            int j = k + (int)(rng_next() % (uint64_t)(E - k));
            int tmp = perm[k];
            perm[k] = perm[j];
            perm[j] = tmp;
            ids[(int64_t)t * K + k] = perm[k];
            w[(int64_t)t * K + k] = rng_unit();
        }
    }

    /* the oracle */
    int32_t *o_cnt = malloc(sizeof(int32_t) * E), *o_off = malloc(sizeof(int32_t) * (E + 1));
    int32_t *o_ro = malloc(sizeof(int32_t) * (R + 1)), *o_src = malloc(sizeof(int32_t) * n);
    int32_t *o_dst = malloc(sizeof(int32_t) * n);
    uint32_t o_err = oracle_layout(ids, T, K, E, R, o_cnt, o_off, o_ro, o_src, o_dst);
    size_t row_bytes = fp8 ? (size_t)H : (size_t)H * 2, nb = (size_t)H / 128;
    uint8_t *o_packed = malloc(row_bytes * (size_t)rows);
    float *o_scales = fp8 ? malloc(sizeof(float) * nb * (size_t)rows) : NULL;
    uint16_t *o_out = malloc(sizeof(uint16_t) * (size_t)T * H);
    if (fp8) oracle_dispatch_fp8(tokens, T, H, K, o_dst, o_packed, o_scales);
    else oracle_dispatch_bf16(tokens, T, H, K, o_dst, (uint16_t *)o_packed);

    /* the library, through the C ABI only */
    int32_t *d_ids = dev_copy(ids, sizeof(int32_t) * (size_t)n);
    void *d_tok = dev_copy(tokens, sizeof(uint16_t) * (size_t)T * H);
    float *d_w = dev_copy(w, sizeof(float) * (size_t)n);
    int32_t *d_cnt = dev_copy(NULL, sizeof(int32_t) * E), *d_off = dev_copy(NULL, sizeof(int32_t) * (E + 1));
    int32_t *d_ro = dev_copy(NULL, sizeof(int32_t) * (R + 1)), *d_src = dev_copy(NULL, sizeof(int32_t) * n);
    int32_t *d_dst = dev_copy(NULL, sizeof(int32_t) * n);
    uint32_t *d_err = dev_copy(NULL, sizeof(uint32_t));
    void *d_packed = dev_copy(NULL, row_bytes * (size_t)rows);
    float *d_scales = fp8 ? dev_copy(NULL, sizeof(float) * nb * (size_t)rows) : NULL;
    size_t ws_bytes = moe_layout_workspace_bytes(T, K, E);
    void *d_ws = ws_bytes ? dev_copy(NULL, ws_bytes) : NULL;
    moe_status_t st = moe_layout_dispatch(d_ids, d_tok, T, H, K, E, R, fp8, d_cnt, d_off, d_ro,
                                          d_src, d_dst, d_err, d_packed, d_scales, d_ws,
                                          ws_bytes, 0);
    CHECK(st == MOE_OK, "moe_layout_dispatch: %s", moe_status_string(st));
    CUDA_OK(cudaDeviceSynchronize());

    int32_t *g_cnt = malloc(sizeof(int32_t) * E), *g_off = malloc(sizeof(int32_t) * (E + 1));
    int32_t *g_ro = malloc(sizeof(int32_t) * (R + 1)), *g_src = malloc(sizeof(int32_t) * n);
    int32_t *g_dst = malloc(sizeof(int32_t) * n);
    uint32_t g_err = 0xffffffffu;
    uint8_t *g_packed = malloc(row_bytes * (size_t)rows);
    CUDA_OK(cudaMemcpy(g_cnt, d_cnt, sizeof(int32_t) * E, cudaMemcpyDeviceToHost));
    CUDA_OK(cudaMemcpy(g_off, d_off, sizeof(int32_t) * (E + 1), cudaMemcpyDeviceToHost));
    CUDA_OK(cudaMemcpy(g_ro, d_ro, sizeof(int32_t) * (R + 1), cudaMemcpyDeviceToHost));
    CUDA_OK(cudaMemcpy(g_src, d_src, sizeof(int32_t) * n, cudaMemcpyDeviceToHost));
    CUDA_OK(cudaMemcpy(g_dst, d_dst, sizeof(int32_t) * n, cudaMemcpyDeviceToHost));
    CUDA_OK(cudaMemcpy(&g_err, d_err, sizeof(uint32_t), cudaMemcpyDeviceToHost));
    CUDA_OK(cudaMemcpy(g_packed, d_packed, row_bytes * (size_t)rows, cudaMemcpyDeviceToHost));
    CHECK(g_err == o_err, "error word %u against %u", g_err, o_err);
    same(g_cnt, o_cnt, sizeof(int32_t) * E, "expert_counts", T);
    same(g_off, o_off, sizeof(int32_t) * (E + 1), "expert_offsets", T);
    same(g_ro, o_ro, sizeof(int32_t) * (R + 1), "rank_offsets", T);
    same(g_src, o_src, sizeof(int32_t) * n, "src_token", T);
    same(g_dst, o_dst, sizeof(int32_t) * n, "dst_row", T);
    same(g_packed, o_packed, row_bytes * (size_t)rows, fp8 ? "FP8 codes" : "packed rows", T);
    if (fp8) {
        float *g_scales = malloc(sizeof(float) * nb * (size_t)rows);
        CUDA_OK(cudaMemcpy(g_scales, d_scales, sizeof(float) * nb * (size_t)rows,
                           cudaMemcpyDeviceToHost));
        same(g_scales, o_scales, sizeof(float) * nb * (size_t)rows, "FP8 scales", T);
        free(g_scales);
    } else {
        /* identity experts: combine the packed rows back */
        void *d_out = dev_copy(NULL, sizeof(uint16_t) * (size_t)T * H);
        st = moe_combine(d_packed, d_w, d_dst, T, H, K, d_out, 0);
        CHECK(st == MOE_OK, "moe_combine: %s", moe_status_string(st));
        CUDA_OK(cudaDeviceSynchronize());
        uint16_t *g_out = malloc(sizeof(uint16_t) * (size_t)T * H);
        CUDA_OK(cudaMemcpy(g_out, d_out, sizeof(uint16_t) * (size_t)T * H, cudaMemcpyDeviceToHost));
        oracle_combine((const uint16_t *)o_packed, w, o_dst, T, H, K, o_out);
        same(g_out, o_out, sizeof(uint16_t) * (size_t)T * H, "combine output", T);
        free(g_out);
        CUDA_OK(cudaFree(d_out));
    }
    printf("case T=%d H=%d K=%d E=%d R=%d %s: %d launches, done\n", T, H, K, E, R,
           fp8 ? "fp8" : "bf16", moe_layout_dispatch_kernels(T, H, K, E, fp8));

    void *dev[] = {d_ids, d_tok, d_w, d_cnt, d_off, d_ro, d_src, d_dst, d_err, d_packed,
                   d_scales, d_ws};
    for (size_t i = 0; i < sizeof(dev) / sizeof(dev[0]); ++i)
        if (dev[i]) CUDA_OK(cudaFree(dev[i]));
    void *host[] = {tokens, ids, w, perm, o_cnt, o_off, o_ro, o_src, o_dst, o_packed, o_scales,
                    o_out, g_cnt, g_off, g_ro, g_src, g_dst, g_packed};
    for (size_t i = 0; i < sizeof(host) / sizeof(host[0]); ++i) free(host[i]);
}

int main(int argc, char **argv)
{
    if (argc < 2 || (strcmp(argv[1], "host") && strcmp(argv[1], "gpu"))) {
        fprintf(stderr, "usage: %s host|gpu\n", argv[0]);
        return 2;
    }
    host_checks();
    if (strcmp(argv[1], "gpu") == 0) {
        gpu_case(128, 1024, 8, 64, 8, 0);      /* decode-sized: one kernel */
        gpu_case(128, 1024, 8, 64, 8, 1);
        gpu_case(4096, 1024, 8, 128, 16, 0);   /* prefill-sized: two launches */
        gpu_case(4096, 1024, 8, 128, 16, 1);
    }
    if (failures) {
        fprintf(stderr, "%d check(s) failed\n", failures);
        return 1;
    }
    printf("c client %s: all checks passed\n", argv[1]);
    return 0;
}
