/*
 * The C ABI used from plain C99: no Python, no PyTorch. Device memory comes
 * from the CUDA runtime's C API; every value checked is fixed by a closed form
 * (no oracle needed):
 *
 *  - host helpers: the vocabulary padding of the LIT-022 digest ("Key
 *    takeaways": 50,257 ids padded to 51,200 for t = 8, a multiple of 128 t),
 *    and a shape the host check rejects (f % t != 0) before any launch;
 *  - tp_mlp_forward with A the identity on its first h columns (zero beyond)
 *    and B the identity on its first h rows: U = X on those columns, Y =
 *    GeLU(U) and Z = Y[:, :h], so Z = GeLU(X) elementwise up to the bf16
 *    roundings of Y and Z ("Mathematical Foundations of Megatron-LM 1D
 *    Slicing", sections "Column-Parallel Linear Layer" and "Row-Parallel
 *    Linear Layer": the shard that owns the identity columns carries the
 *    result, the other shard adds exact zeros);
 *  - vocab_parallel_ce with E = 0: every logit is 0, so loss = ln(v_valid)
 *    for every token whatever its target, dH = dl E = 0 exactly, and the
 *    padded rows of dE are 0.
 *
 * Prints "tpce C ABI smoke: ok" and exits 0, or names the first failure and
 * exits 1. Built and run by tests/test_c_abi.py.
 */
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime_api.h>

#include "tpce.h"

static int failures = 0;

#define CHECK(cond, ...)                      \
    do {                                      \
        if (!(cond)) {                        \
            fprintf(stderr, "FAIL: ");        \
            fprintf(stderr, __VA_ARGS__);     \
            fprintf(stderr, "\n");            \
            ++failures;                       \
        }                                     \
    } while (0)

/* bf16 <-> fp32 by the bit pattern (round to nearest even; no NaNs here) */
static uint16_t to_bf16(float f) {
    uint32_t u;
    memcpy(&u, &f, 4);
    u += 0x7FFFu + ((u >> 16) & 1u);
    return (uint16_t)(u >> 16);
}
static float from_bf16(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}

/* a fixed sequence of values in [-3, 3) */
static float next_value(uint32_t *s) {
    *s = *s * 1664525u + 1013904223u;
    return 6.0f * (float)(*s >> 8) / 16777216.0f - 3.0f;
}

static void *dev_copy(const void *host, size_t bytes) {
    void *d = NULL;
    if (cudaMalloc(&d, bytes) != cudaSuccess) return NULL;
    if (host && cudaMemcpy(d, host, bytes, cudaMemcpyHostToDevice) != cudaSuccess) return NULL;
    if (!host && cudaMemset(d, 0, bytes) != cudaSuccess) return NULL;
    return d;
}

static void host_helpers(void) {
    CHECK(tpce_version() > 0, "tpce_version");
    CHECK(tpce_pad_vocab(50257, 8, 128) == 51200, "pad_vocab(50257, 8, 128) = %lld",
          (long long)tpce_pad_vocab(50257, 8, 128));
    CHECK(tpce_status_string(TPCE_ERR_SHAPE) != NULL, "status string");
    /* f % t != 0: rejected by the host check, nothing is launched or dereferenced */
    tpce_status st = tp_mlp_forward((void *)16, (void *)16, NULL, (void *)16, NULL, 32, 64, 250, 4, TPCE_BF16,
                                    (void *)16, (void *)16, (void *)16, NULL, 0, NULL);
    CHECK(st == TPCE_ERR_SHAPE, "f %% t != 0 gave status %d", (int)st);
}

static void mlp_identity(void) {
    const int64_t T = 128, h = 64, f = 128;
    const int t = 2;
    uint16_t *X = malloc(T * h * 2), *A = calloc(h * f, 2), *B = calloc(f * h, 2), *Z = malloc(T * h * 2);
    uint32_t seed = 12345u;
    for (int64_t i = 0; i < T * h; ++i) X[i] = to_bf16(next_value(&seed));
    for (int64_t i = 0; i < h; ++i) {
        A[i * f + i] = to_bf16(1.0f); /* A [h, f]: identity on columns 0 .. h-1 */
        B[i * h + i] = to_bf16(1.0f); /* B [f, h]: identity on rows 0 .. h-1 */
    }
    void *dX = dev_copy(X, T * h * 2), *dA = dev_copy(A, h * f * 2), *dB = dev_copy(B, f * h * 2);
    void *dZ = dev_copy(NULL, T * h * 2), *dU = dev_copy(NULL, T * f * 2), *dY = dev_copy(NULL, T * f * 2);
    CHECK(dX && dA && dB && dZ && dU && dY, "device allocations");
    if (failures) return;
    tpce_status st = tp_mlp_forward(dX, dA, NULL, dB, NULL, T, h, f, t, TPCE_BF16, dZ, dU, dY, NULL, 0, NULL);
    CHECK(st == TPCE_OK, "tp_mlp_forward: %s (%s)", tpce_status_string(st), tpce_last_error());
    CHECK(cudaMemcpy(Z, dZ, T * h * 2, cudaMemcpyDeviceToHost) == cudaSuccess, "copy Z back");
    double worst = 0.0;
    for (int64_t i = 0; i < T * h; ++i) {
        const double x = from_bf16(X[i]);
        const double g = 0.5 * x * (1.0 + erf(x / sqrt(2.0))); /* GeLU(x) = x Phi(x) */
        const double err = fabs(from_bf16(Z[i]) - g) / (fabs(g) + 1e-6);
        if (err > worst) worst = err;
    }
    /* Y is GeLU(U) rounded once to bf16 (2^-9 relative) and Z = Y (one nonzero term per sum) */
    CHECK(worst <= 1.0 / 256.0, "Z = GeLU(X): worst relative error %.3e", worst);
    void *dev[] = {dX, dA, dB, dZ, dU, dY};
    for (size_t i = 0; i < sizeof dev / sizeof dev[0]; ++i) cudaFree(dev[i]);
    free(X);
    free(A);
    free(B);
    free(Z);
}

static void ce_zero_embedding(void) {
    const int64_t T = 96, h = 64, v_pad = 512, v_valid = 500;
    const int t = 2;
    uint16_t *H = malloc(T * h * 2), *dHh = malloc(T * h * 2), *dEh = malloc(v_pad * h * 2);
    int32_t *y = malloc(T * 4);
    float *loss = malloc(T * 4), *lse = malloc(T * 4);
    uint32_t seed = 777u;
    for (int64_t i = 0; i < T * h; ++i) H[i] = to_bf16(next_value(&seed));
    for (int64_t i = 0; i < T; ++i) y[i] = (int32_t)((i * 37) % v_valid);
    const size_t ws_bytes = tpce_ce_workspace_bytes(T, h, v_pad, t, TPCE_BF16, 1);
    void *dH_in = dev_copy(H, T * h * 2), *dE_in = dev_copy(NULL, v_pad * h * 2), *dy = dev_copy(y, T * 4);
    void *dloss = dev_copy(NULL, T * 4), *dlse = dev_copy(NULL, T * 4);
    void *ddH = dev_copy(NULL, T * h * 2), *ddE = dev_copy(NULL, v_pad * h * 2), *ws = dev_copy(NULL, ws_bytes);
    CHECK(ws_bytes > 0 && dH_in && dE_in && dy && dloss && dlse && ddH && ddE && ws, "device allocations");
    if (failures) return;
    /* dE and dH poisoned first, so that "written as zero" is what is checked */
    cudaMemset(ddH, 0x7f, T * h * 2);
    cudaMemset(ddE, 0x7f, v_pad * h * 2);
    tpce_status st = vocab_parallel_ce(dH_in, dE_in, dy, T, h, v_pad, v_valid, t, 1.0f, TPCE_BF16, dloss, dlse, ddH,
                                       ddE, ws, ws_bytes, NULL);
    CHECK(st == TPCE_OK, "vocab_parallel_ce: %s (%s)", tpce_status_string(st), tpce_last_error());
    cudaMemcpy(loss, dloss, T * 4, cudaMemcpyDeviceToHost);
    cudaMemcpy(lse, dlse, T * 4, cudaMemcpyDeviceToHost);
    cudaMemcpy(dHh, ddH, T * h * 2, cudaMemcpyDeviceToHost);
    cudaMemcpy(dEh, ddE, v_pad * h * 2, cudaMemcpyDeviceToHost);
    const double ln_v = log((double)v_valid);
    double worst = 0.0;
    for (int64_t i = 0; i < T; ++i) {
        const double e = fmax(fabs(loss[i] - ln_v), fabs(lse[i] - ln_v));
        if (e > worst) worst = e;
    }
    CHECK(worst <= 1e-5, "loss = lse = ln(v_valid): worst error %.3e", worst);
    int64_t nonzero_dH = 0, nonzero_pad = 0;
    for (int64_t i = 0; i < T * h; ++i) nonzero_dH += (dHh[i] & 0x7fff) != 0;
    for (int64_t i = v_valid * h; i < v_pad * h; ++i) nonzero_pad += (dEh[i] & 0x7fff) != 0;
    CHECK(nonzero_dH == 0, "dH = dl E = 0: %lld nonzero", (long long)nonzero_dH);
    CHECK(nonzero_pad == 0, "padded rows of dE = 0: %lld nonzero", (long long)nonzero_pad);
    void *dev[] = {dH_in, dE_in, dy, dloss, dlse, ddH, ddE, ws};
    for (size_t i = 0; i < sizeof dev / sizeof dev[0]; ++i) cudaFree(dev[i]);
    free(H);
    free(dHh);
    free(dEh);
    free(y);
    free(loss);
    free(lse);
}

int main(void) {
    host_helpers();
    mlp_identity();
    ce_zero_embedding();
    uint32_t detail = 0;
    const tpce_status ds = tpce_device_status(NULL, 0, &detail);
    CHECK(ds == TPCE_OK, "device status %d (detail 0x%x)", (int)ds, (unsigned)detail);
    if (failures) {
        fprintf(stderr, "tpce C ABI smoke: %d failure(s)\n", failures);
        return 1;
    }
    printf("tpce C ABI smoke: ok\n");
    return 0;
}
