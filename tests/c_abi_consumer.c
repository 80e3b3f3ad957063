/* A plain C consumer of the library: no C++, no Python, no torch. It includes
 * the public header, links libw4a16.so and exercises the calls that need no
 * device work: status strings, set-up (W4_OK with a GPU, W4_ERR_NO_DEVICE
 * without one) and argument validation, which runs before any launch. */
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime.h>

#include "w4a16.h"

/* With a device: a closed-form GEMV through plain cudaMalloc'ed buffers. Every
 * code is 9 (value +1 * step), every step 0.5 (bf16 0x3F00), x = 1 (0x3F80):
 * y[n] = K * 0.5 exactly. */
static int device_gemv(void)
{
    const int M = 1, N = 256, K = 4096, group = 32;
    const size_t nw = (size_t)N * K / 8, ns = (size_t)N * K / group;
    uint32_t *hq = malloc(nw * sizeof(uint32_t));
    uint16_t *hs = malloc(ns * sizeof(uint16_t)), *hx = malloc((size_t)K * sizeof(uint16_t));
    float *hy = malloc((size_t)N * sizeof(float));
    if (!hq || !hs || !hx || !hy)
        return 10;
    for (size_t i = 0; i < nw; ++i)
        hq[i] = 0x99999999u;
    for (size_t i = 0; i < ns; ++i)
        hs[i] = 0x3F00;
    for (int i = 0; i < K; ++i)
        hx[i] = 0x3F80;
    uint32_t *dq = NULL;
    uint16_t *ds = NULL, *dx = NULL;
    float *dy = NULL;
    if (cudaMalloc((void **)&dq, nw * sizeof(uint32_t)) != cudaSuccess ||
        cudaMalloc((void **)&ds, ns * sizeof(uint16_t)) != cudaSuccess ||
        cudaMalloc((void **)&dx, (size_t)K * sizeof(uint16_t)) != cudaSuccess ||
        cudaMalloc((void **)&dy, (size_t)N * sizeof(float)) != cudaSuccess)
        return 11;
    cudaMemcpy(dq, hq, nw * sizeof(uint32_t), cudaMemcpyHostToDevice);
    cudaMemcpy(ds, hs, ns * sizeof(uint16_t), cudaMemcpyHostToDevice);
    cudaMemcpy(dx, hx, (size_t)K * sizeof(uint16_t), cudaMemcpyHostToDevice);
    const int rc = w4a16_gemv(dy, dx, dq, ds, M, N, K, group, NULL);
    if (rc != W4_OK) {
        fprintf(stderr, "w4a16_gemv: %s %s\n", w4_status_string(rc), w4_last_cuda_error());
        return 12;
    }
    if (cudaMemcpy(hy, dy, (size_t)N * sizeof(float), cudaMemcpyDeviceToHost) != cudaSuccess)
        return 13;
    for (int n = 0; n < N; ++n)
        if (hy[n] != 0.5f * (float)K) {
            fprintf(stderr, "y[%d] = %g, want %g\n", n, hy[n], 0.5 * K);
            return 14;
        }
    int32_t code = -1;
    if (w4_device_error(&code) != W4_OK || code != 0)
        return 15;
    cudaFree(dq);
    cudaFree(ds);
    cudaFree(dx);
    cudaFree(dy);
    free(hq);
    free(hs);
    free(hx);
    free(hy);
    return 0;
}

int main(void)
{
    if (strcmp(w4_status_string(W4_OK), "W4_OK") != 0 ||
        strcmp(w4_status_string(W4_ERR_MISALIGNED), "W4_ERR_MISALIGNED") != 0) {
        fprintf(stderr, "status strings\n");
        return 1;
    }
    const int init = w4_init();
    if (init != W4_OK && init != W4_ERR_NO_DEVICE) {
        fprintf(stderr, "w4_init: %d (%s)\n", init, w4_status_string(init));
        return 2;
    }
    /* NULL output: rejected by validation, no device touched. */
    if (w4a16_gemv(NULL, NULL, NULL, NULL, 1, 16, 64, 32, NULL) != W4_ERR_INVALID_ARG) {
        fprintf(stderr, "validation\n");
        return 3;
    }
    /* An unsupported group size. */
    char buf[64] __attribute__((aligned(16)));
    if (w4a16_gemv((float *)buf, (const uint16_t *)buf, (const uint32_t *)buf, (const uint16_t *)buf, 1, 16,
                   96, 48, NULL) != W4_ERR_UNSUPPORTED) {
        fprintf(stderr, "group check\n");
        return 4;
    }
    if (init == W4_OK) {
        const int rc = device_gemv();
        if (rc != 0)
            return rc;
        printf("device GEMV through cudaMalloc'ed buffers: exact\n");
    }
    printf("c consumer ok (w4_init = %s)\n", w4_status_string(init));
    return 0;
}
