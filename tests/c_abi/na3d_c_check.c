/* The NA3D C ABI called from C, without Python: device buffers from the CUDA
 * runtime, na3d_fwd on problems whose results have a closed form, and the
 * status codes of invalid arguments. Test infrastructure (built and run by
 * tests/test_c_abi.py); exit status 0 when every check passes.
 *
 *  1. Window (1,1,1): every query attends to its own key only (p = 1, l = 1),
 *     so out equals v bit for bit.
 *  2. v constant (0.75, exact in bf16), window (3,5,5): every output is the
 *     constant, within one bf16 ulp (2^-8 at 0.75).
 *  3. An even window length returns NA3D_ERR_KERNEL, a NULL pointer
 *     NA3D_ERR_NULL, both before anything is launched.
 */
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime.h>

#include "na3d.h"

static uint64_t rng_state = 0x9E3779B97F4A7C15ull;

static uint64_t next_u64(void) { /* xorshift64* */
    rng_state ^= rng_state >> 12;
    rng_state ^= rng_state << 25;
    rng_state ^= rng_state >> 27;
    return rng_state * 0x2545F4914F6CDD1Dull;
}

/* float -> bf16, round to nearest even (finite inputs) */
static uint16_t to_bf16(float f) {
    uint32_t u;
    memcpy(&u, &f, 4);
    u += 0x7FFFu + ((u >> 16) & 1u);
    return (uint16_t)(u >> 16);
}

static float from_bf16(uint16_t h) {
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}

#define CHECK_CUDA(x)                                                              \
    do {                                                                           \
        cudaError_t e_ = (x);                                                      \
        if (e_ != cudaSuccess) {                                                   \
            fprintf(stderr, "%s: %s\n", #x, cudaGetErrorString(e_));               \
            return 1;                                                              \
        }                                                                          \
    } while (0)

int main(void) {
    const int64_t B = 2, T = 5, H = 7, W = 9, NH = 2, HD = 64;
    const size_t n = (size_t)(B * T * H * W * NH * HD);
    const size_t bytes = n * sizeof(uint16_t);
    uint16_t *hq = malloc(bytes), *hk = malloc(bytes), *hv = malloc(bytes), *ho = malloc(bytes);
    if (!hq || !hk || !hv || !ho) return 1;
    const float scale = 1.0f / sqrtf((float)HD);
    for (size_t i = 0; i < n; ++i) {
        /* uniform in [-2, 2) */
        const float a = (float)(next_u64() >> 40) / (float)(1u << 24) * 4.0f - 2.0f;
        const float b = (float)(next_u64() >> 40) / (float)(1u << 24) * 4.0f - 2.0f;
        const float c = (float)(next_u64() >> 40) / (float)(1u << 24) * 4.0f - 2.0f;
        hq[i] = to_bf16(a * scale);
        hk[i] = to_bf16(b);
        hv[i] = to_bf16(c);
    }
    void *dq, *dk, *dv, *dout;
    CHECK_CUDA(cudaMalloc(&dq, bytes));
    CHECK_CUDA(cudaMalloc(&dk, bytes));
    CHECK_CUDA(cudaMalloc(&dv, bytes));
    CHECK_CUDA(cudaMalloc(&dout, bytes));
    CHECK_CUDA(cudaMemcpy(dq, hq, bytes, cudaMemcpyHostToDevice));
    CHECK_CUDA(cudaMemcpy(dk, hk, bytes, cudaMemcpyHostToDevice));
    CHECK_CUDA(cudaMemcpy(dv, hv, bytes, cudaMemcpyHostToDevice));
    cudaStream_t stream;
    CHECK_CUDA(cudaStreamCreate(&stream));
    int failures = 0;

    /* 1. window (1,1,1) returns v */
    int rc = na3d_fwd(dq, dk, dv, dout, B, T, H, W, NH, HD, 1, 1, 1, stream);
    CHECK_CUDA(cudaStreamSynchronize(stream));
    CHECK_CUDA(cudaMemcpy(ho, dout, bytes, cudaMemcpyDeviceToHost));
    size_t diff = 0;
    for (size_t i = 0; i < n; ++i) diff += ho[i] != hv[i];
    printf("window (1,1,1): status %d (%s), %zu of %zu outputs differ from v\n", rc,
           na3d_status_string(rc), diff, n);
    failures += rc != NA3D_OK || diff != 0;

    /* 2. constant v */
    for (size_t i = 0; i < n; ++i) hv[i] = to_bf16(0.75f);
    CHECK_CUDA(cudaMemcpy(dv, hv, bytes, cudaMemcpyHostToDevice));
    rc = na3d_fwd(dq, dk, dv, dout, B, T, H, W, NH, HD, 3, 5, 5, stream);
    CHECK_CUDA(cudaStreamSynchronize(stream));
    CHECK_CUDA(cudaMemcpy(ho, dout, bytes, cudaMemcpyDeviceToHost));
    double worst = 0.0;
    for (size_t i = 0; i < n; ++i) {
        const double e = fabs((double)from_bf16(ho[i]) - 0.75);
        if (!(e <= worst)) worst = e; /* also catches NaN */
    }
    printf("constant v, window (3,5,5): status %d, max |out - 0.75| = %g\n", rc, worst);
    failures += rc != NA3D_OK || !(worst <= 1.0 / 256.0);

    /* 3. argument errors, returned before any launch */
    rc = na3d_fwd(dq, dk, dv, dout, B, T, H, W, NH, HD, 3, 4, 5, stream);
    printf("even window length: status %d (%s)\n", rc, na3d_status_string(rc));
    failures += rc != NA3D_ERR_KERNEL;
    rc = na3d_fwd(NULL, dk, dv, dout, B, T, H, W, NH, HD, 3, 5, 5, stream);
    printf("NULL q: status %d (%s)\n", rc, na3d_status_string(rc));
    failures += rc != NA3D_ERR_NULL;

    rc = na3d_device_status(stream);
    printf("device status: %d\n", rc);
    failures += rc != NA3D_OK;

    cudaStreamDestroy(stream);
    cudaFree(dq);
    cudaFree(dk);
    cudaFree(dv);
    cudaFree(dout);
    free(hq);
    free(hk);
    free(hv);
    free(ho);
    printf("%s\n", failures ? "FAILED" : "all checks passed");
    return failures ? 1 : 0;
}
