/*
 * A plain C11 caller of libmoe_finalize.so: device memory from the CUDA
 * runtime, the library's C ABI, results checked against closed forms.
 *
 *  1. finalize + RMSNorm (flashinfer.comm.tp_moe_finalize_rmsnorm): every
 *     gathered row is the constant 1 and the 8 weights are 1/8, so acc = 1;
 *     norm_weight 0 with gain_center 1 gives g = 1, and eps = 3 gives
 *     y = 1 / sqrt(1 + 3) = 0.5 exactly, for both orderings.  A token whose
 *     slots are all invalid gives 0.
 *  2. Beam finalize (beam_moe_finalize): top_k 1, weight 1, scale 1, no norm
 *     returns its input bit for bit.
 *  3. A misaligned output pointer is rejected with MF_ERR_ALIGN before any launch.
 *
 * Exit status 0 when every check passes.
 */
#include <cuda_runtime.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include "moe_finalize.h"

#define CHECK(cond, ...)                                   \
    do {                                                   \
        if (!(cond)) {                                     \
            fprintf(stderr, "FAIL %s:%d: ", __FILE__, __LINE__); \
            fprintf(stderr, __VA_ARGS__);                  \
            fputc('\n', stderr);                           \
            return 1;                                      \
        }                                                  \
    } while (0)

static uint16_t bf16(float f) {
    uint32_t u;
    memcpy(&u, &f, 4);
    return (uint16_t)(u >> 16); /* exact for the values used here */
}

static int finalize_closed_form(int before) {
    enum { T = 5, K = 8, H = 4096, ROWS = 40 };
    uint16_t *h_rows = malloc(sizeof(uint16_t) * ROWS * H);
    uint16_t *h_out = malloc(sizeof(uint16_t) * T * H);
    uint16_t h_nw[H];
    int32_t h_idx[T * K];
    float h_w[T * K];
    for (int i = 0; i < ROWS * H; ++i) h_rows[i] = bf16(1.0f);
    for (int h = 0; h < H; ++h) h_nw[h] = 0;
    for (int t = 0; t < T; ++t)
        for (int k = 0; k < K; ++k) {
            h_idx[t * K + k] = (t == T - 1) ? -1 : (t * K + k) % ROWS; /* last token: none valid */
            h_w[t * K + k] = 0.125f;
        }
    void *d_rows, *d_w, *d_idx, *d_nw, *d_out;
    CHECK(cudaMalloc(&d_rows, sizeof(uint16_t) * ROWS * H) == cudaSuccess, "cudaMalloc");
    CHECK(cudaMalloc(&d_w, sizeof h_w) == cudaSuccess, "cudaMalloc");
    CHECK(cudaMalloc(&d_idx, sizeof h_idx) == cudaSuccess, "cudaMalloc");
    CHECK(cudaMalloc(&d_nw, sizeof h_nw) == cudaSuccess, "cudaMalloc");
    CHECK(cudaMalloc(&d_out, sizeof(uint16_t) * T * H) == cudaSuccess, "cudaMalloc");
    cudaMemcpy(d_rows, h_rows, sizeof(uint16_t) * ROWS * H, cudaMemcpyHostToDevice);
    cudaMemcpy(d_w, h_w, sizeof h_w, cudaMemcpyHostToDevice);
    cudaMemcpy(d_idx, h_idx, sizeof h_idx, cudaMemcpyHostToDevice);
    cudaMemcpy(d_nw, h_nw, sizeof h_nw, cudaMemcpyHostToDevice);

    mf_status st = moe_finalize_rmsnorm(d_rows, ROWS, H, d_w, MF_DTYPE_FP32, (const int32_t *)d_idx,
                                        d_nw, d_out, T, H, K, 3.0f, 1.0f, before, NULL);
    CHECK(st == MF_OK, "moe_finalize_rmsnorm: %s", mf_status_string(st));
    CHECK(cudaMemcpy(h_out, d_out, sizeof(uint16_t) * T * H, cudaMemcpyDeviceToHost) == cudaSuccess,
          "copy back");
    for (int t = 0; t < T; ++t)
        for (int h = 0; h < H; ++h) {
            uint16_t want = (t == T - 1) ? 0 : bf16(0.5f);
            CHECK(h_out[t * H + h] == want, "token %d col %d: 0x%04x != 0x%04x", t, h,
                  h_out[t * H + h], want);
        }
    /* a misaligned output is rejected before anything runs */
    st = moe_finalize_rmsnorm(d_rows, ROWS, H, d_w, MF_DTYPE_FP32, (const int32_t *)d_idx, d_nw,
                              (char *)d_out + 8, T, H, K, 3.0f, 1.0f, before, NULL);
    CHECK(st == MF_ERR_ALIGN, "misaligned output: %s", mf_status_string(st));
    cudaFree(d_rows); cudaFree(d_w); cudaFree(d_idx); cudaFree(d_nw); cudaFree(d_out);
    free(h_rows); free(h_out);
    return 0;
}

static int beam_identity(void) {
    enum { CAP = 6, LIVE = 5, H = 512 };
    uint16_t h_x[CAP * H], h_out[LIVE * H];
    float h_w[CAP];
    for (int i = 0; i < CAP * H; ++i) h_x[i] = (uint16_t)(0x3F00 + (i * 37) % 1024); /* finite BF16 */
    for (int t = 0; t < CAP; ++t) h_w[t] = 1.0f;
    void *d_x, *d_w, *d_out;
    CHECK(cudaMalloc(&d_x, sizeof h_x) == cudaSuccess, "cudaMalloc");
    CHECK(cudaMalloc(&d_w, sizeof h_w) == cudaSuccess, "cudaMalloc");
    CHECK(cudaMalloc(&d_out, sizeof h_out) == cudaSuccess, "cudaMalloc");
    cudaMemcpy(d_x, h_x, sizeof h_x, cudaMemcpyHostToDevice);
    cudaMemcpy(d_w, h_w, sizeof h_w, cudaMemcpyHostToDevice);
    mf_status st = beam_moe_finalize(d_x, CAP, (const float *)d_w, CAP, d_out, LIVE, 1, H, 1.0f,
                                     NULL, 0.0f, 0, NULL);
    CHECK(st == MF_OK, "beam_moe_finalize: %s", mf_status_string(st));
    CHECK(cudaMemcpy(h_out, d_out, sizeof h_out, cudaMemcpyDeviceToHost) == cudaSuccess, "copy");
    CHECK(memcmp(h_out, h_x, sizeof h_out) == 0, "Beam identity differs");
    cudaFree(d_x); cudaFree(d_w); cudaFree(d_out);
    return 0;
}

int main(void) {
    if (finalize_closed_form(0) || finalize_closed_form(1) || beam_identity()) return 1;
    mf_status st = mf_device_status(1);
    CHECK(st == MF_OK, "device status: %s", mf_status_string(st));
    printf("c abi: ok (library version %d)\n", (int)mf_version());
    return 0;
}
