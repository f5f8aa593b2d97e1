/* One forward of the expert layer driven from plain C through the library's
 * C ABI (include/moe.h): the caller sizes and allocates the workspace and
 * the weight store, transforms canonical FP8 weights, runs the forward on
 * the default stream and reads y back.  Inputs come from a bundle file,
 * the output goes to a file of raw BF16 bits.
 *
 *   forward_from_c <bundle> <y_out>
 *
 * Bundle: five int32 (T, H, I, E, k), then x u8 [T,H], x_sf f32 [T,H/128],
 * topk_idx int32 [T,k], topk_weights f32 [T,k], w1 u8 [E,2I,H],
 * w1_sf f32 [E,2I/128,H/128], w2 u8 [E,H,I], w2_sf f32 [E,H/128,I/128].
 * Exit status 0 on success, 1 bad arguments or file, 2 CUDA error, 3 library
 * error. */
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>

#include <cuda_runtime.h>

#include "moe.h"

#define CUDA_OK(call)                                                              \
    do {                                                                           \
        cudaError_t e_ = (call);                                                   \
        if (e_ != cudaSuccess) {                                                   \
            fprintf(stderr, "%s: %s\n", #call, cudaGetErrorString(e_));            \
            return 2;                                                              \
        }                                                                          \
    } while (0)

#define MOE_OK_OR_EXIT(call)                                                       \
    do {                                                                           \
        int r_ = (call);                                                           \
        if (r_ != MOE_OK) {                                                        \
            fprintf(stderr, "%s: %s\n", #call, moe_strerror(r_));                  \
            return 3;                                                              \
        }                                                                          \
    } while (0)

enum { X, XSF, IDX, W, W1, W1SF, W2, W2SF, NBUF };

int main(int argc, char **argv) {
    if (argc != 3) {
        fprintf(stderr, "usage: %s <bundle> <y_out>\n", argv[0]);
        return 1;
    }
    FILE *f = fopen(argv[1], "rb");
    int32_t hdr[5];
    if (!f || fread(hdr, sizeof(int32_t), 5, f) != 5) return 1;
    const size_t T = hdr[0], H = hdr[1], I = hdr[2], E = hdr[3], k = hdr[4];
    const size_t bytes[NBUF] = {
        T * H, T * (H / 128) * 4, T * k * 4, T * k * 4,
        E * 2 * I * H, E * (2 * I / 128) * (H / 128) * 4, E * H * I, E * (H / 128) * (I / 128) * 4,
    };
    void *host[NBUF], *dev[NBUF];
    for (int i = 0; i < NBUF; ++i) {
        host[i] = malloc(bytes[i]);
        if (!host[i] || fread(host[i], 1, bytes[i], f) != bytes[i]) return 1;
    }
    fclose(f);

    CUDA_OK(cudaSetDevice(0));
    const moe_config cfg = {(int)T, (int)H, (int)I, (int)E, (int)k, MOE_W_FP8_BLK128, INFINITY, 0};
    const size_t ws_bytes = moe_workspace_bytes(&cfg), wt_bytes = moe_weight_bytes(&cfg);
    if (!ws_bytes || !wt_bytes) return 3;
    void *ws = NULL, *wt = NULL, *y = NULL;
    CUDA_OK(cudaMalloc(&ws, ws_bytes));   /* 256-byte aligned, as moe_create requires */
    CUDA_OK(cudaMalloc(&wt, wt_bytes));
    CUDA_OK(cudaMalloc(&y, T * H * 2));
    for (int i = 0; i < NBUF; ++i) {
        CUDA_OK(cudaMalloc(&dev[i], bytes[i]));
        CUDA_OK(cudaMemcpy(dev[i], host[i], bytes[i], cudaMemcpyHostToDevice));
    }

    moe_ctx *ctx = NULL;
    MOE_OK_OR_EXIT(moe_create(&ctx, &cfg, ws, wt));
    MOE_OK_OR_EXIT(moe_transform_weights(ctx, dev[W1], dev[W1SF], dev[W2], dev[W2SF], NULL));
    CUDA_OK(cudaDeviceSynchronize());
    /* the canonical weights are no longer needed once the transform has run */
    for (int i = W1; i <= W2SF; ++i) CUDA_OK(cudaFree(dev[i]));

    MOE_OK_OR_EXIT(moe_forward(ctx, (int)T, dev[X], dev[XSF], (const int32_t *)dev[IDX], (const float *)dev[W], y,
                               NULL, NULL));
    CUDA_OK(cudaDeviceSynchronize());
    MOE_OK_OR_EXIT(moe_device_status(ctx));

    uint16_t *hy = (uint16_t *)malloc(T * H * 2);
    if (!hy) return 1;
    CUDA_OK(cudaMemcpy(hy, y, T * H * 2, cudaMemcpyDeviceToHost));
    FILE *o = fopen(argv[2], "wb");
    if (!o || fwrite(hy, 2, T * H, o) != T * H) return 1;
    fclose(o);

    moe_destroy(ctx);
    for (int i = X; i <= W; ++i) CUDA_OK(cudaFree(dev[i]));
    CUDA_OK(cudaFree(y));
    CUDA_OK(cudaFree(wt));
    CUDA_OK(cudaFree(ws));
    for (int i = 0; i < NBUF; ++i) free(host[i]);
    free(hy);
    return 0;
}
