// moe_transform.cu -- canonical weights -> kernel layout.
//
// W1 rows are interleaved in groups of 8 along N: interleaved row 16g + m is
// gate row 8g + m for m < 8 and up row I + 8g + m - 8 otherwise (MegaMoE SM90
// Implementation Design (Final), §15.1 "SM90 Weight Transform"), so every
// 256-row tile of the L1 GEMM holds 128 matching gate/up pairs and every
// thread of its epilogue sees both halves of its SwiGLU inputs.  An
// interleaved 128-row block j holds gate rows [64j, 64j+64) and up rows
// [I+64j, I+64j+64): its scales are the pair (gate block j/2, up block
// I/128 + j/2) of the canonical [E, 2I/128, H/128] scale array (design §15.2).
// W2 and its scales keep the canonical layout.
#include "moe_device.cuh"
#include "moe_internal.h"

namespace moe {
namespace {

__global__ void interleave_w1_kernel(const uint8_t *__restrict__ w1, uint8_t *__restrict__ w1i,
                                     int rows_total, int H, int I) {
    const int vecs = H / 16;
    for (int row = blockIdx.x; row < rows_total; row += gridDim.x) {
        const int e = row / (2 * I);
        const int r = row - e * 2 * I;
        const int g = r >> 4, m = r & 15;
        const int src = (m < 8) ? (8 * g + m) : (I + 8 * g + m - 8);
        const uint4 *s = reinterpret_cast<const uint4 *>(w1 + ((size_t)e * 2 * I + src) * H);
        uint4 *d = reinterpret_cast<uint4 *>(w1i + (size_t)row * H);
        for (int v = threadIdx.x; v < vecs; v += blockDim.x) d[v] = s[v];
    }
}

__global__ void interleave_w1_sf_kernel(const float *__restrict__ sf, float2 *__restrict__ sfi, int E,
                                        int H, int I) {
    const int KB = H / 128, NBLK = 2 * I / 128;
    const int n = E * NBLK * KB;
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x) {
        const int kb = i % KB;
        const int j = (i / KB) % NBLK;
        const int e = i / (KB * NBLK);
        const float g = sf[((size_t)e * NBLK + j / 2) * KB + kb];
        const float u = sf[((size_t)e * NBLK + I / 128 + j / 2) * KB + kb];
        sfi[i] = make_float2(g, u);
    }
}

}  // namespace

void launch_transform_w1(const uint8_t *w1, const float *w1_sf, uint8_t *w1i, float2 *w1i_sf, int E,
                         int H, int I, cudaStream_t s) {
    const int rows = E * 2 * I;
    interleave_w1_kernel<<<min(rows, 65535), 256, 0, s>>>(w1, w1i, rows, H, I);
    const int n = E * (2 * I / 128) * (H / 128);
    interleave_w1_sf_kernel<<<min((n + 255) / 256, 4096), 256, 0, s>>>(w1_sf, w1i_sf, E, H, I);
}

}  // namespace moe
