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
// W2 and its scales keep the canonical layout.  In the FP4-weight format the
// same row order applies to the packed E2M1 rows and to their per-32 UE8M0
// scale rows.
#include "moe_device.cuh"
#include "moe_internal.h"

namespace moe {
namespace {

// Rows of [E, 2I, row_bytes] in the interleaved order, written with a row
// pitch of dst_pitch bytes; row_bytes and dst_pitch multiples of 4.
__global__ void interleave_rows_kernel(const uint8_t *__restrict__ src_rows, uint8_t *__restrict__ dst_rows,
                                       int rows_total, int row_bytes, int dst_pitch, int I) {
    const int words = row_bytes / 4;
    for (int row = blockIdx.x; row < rows_total; row += gridDim.x) {
        const int e = row / (2 * I);
        const int r = row - e * 2 * I;
        const int g = r >> 4, m = r & 15;
        const int src = (m < 8) ? (8 * g + m) : (I + 8 * g + m - 8);
        const uint32_t *s = reinterpret_cast<const uint32_t *>(src_rows + ((size_t)e * 2 * I + src) * row_bytes);
        uint32_t *d = reinterpret_cast<uint32_t *>(dst_rows + (size_t)row * dst_pitch);
        for (int v = threadIdx.x; v < words; v += blockDim.x) d[v] = s[v];
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

void launch_transform_w1(const uint8_t *w1, const float *w1_sf, uint8_t *w1i, int w1i_pitch,
                         float2 *w1i_sf, int E, int H, int I, cudaStream_t s) {
    const int rows = E * 2 * I;
    interleave_rows_kernel<<<min(rows, 65535), 256, 0, s>>>(w1, w1i, rows, H, w1i_pitch, I);
    const int n = E * (2 * I / 128) * (H / 128);
    interleave_w1_sf_kernel<<<min((n + 255) / 256, 4096), 256, 0, s>>>(w1_sf, w1i_sf, E, H, I);
}

void launch_interleave_rows(const uint8_t *src, uint8_t *dst, int E, int I, int row_bytes,
                            int dst_pitch, cudaStream_t s) {
    const int rows = E * 2 * I;
    interleave_rows_kernel<<<min(rows, 65535), 128, 0, s>>>(src, dst, rows, row_bytes, dst_pitch, I);
}

}  // namespace moe
