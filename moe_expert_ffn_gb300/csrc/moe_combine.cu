// moe_combine.cu -- top-k combine reduce back to BF16 y.
//
// y[t, h] = bf16( sum over active slots j = 0..k-1, in slot order, of the
// BF16 L2 output of pair (t, j) taken to FP32 ), the accumulator starting at
// zero (MegaMoE SM90 Implementation Design (Final), §11.2 "Combine Reduce";
// PR357 Green-Context Split MegaMoE code review, §6.3 "K3 combine_reduce").
// The pages' cross-rank combine buffer is, on one GPU, the L2 output in pool
// order plus the pair -> pool-row map from dispatch.
//
// HBM-bound: every thread owns 8 consecutive hidden columns (one 16-byte
// vector), issues the loads of all slots before summing, and writes one
// 16-byte vector of y.
#include "moe_device.cuh"
#include "moe_internal.h"

namespace moe {
namespace {

constexpr int kThreads = 256;
constexpr int kVec = 8;            // bf16 per 16-byte vector
constexpr int kSlotBatch = 8;      // slots loaded before accumulating

__device__ __forceinline__ uint4 ld_stream(const uint4 *p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ void acc_bf16x2(uint32_t w, float &a, float &b) {
    a += __uint_as_float(w << 16);
    b += __uint_as_float(w & 0xFFFF0000u);
}

__global__ void __launch_bounds__(kThreads)
    combine_kernel(const uint16_t *__restrict__ l2_out, const int32_t *__restrict__ pair_pool, int k,
                   int H, uint16_t *__restrict__ y, const int *err) {
    if (forward_aborted(err)) return;   // an earlier step of this forward timed out
    const int t = blockIdx.x;
    const int h0 = (blockIdx.y * kThreads + threadIdx.x) * kVec;
    if (h0 >= H) return;
    float acc[kVec];
#pragma unroll
    for (int i = 0; i < kVec; ++i) acc[i] = 0.0f;
    const int32_t *pp = pair_pool + (size_t)t * k;
    for (int j0 = 0; j0 < k; j0 += kSlotBatch) {
        int rows[kSlotBatch];
        uint4 v[kSlotBatch];
#pragma unroll
        for (int jj = 0; jj < kSlotBatch; ++jj) rows[jj] = (j0 + jj < k) ? __ldg(pp + j0 + jj) : -1;
#pragma unroll
        for (int jj = 0; jj < kSlotBatch; ++jj)
            if (rows[jj] >= 0)
                v[jj] = ld_stream(reinterpret_cast<const uint4 *>(l2_out + (size_t)rows[jj] * H + h0));
#pragma unroll
        for (int jj = 0; jj < kSlotBatch; ++jj) {
            if (rows[jj] < 0) continue;
            acc_bf16x2(v[jj].x, acc[0], acc[1]);
            acc_bf16x2(v[jj].y, acc[2], acc[3]);
            acc_bf16x2(v[jj].z, acc[4], acc[5]);
            acc_bf16x2(v[jj].w, acc[6], acc[7]);
        }
    }
    uint4 out;
    out.x = bf16x2(acc[0], acc[1]);
    out.y = bf16x2(acc[2], acc[3]);
    out.z = bf16x2(acc[4], acc[5]);
    out.w = bf16x2(acc[6], acc[7]);
    *reinterpret_cast<uint4 *>(y + (size_t)t * H + h0) = out;
}

}  // namespace

void launch_combine(const uint16_t *l2_out, const int32_t *pair_pool, int T, int k, int H,
                    uint16_t *y, const int *err, cudaStream_t s) {
    dim3 grid(T, (H / kVec + kThreads - 1) / kThreads);
    combine_kernel<<<grid, kThreads, 0, s>>>(l2_out, pair_pool, k, H, y, err);
}

}  // namespace moe
