// moe_internal.h -- launch interface between the C ABI (moe_api.cu) and the
// kernels (dispatch, grouped GEMMs, combine, weight transform).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

namespace moe {

// A kernel's dynamic shared-memory limit is an attribute of the function on
// each device: set it once per device (one bit per device in `done`, so a
// process that drives several GPUs sets it on each).
inline cudaError_t smem_limit_once(const void *func, size_t bytes, std::atomic<uint32_t> &done) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return cudaErrorInvalidDevice;
    const uint32_t bit = 1u << (dev & 31);
    if (done.load(std::memory_order_acquire) & bit) return cudaSuccess;
    const cudaError_t e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
    if (e == cudaSuccess) done.fetch_or(bit, std::memory_order_acq_rel);
    return e;
}

constexpr int kBM = 128;   // pool rows (routed pairs) per M block
constexpr int kBK = 128;   // K bytes per pipeline stage (one scale block)
constexpr int kNMajorMinRows = 256;  // experts with at least this many pairs walk N-major

// Tensor maps of an A operand (rows of 128 bytes): with tile::gather4 the
// first map covers x [T, H] with one-row boxes; otherwise box[i] covers the
// pool / L2 activations [Pmax, K] with boxes of 32 << i rows, and a tile loads
// the smallest box that covers its valid rows.
struct AMaps {
    CUtensorMap box[3];
};

// Dispatch result: where the pairs of each expert sit in the pool.
struct DispatchOut {
    int32_t *count;        // [E]
    int32_t *offset;       // [E+1]  exclusive prefix of count
    int32_t *mb_prefix;    // [E+2]  first 128-row block of each expert (blocks of experts with
                           //        several blocks first, then one-block experts); [E] all
                           //        blocks, [E+1] those of the several-block experts
    int32_t *mblk_expert;  // [max M blocks]  expert of each M block
    int32_t *mb2_prefix;   // [E+1]  exclusive prefix of ceil(count/256), or null
    int32_t *mblk2_expert; // [max pair blocks]  expert of each 256-row block
    int32_t *gather;       // [T*k]  pool row -> pair id t*k+j (stable order)
    int32_t *pair_pool;    // [T*k]  pair id -> pool row, -1 if inactive
    int32_t *stats;        // [E] or null: += count
    int *err;              // device error word
};

cudaError_t launch_dispatch(const int32_t *topk_idx, int T, int k, int E, const DispatchOut &o,
                            cudaStream_t s);

// The same dispatch over `ctas` CTAs of one cooperative launch (large
// batches): cta_cnt [ctas, E] scratch; bar = words 3-4 of the error block
// (the barrier counter and the forward's abort word, both zeroed here, in
// the stream, before the launch).  Fails without launching when not every
// CTA can be resident.
constexpr int kDispatchMcMinPairs = 8192;   // smaller batches: one CTA (measured faster at 4096)
constexpr int kDispatchMcMaxCtas = 256;
cudaError_t launch_dispatch_mc(const int32_t *topk_idx, int T, int k, int E, const DispatchOut &o,
                               int32_t *cta_cnt, int *bar, int ctas, cudaStream_t s);

// L1: x (gathered by pool row) . W1i^T, SwiGLU * w, per-64 FP8 requant.
struct L1Params {
    const int32_t *gather, *offset, *mb_prefix, *mblk_expert;
    const int32_t *mb2_prefix, *mblk2_expert;   // 256-row blocks (CTA-pair kernel)
    const float *x_sf;        // [T, H/128]
    const float *topk_w;      // [T*k]
    const float2 *w1_sf;      // [E, 2I/128, H/128] (gate scale, up scale) per interleaved block
    uint8_t *l2_acts;         // [Pmax, I], row pitch acts_pitch bytes
    float *l2_sf;             // [Pmax, I/64]
    int *err;
    int H, I, E, k, Pmax, acts_pitch;
    float clamp;
};
// gather_a: tm_a maps x [T, H] with one-row boxes (rows gathered in the
// kernel); otherwise tm_a maps the pool [Pmax, H] with 128-row boxes.
// tm_acts: l2_acts [Pmax, I] with 32-row x 64-byte boxes (64-byte swizzle),
// the TMA stores of the epilogue.
void launch_l1(const AMaps &tm_a, const CUtensorMap &tm_w1, const CUtensorMap &tm_acts, const L1Params &p,
               int fast_math, bool gather_a, int num_sms, cudaStream_t s);

// L1 on CTA pairs (moe_gemm_pair.cu): 256 x 256 tiles, one M=256 MMA over
// both CTAs, stages of two 128-K blocks.  tm_a: the 2-D A maps (gather4 from
// x, or pool boxes); tm_a3 / tm_w1h: the pool / W1i as 3-D [K panel][row][128
// bytes] with 128-row x 2-panel boxes.  Requires H % 256 == 0.
cudaError_t launch_l1_pair(const AMaps &tm_a, const CUtensorMap &tm_a3, const CUtensorMap &tm_w1h,
                           const CUtensorMap &tm_acts, const L1Params &p, int fast_math, bool gather_a, int num_sms,
                           cudaStream_t s);

// Pool of token rows in dispatch order: pool[r] = x[gather[r] / k] for the
// first offset[E] rows (rows_bound = T*k is the host-side upper bound).
void launch_pool_gather(const uint8_t *x, const int32_t *gather, const int32_t *offset_E, int k,
                        int H, int rows_bound, uint8_t *pool, int pool_pitch, const int *err, cudaStream_t s);

// L2: l2_acts . W2^T with per-64 activation scales, BF16 out in pool order.
struct L2Params {
    const int32_t *offset, *mb_prefix, *mblk_expert;
    const float *l2_sf;       // [Pmax, I/64]
    const float *w2_sf;       // [E, H/128, I/128]
    uint16_t *l2_out;         // [Pmax, H] bf16
    int *err;
    int H, I, E, Pmax;
};
// What the one-launch forward needs besides the GEMMs' parameters.
struct FusedParams {
    const int32_t *topk_idx;   // [T, k]
    int T, k;
    DispatchOut d;             // the dispatch tables it writes (mb2 tables unused)
    int32_t *cta_cnt;          // [grid, E] scratch
    int *bar;                  // grid-barrier counter; zero, with the abort word after it, before the launch
    const uint8_t *x;          // token rows, copied into `pool` unless L1 gathers them itself
    uint8_t *pool;
    int pool_pitch;
    uint16_t *y;               // [T, H]
};
// The whole FP8 forward in one cooperative launch: dispatch, pool copy, both
// GEMMs (L2 tiles wait per M block on the L1 tiles' arrival counters in
// `ready`, [M blocks] zeroed beforehand) and the combine, with grid-wide
// barriers between the phases.  Fails without launching when not every CTA
// can be resident (or num_sms > kDispatchMcMaxCtas, E > 1024).
cudaError_t launch_fused(const AMaps &tm_a1, const CUtensorMap &tm_w1, const CUtensorMap &tm_acts, const AMaps &tm_a2,
                         const CUtensorMap &tm_w2, const CUtensorMap &tm_out, const L1Params &p1, const L2Params &p2,
                         int *ready, const FusedParams &f, int fast_math, bool gather_a, int num_sms, cudaStream_t s);

// The two FP8 GEMMs at the same time on disjoint CTA sets of one cooperative
// launch: CTAs [0, n1) run L1, the other num_sms - n1 run L2, each L2 tile
// waiting on its M block's counter in `ready` ([M blocks], zeroed
// beforehand).  Fails without launching when not every CTA can be resident.
cudaError_t launch_split(const AMaps &tm_a1, const CUtensorMap &tm_w1, const CUtensorMap &tm_acts, const AMaps &tm_a2,
                         const CUtensorMap &tm_w2, const CUtensorMap &tm_out, const L1Params &p1, const L2Params &p2,
                         int *ready, int n1, int fast_math, bool gather_a, int num_sms, cudaStream_t s);

// tm_out: l2_out [Pmax, H] BF16 with 32-row x 64-column boxes (128-byte swizzle).
void launch_l2(const AMaps &tm_a, const CUtensorMap &tm_w2, const CUtensorMap &tm_out, const L2Params &p,
               int num_sms, cudaStream_t s);

// FP4-weight configuration: both GEMMs with UE8M0 block scales applied by the
// tensor core (moe_gemm_fp4.cu).
struct Fp4Params {
    const int32_t *gather, *offset, *mb_prefix, *mblk_expert;
    const uint8_t *a_sf;      // L1: x scales u8 [T, H/32]; L2: l2 act scales u8 [Pmax, I/32]
    const uint8_t *b_sf;      // L1: W1 scales u8 [E*2I, H/32] (interleaved rows); L2: u8 [E*H, I/32]
    const float *topk_w;      // [T*k] (L1)
    uint8_t *l2_acts;         // [Pmax, I] (L1 output), row pitch acts_pitch bytes
    uint8_t *l2_sf;           // u8 [Pmax, I/32] (L1 output)
    uint16_t *l2_out;         // bf16 [Pmax, H] (L2 output)
    int *err;
    int H, I, E, k, Pmax, acts_pitch;
    float clamp;
};
void launch_fp4_l1(const AMaps &tm_a, const CUtensorMap &tm_w1, const Fp4Params &p,
                   int fast_math, bool gather_a, int num_sms, cudaStream_t s);
// tm_out: l2_out [Pmax, H] BF16 with 32-row x 64-column boxes (128-byte swizzle).
void launch_fp4_l2(const AMaps &tm_a, const CUtensorMap &tm_w2, const CUtensorMap &tm_out, const Fp4Params &p,
                   int num_sms, cudaStream_t s);

// FP4 weight transform: W1 packed rows and their UE8M0 scale rows interleaved
// like the FP8 rows (row bytes given), W2 copied by the caller.
void launch_interleave_rows(const uint8_t *src, uint8_t *dst, int E, int I, int row_bytes,
                            int dst_pitch, cudaStream_t s);

// Combine: y[t] = bf16( sum_j bf16 l2_out[pair_pool[t*k+j]] ) in slot order.
void launch_combine(const uint16_t *l2_out, const int32_t *pair_pool, int T, int k, int H,
                    uint16_t *y, const int *err, cudaStream_t s);

// Weight transform (W1 gate/up interleave in groups of 8 rows, scale pairs).
void launch_transform_w1(const uint8_t *w1, const float *w1_sf, uint8_t *w1i, int w1i_pitch,
                         float2 *w1i_sf, int E, int H, int I, cudaStream_t s);


}  // namespace moe
