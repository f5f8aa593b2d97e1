// moe_gemm.cu -- the two grouped GEMMs of the expert layer on tcgen05.
//
// L1 (MegaMoE SM90 Implementation Design (Final), §5, §10.1): for every
// expert e and every routed pair r of e,
//     h[r, n] = sum_K x[t(r), K] x_sf[t(r), K/128] * W1[e, n, K] w1_sf[e, n/128, K/128]
// followed in the epilogue by a = silu(clamp(gate)) * clamp(up) * w(r) and the
// per-64-column FP8 requantisation sf = amax/448, q = e4m3(a/sf).
// L2 (design §5.4, §11.1): o[r, h] = sum_i q[r, i] sf[r, i/64] * W2[e, h, i] w2_sf[..]
// rounded to BF16.
//
// Both kernels are persistent (one CTA per SM) and walk a tile list derived
// on the device from the dispatch counts (design §12: experts in order, N-major
// inside experts with many rows).  Warp roles, 10 warps:
//   warp 0      TMA producer (token rows gathered from x with tile::gather4 in
//               L1; plain 2-D tiles elsewhere), multi-stage smem ring;
//   warp 1      TMEM allocation, then MMA issuer: one thread issues
//               tcgen05.mma kind::f8f6f4 into TMEM; every 128-K block (L1) or
//               64-K half (L2) gets its own accumulator so the float block
//               scales can be applied exactly;
//   warps 2-9   epilogue (warp w reads TMEM lanes 32*(w%4)..+31): tcgen05.ld each finished block accumulator, FMA it
//               into FP32 registers with its scale product (the pages'
//               "promotion"), then SwiGLU/quantise (L1) or BF16 (L2) and store.
// TMEM holds two accumulator buffers so the MMA of block k+1 overlaps the
// promotion of block k.
#include "moe_device.cuh"
#include "moe_internal.h"

namespace moe {
namespace {

constexpr int kThreads = 320;      // 10 warps: 200 registers per thread
constexpr int kNumEpiWarps = 8;
constexpr int kEpiWarp0 = 2;       // warps 2..9 run the epilogue
constexpr uint32_t kTmemCols = 512;

constexpr int kL1BN = 256;            // interleaved W1 rows per tile (128 gate/up pairs)
constexpr int kL1Stages = 4;
constexpr uint32_t kL1ABytes = kBM * kBK;
constexpr uint32_t kL1BBytes = kL1BN * kBK;
constexpr uint32_t kL1StageBytes = kL1ABytes + kL1BBytes;

constexpr int kL2BN = 128;            // hidden columns per tile
constexpr int kL2Stages = 6;
constexpr uint32_t kL2ABytes = kBM * kBK;
constexpr uint32_t kL2BBytes = kL2BN * kBK;
constexpr uint32_t kL2StageBytes = kL2ABytes + kL2BBytes;

constexpr int kMaxStages = 8;

struct alignas(8) Ctrl {
    uint64_t full[kMaxStages];
    uint64_t empty[kMaxStages];
    uint64_t tfull[2];
    uint64_t tempty[2];
    uint32_t tmem_base;
    int abort;
};

constexpr size_t kCtrlBytes = 1024;
static_assert(sizeof(Ctrl) <= kCtrlBytes, "ctrl block");

struct Tile {
    int e, row0, rows, nb, nmb;   // nmb: M blocks of expert e
};

// Tile `tile` of a grouped GEMM with NB column blocks: experts in ascending
// order, each expert's M blocks x NB column blocks walked N-major when the
// expert has at least kNMajorMinRows pairs (weight tile reused across
// consecutive CTAs), M-major otherwise (design §12.2 "Auto N-Major").
__device__ __forceinline__ Tile decode_tile(int tile, int NB, const int32_t *__restrict__ offset,
                                            const int32_t *__restrict__ mb_prefix,
                                            const int32_t *__restrict__ mblk_expert) {
    Tile t;
    const int mbi = tile / NB;
    const int e = __ldg(mblk_expert + mbi);
    const int first = __ldg(mb_prefix + e);
    const int nmb = __ldg(mb_prefix + e + 1) - first;
    const int off = __ldg(offset + e);
    const int cnt = __ldg(offset + e + 1) - off;
    const int local = tile - first * NB;
    int mb, nb;
    if (cnt >= kNMajorMinRows) {
        mb = local % nmb;
        nb = local / nmb;
    } else {
        mb = local / NB;
        nb = local % NB;
    }
    t.e = e;
    t.row0 = off + mb * kBM;
    t.rows = min(kBM, cnt - mb * kBM);
    t.nb = nb;
    t.nmb = nmb;
    return t;
}

__device__ __forceinline__ uint32_t align1024(uint32_t a) { return (a + 1023u) & ~1023u; }

// Bounded wait used only on the abort path (does not look at the abort flag).
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity) {
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(bar, parity))
        if (globaltimer_ns() - t0 > kWaitTimeoutNs) return;
}

// Common prologue: barriers, TMEM allocation.  Returns the TMEM base.
__device__ __forceinline__ uint32_t gemm_setup(Ctrl *ctrl, int stages, int warp) {
    if (threadIdx.x == 0) {
        for (int s = 0; s < stages; ++s) {
            mbar_init(smem_u32(&ctrl->full[s]), 1);
            mbar_init(smem_u32(&ctrl->empty[s]), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(smem_u32(&ctrl->tfull[b]), 1);
            mbar_init(smem_u32(&ctrl->tempty[b]), kNumEpiWarps);
        }
        ctrl->abort = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(&ctrl->tmem_base), kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    return ctrl->tmem_base;
}

__device__ __forceinline__ void gemm_teardown(uint32_t tmem, int warp) {
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

// ============================================================================
// L1: gate/up GEMM + SwiGLU * w + per-64 FP8 requantisation
// ============================================================================
// kGatherA: A rows gathered from x by token with tile::gather4 (tm_a = x,
// boxes one row high); otherwise A is the pool of gathered rows written by
// the dispatch step (tm_a = pool, 128-row boxes).
template <bool kFast, bool kGatherA>
__global__ void __launch_bounds__(kThreads, 1)
    l1_kernel(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_w1,
              const L1Params p) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = align1024(raw);
    Ctrl *ctrl = reinterpret_cast<Ctrl *>(smem_raw + (base - raw) + kL1Stages * kL1StageBytes);
    const int warp = threadIdx.x >> 5;
    const uint32_t lane = threadIdx.x & 31;

    const int NB = p.I / 128;   // 256-row blocks of the interleaved 2I rows
    const int KB = p.H / kBK;
    const int total = __ldg(p.mb_prefix + p.E) * NB;

    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tm_a);
        tma_prefetch_desc(&tm_w1);
    }
    const uint32_t tmem = gemm_setup(ctrl, kL1Stages, warp);
    volatile int *abort_flag = &ctrl->abort;

    if (warp == 0) {
        // ---------------- TMA producer ----------------
        // weights of an expert with one M block are read once (evict first);
        // with several M blocks the tile is shared by neighbouring CTAs
        const uint64_t pol_once = policy_evict_first();
        const uint64_t pol_shared = policy_evict_normal();
        const uint64_t pol_x = policy_evict_last();
        int it = 0;
        bool ok = true;
        for (int tile = blockIdx.x; ok && tile < total; tile += gridDim.x) {
            const Tile t = decode_tile(tile, NB, p.offset, p.mb_prefix, p.mblk_expert);
            const uint64_t pol_w = t.nmb > 1 ? pol_shared : pol_once;
            int tok[4] = {0, 0, 0, 0};
            if (kGatherA) {
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int r = (int)lane * 4 + i;
                    tok[i] = r < t.rows ? __ldg(p.gather + t.row0 + r) / p.k : 0;
                }
            }
            const int wrow = t.e * 2 * p.I + t.nb * kL1BN;
            // gather4: only the requests that carry valid rows; the other smem
            // rows keep stale bytes, which reach only masked accumulator rows
            const int n_g4 = (t.rows + 3) >> 2;
            const uint32_t tx = kGatherA ? (uint32_t)n_g4 * 4 * kBK + kL1BBytes : kL1StageBytes;
            for (int kb = 0; kb < KB; ++kb, ++it) {
                const int s = it % kL1Stages;
                const uint32_t ph = (it / kL1Stages) & 1;
                if (!mbar_wait(smem_u32(&ctrl->empty[s]), ph ^ 1, abort_flag, p.err)) {
                    ok = false;
                    break;
                }
                const uint32_t full = smem_u32(&ctrl->full[s]);
                if (lane == 0) mbar_arrive_expect_tx(full, tx);
                __syncwarp();
                if (kGatherA) {
                    if ((int)lane < n_g4)
                        tma_gather4(base + s * kL1StageBytes + lane * 512, &tm_a, kb * kBK, tok[0],
                                    tok[1], tok[2], tok[3], full, pol_x);
                } else if (lane == 0) {
                    tma_load_2d(base + s * kL1StageBytes, &tm_a, kb * kBK, t.row0, full, pol_x);
                }
                if (lane == 0)
                    tma_load_2d(base + s * kL1StageBytes + kL1ABytes, &tm_w1, kb * kBK, wrow, full,
                                pol_w);
            }
        }
        if (!ok) {  // let copies already issued land before the CTA exits
            for (int i = max(0, it - kL1Stages); i < it; ++i)
                drain_wait(smem_u32(&ctrl->full[i % kL1Stages]), (i / kL1Stages) & 1);
        }
    } else if (warp == 1) {
        // ---------------- MMA issuer ----------------
        constexpr uint32_t idesc = idesc_e4m3_f32(kBM, kL1BN);
        int it = 0, kt = 0;
        bool ok = true;
        for (int tile = blockIdx.x; ok && tile < total; tile += gridDim.x) {
            for (int kb = 0; kb < KB; ++kb, ++it, ++kt) {
                const int s = it % kL1Stages;
                const uint32_t ph = (it / kL1Stages) & 1;
                const int b = kt & 1;
                const uint32_t tph = (kt >> 1) & 1;
                if (!mbar_wait(smem_u32(&ctrl->full[s]), ph, abort_flag, p.err) ||
                    !mbar_wait(smem_u32(&ctrl->tempty[b]), tph ^ 1, abort_flag, p.err)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                if (lane == 0) {
                    const uint64_t ad = sw128_kmajor_desc(base + s * kL1StageBytes);
                    const uint64_t bd = sw128_kmajor_desc(base + s * kL1StageBytes + kL1ABytes);
#pragma unroll
                    for (int kk = 0; kk < kBK / 32; ++kk)
                        umma_e4m3(tmem + b * kL1BN, ad + 2 * kk, bd + 2 * kk, idesc, kk > 0);
                    umma_commit(smem_u32(&ctrl->empty[s]));
                    umma_commit(smem_u32(&ctrl->tfull[b]));
                }
                __syncwarp();
            }
        }
        if (!ok && it > 0)
            drain_wait(smem_u32(&ctrl->empty[(it - 1) % kL1Stages]), ((it - 1) / kL1Stages) & 1);
    } else {
        // ---------------- epilogue ----------------
        const int q = warp & 3;                  // TMEM lane quadrant this warp may access
        const int h = (warp - kEpiWarp0) >> 2;   // which 128 of the 256 tile columns
        const int lrow = q * 32 + (int)lane;
        const uint32_t t_lane = tmem + (static_cast<uint32_t>(q * 32) << 16);
        const float clampv = p.clamp;
        int kt = 0;
        bool ok = true;
        for (int tile = blockIdx.x; ok && tile < total; tile += gridDim.x) {
            const Tile t = decode_tile(tile, NB, p.offset, p.mb_prefix, p.mblk_expert);
            const bool valid = lrow < t.rows;
            const bool warp_on = q * 32 < t.rows;
            const int row = t.row0 + lrow;
            const int pair = valid ? __ldg(p.gather + row) : 0;
            const int tok = pair / p.k;
            const float wgt = valid ? __ldg(p.topk_w + pair) : 0.0f;
            const int jb = t.nb * 2 + h;     // interleaved 128-row block = output 64-group
            const float2 *sfb = p.w1_sf + ((size_t)t.e * (2 * p.I / 128) + jb) * KB;
            const float *sfa = p.x_sf + (size_t)tok * KB;

            float acc[128];
#pragma unroll
            for (int i = 0; i < 128; ++i) acc[i] = 0.0f;

            // scale factors prefetched two K blocks ahead (global-load latency
            // would otherwise sit on the critical path of every block)
            float sa1 = valid ? __ldg(sfa) : 0.0f;
            float2 sb1 = __ldg(sfb);
            float sa2 = (valid && KB > 1) ? __ldg(sfa + 1) : 0.0f;
            float2 sb2 = KB > 1 ? __ldg(sfb + 1) : make_float2(0.0f, 0.0f);
            for (int kb = 0; kb < KB; ++kb, ++kt) {
                const int b = kt & 1;
                const uint32_t tph = (kt >> 1) & 1;
                const float sa = sa1;
                const float2 sb = sb1;
                sa1 = sa2;
                sb1 = sb2;
                if (kb + 2 < KB) {
                    sa2 = valid ? __ldg(sfa + kb + 2) : 0.0f;
                    sb2 = __ldg(sfb + kb + 2);
                }
                const float sg = sa * sb.x, su = sa * sb.y;
                if (!mbar_wait(smem_u32(&ctrl->tfull[b]), tph, abort_flag, p.err)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                if (warp_on) {
                    const uint32_t tcol = t_lane + b * kL1BN + h * 128;
#pragma unroll
                    for (int c = 0; c < 4; c += 2) {
                        float v0[32], v1[32];
                        tmem_ld32(tcol + c * 32, v0);
                        tmem_ld32(tcol + c * 32 + 32, v1);
                        tmem_ld_wait();
#pragma unroll
                        for (int i = 0; i < 32; i += 2)
                            ffma2(acc[c * 32 + i], acc[c * 32 + i + 1], v0[i], v0[i + 1],
                                  (i & 8) ? su : sg);
#pragma unroll
                        for (int i = 0; i < 32; i += 2)
                            ffma2(acc[c * 32 + 32 + i], acc[c * 32 + 33 + i], v1[i], v1[i + 1],
                                  (i & 8) ? su : sg);
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&ctrl->tempty[b]));
            }
            if (!ok || !valid) continue;

            // SwiGLU * top-k weight (gate columns 0-7, up columns 8-15 of every 16)
            float amax = 0.0f;
#pragma unroll
            for (int o = 0; o < 64; ++o) {
                const int gi = 16 * (o >> 3) + (o & 7);
                const float g = fminf(fmaxf(acc[gi], -clampv), clampv);
                const float u = fminf(fmaxf(acc[gi + 8], -clampv), clampv);
                float silu;
                if (kFast)
                    silu = __fdividef(g, 1.0f + __expf(-g));
                else
                    silu = g / (1.0f + expf(-g));
                const float a = silu * u * wgt;
                acc[gi] = a;
                amax = fmaxf(amax, fabsf(a));
            }
            // per-64 FP8 requantisation: sf = amax / 448, q = e4m3(a / sf)
            const float sf = amax / 448.0f;
            uint32_t pk[16];
#pragma unroll
            for (int w4 = 0; w4 < 16; ++w4) {
                float qv[4];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int o = w4 * 4 + j;
                    const float a = acc[16 * (o >> 3) + (o & 7)];
                    qv[j] = (sf == 0.0f) ? 0.0f : __fdiv_rn(a, sf);
                }
                pk[w4] = e4m3x2(qv[0], qv[1]) | (e4m3x2(qv[2], qv[3]) << 16);
            }
            uint4 *dst = reinterpret_cast<uint4 *>(p.l2_acts + (size_t)row * p.I + jb * 64);
#pragma unroll
            for (int v = 0; v < 4; ++v)
                dst[v] = make_uint4(pk[4 * v], pk[4 * v + 1], pk[4 * v + 2], pk[4 * v + 3]);
            p.l2_sf[(size_t)jb * p.Pmax + row] = sf;
        }
    }
    gemm_teardown(tmem, warp);
}

// ============================================================================
// L2: down GEMM with per-64 activation scales, BF16 output in pool order
// ============================================================================
__global__ void __launch_bounds__(kThreads, 1)
    l2_kernel(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_w2,
              const L2Params p) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = align1024(raw);
    Ctrl *ctrl = reinterpret_cast<Ctrl *>(smem_raw + (base - raw) + kL2Stages * kL2StageBytes);
    const int warp = threadIdx.x >> 5;
    const uint32_t lane = threadIdx.x & 31;

    const int NB = p.H / kL2BN;
    const int KB = p.I / kBK;
    const int total = __ldg(p.mb_prefix + p.E) * NB;

    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tm_a);
        tma_prefetch_desc(&tm_w2);
    }
    const uint32_t tmem = gemm_setup(ctrl, kL2Stages, warp);
    volatile int *abort_flag = &ctrl->abort;

    if (warp == 0) {
        if (lane == 0) {
            const uint64_t pol_once = policy_evict_first();
            const uint64_t pol_shared = policy_evict_normal();
            const uint64_t pol_a = policy_evict_last();
            int it = 0;
            bool ok = true;
            for (int tile = blockIdx.x; ok && tile < total; tile += gridDim.x) {
                const Tile t = decode_tile(tile, NB, p.offset, p.mb_prefix, p.mblk_expert);
                const uint64_t pol_w = t.nmb > 1 ? pol_shared : pol_once;
                const int wrow = t.e * p.H + t.nb * kL2BN;
                for (int kb = 0; kb < KB; ++kb, ++it) {
                    const int s = it % kL2Stages;
                    const uint32_t ph = (it / kL2Stages) & 1;
                    if (!mbar_wait(smem_u32(&ctrl->empty[s]), ph ^ 1, abort_flag, p.err)) {
                        ok = false;
                        break;
                    }
                    const uint32_t full = smem_u32(&ctrl->full[s]);
                    mbar_arrive_expect_tx(full, kL2StageBytes);
                    tma_load_2d(base + s * kL2StageBytes, &tm_a, kb * kBK, t.row0, full, pol_a);
                    tma_load_2d(base + s * kL2StageBytes + kL2ABytes, &tm_w2, kb * kBK, wrow, full,
                                pol_w);
                }
            }
            if (!ok) {
                for (int i = max(0, it - kL2Stages); i < it; ++i)
                    drain_wait(smem_u32(&ctrl->full[i % kL2Stages]), (i / kL2Stages) & 1);
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        constexpr uint32_t idesc = idesc_e4m3_f32(kBM, kL2BN);
        int it = 0, kt = 0;
        bool ok = true;
        for (int tile = blockIdx.x; ok && tile < total; tile += gridDim.x) {
            for (int kb = 0; kb < KB; ++kb, ++it, ++kt) {
                const int s = it % kL2Stages;
                const uint32_t ph = (it / kL2Stages) & 1;
                const int b = kt & 1;
                const uint32_t tph = (kt >> 1) & 1;
                if (!mbar_wait(smem_u32(&ctrl->full[s]), ph, abort_flag, p.err) ||
                    !mbar_wait(smem_u32(&ctrl->tempty[b]), tph ^ 1, abort_flag, p.err)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                if (lane == 0) {
                    const uint64_t ad = sw128_kmajor_desc(base + s * kL2StageBytes);
                    const uint64_t bd = sw128_kmajor_desc(base + s * kL2StageBytes + kL2ABytes);
                    const uint32_t d0 = tmem + b * 256;         // K half 0: columns [0,128)
                    const uint32_t d1 = tmem + b * 256 + 128;   // K half 1: columns [128,256)
                    umma_e4m3(d0, ad + 0, bd + 0, idesc, 0);
                    umma_e4m3(d0, ad + 2, bd + 2, idesc, 1);
                    umma_e4m3(d1, ad + 4, bd + 4, idesc, 0);
                    umma_e4m3(d1, ad + 6, bd + 6, idesc, 1);
                    umma_commit(smem_u32(&ctrl->empty[s]));
                    umma_commit(smem_u32(&ctrl->tfull[b]));
                }
                __syncwarp();
            }
        }
        if (!ok && it > 0)
            drain_wait(smem_u32(&ctrl->empty[(it - 1) % kL2Stages]), ((it - 1) / kL2Stages) & 1);
    } else {
        const int q = warp & 3;
        const int h = (warp - kEpiWarp0) >> 2;   // which 64 of the 128 tile columns
        const int lrow = q * 32 + (int)lane;
        const uint32_t t_lane = tmem + (static_cast<uint32_t>(q * 32) << 16);
        int kt = 0;
        bool ok = true;
        for (int tile = blockIdx.x; ok && tile < total; tile += gridDim.x) {
            const Tile t = decode_tile(tile, NB, p.offset, p.mb_prefix, p.mblk_expert);
            const bool valid = lrow < t.rows;
            const bool warp_on = q * 32 < t.rows;
            const int row = t.row0 + lrow;
            const float *sfb = p.w2_sf + ((size_t)t.e * NB + t.nb) * KB;

            float acc[64];
#pragma unroll
            for (int i = 0; i < 64; ++i) acc[i] = 0.0f;

            // scales prefetched two K blocks ahead
            const float *sfa = p.l2_sf + row;
            const size_t ps = (size_t)p.Pmax;
            float2 a1 = valid ? make_float2(__ldg(sfa), __ldg(sfa + ps)) : make_float2(0.0f, 0.0f);
            float b1 = __ldg(sfb);
            float2 a2 = (valid && KB > 1) ? make_float2(__ldg(sfa + 2 * ps), __ldg(sfa + 3 * ps))
                                          : make_float2(0.0f, 0.0f);
            float b2 = KB > 1 ? __ldg(sfb + 1) : 0.0f;
            for (int kb = 0; kb < KB; ++kb, ++kt) {
                const int b = kt & 1;
                const uint32_t tph = (kt >> 1) & 1;
                const float2 sa = a1;
                const float sb = b1;
                a1 = a2;
                b1 = b2;
                if (kb + 2 < KB) {
                    if (valid)
                        a2 = make_float2(__ldg(sfa + (size_t)(2 * kb + 4) * ps),
                                         __ldg(sfa + (size_t)(2 * kb + 5) * ps));
                    b2 = __ldg(sfb + kb + 2);
                }
                const float s0 = sa.x * sb, s1 = sa.y * sb;
                if (!mbar_wait(smem_u32(&ctrl->tfull[b]), tph, abort_flag, p.err)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                if (warp_on) {
                    const uint32_t c0 = t_lane + b * 256 + h * 64;
#pragma unroll
                    for (int c = 0; c < 2; ++c) {
                        float v0[32], v1[32];
                        tmem_ld32(c0 + c * 32, v0);
                        tmem_ld32(c0 + 128 + c * 32, v1);
                        tmem_ld_wait();
#pragma unroll
                        for (int i = 0; i < 32; i += 2)
                            ffma2(acc[c * 32 + i], acc[c * 32 + i + 1], v0[i], v0[i + 1], s0);
#pragma unroll
                        for (int i = 0; i < 32; i += 2)
                            ffma2(acc[c * 32 + i], acc[c * 32 + i + 1], v1[i], v1[i + 1], s1);
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&ctrl->tempty[b]));
            }
            if (!ok || !valid) continue;
            uint4 *dst = reinterpret_cast<uint4 *>(p.l2_out + (size_t)row * p.H + t.nb * kL2BN + h * 64);
#pragma unroll
            for (int v = 0; v < 8; ++v)
                dst[v] = make_uint4(bf16x2(acc[8 * v + 0], acc[8 * v + 1]), bf16x2(acc[8 * v + 2], acc[8 * v + 3]),
                                    bf16x2(acc[8 * v + 4], acc[8 * v + 5]), bf16x2(acc[8 * v + 6], acc[8 * v + 7]));
        }
    }
    gemm_teardown(tmem, warp);
}

}  // namespace

size_t l1_smem_bytes() { return 1024 + (size_t)kL1Stages * kL1StageBytes + kCtrlBytes; }
size_t l2_smem_bytes() { return 1024 + (size_t)kL2Stages * kL2StageBytes + kCtrlBytes; }

template <bool kFast, bool kGatherA>
static void launch_l1_t(const CUtensorMap &tm_a, const CUtensorMap &tm_w1, const L1Params &p,
                        int num_sms, cudaStream_t s) {
    static bool configured = false;
    if (!configured) {
        cudaFuncSetAttribute(l1_kernel<kFast, kGatherA>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)l1_smem_bytes());
        configured = true;
    }
    l1_kernel<kFast, kGatherA><<<num_sms, kThreads, l1_smem_bytes(), s>>>(tm_a, tm_w1, p);
}

void launch_l1(const CUtensorMap &tm_a, const CUtensorMap &tm_w1, const L1Params &p, int fast_math,
               bool gather_a, int num_sms, cudaStream_t s) {
    if (fast_math) {
        if (gather_a) launch_l1_t<true, true>(tm_a, tm_w1, p, num_sms, s);
        else launch_l1_t<true, false>(tm_a, tm_w1, p, num_sms, s);
    } else {
        if (gather_a) launch_l1_t<false, true>(tm_a, tm_w1, p, num_sms, s);
        else launch_l1_t<false, false>(tm_a, tm_w1, p, num_sms, s);
    }
}

void launch_l2(const CUtensorMap &tm_a, const CUtensorMap &tm_w2, const L2Params &p, int num_sms,
               cudaStream_t s) {
    static bool configured = false;
    if (!configured) {
        cudaFuncSetAttribute(l2_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)l2_smem_bytes());
        configured = true;
    }
    l2_kernel<<<num_sms, kThreads, l2_smem_bytes(), s>>>(tm_a, tm_w2, p);
}

}  // namespace moe
