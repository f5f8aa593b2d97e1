// moe_gemm_pair.cu -- the L1 grouped GEMM on CTA pairs (tcgen05 cta_group::2).
//
// Same computation and epilogue as l1_kernel in moe_gemm.cu (MegaMoE SM90
// Implementation Design (Final), §5, §10.1): h = x . W1^T with the per-128
// block scales applied in the epilogue, then SwiGLU * w and the per-64 FP8
// requantisation.  What changes is how a tile is fed.  A cluster of two CTAs
// on neighbouring SMs computes a 256 x 256 tile: each CTA stages its own 128
// pool rows and half of the 256 weight rows, and one M=256 MMA issued by the
// even CTA reads both CTAs' halves.  Every SM then receives 32 KB per 128-K
// block instead of 48 KB for the same tensor work; the copy bandwidth into an
// SM, not the tensor core, is what bounds the one-CTA kernel.  A stage holds
// two 128-K blocks (64 KB per CTA, 3 stages): the copy rate into an SM grows
// with the bytes a stage moves (about 70 B/clk at 64 KB against 40-48 at
// 32 KB), and the weight half arrives as one 3-D box of two K panels.
//
// Each CTA's TMEM holds the accumulators of its own 128 rows over all 256
// columns, so the epilogue is the one-CTA epilogue.  Barriers: the even CTA
// owns `full` (both CTAs' copies complete on it) and `tempty` (all 16
// epilogue warps of the pair release into it); the MMA completion is
// multicast to `empty` and `tfull` of both CTAs.
#include "moe_device.cuh"
#include "moe_gemm_common.cuh"
#include "moe_internal.h"

namespace moe {
namespace {

constexpr int kThreads = 320;
constexpr int kEpiWarp0 = 2;
constexpr int kEpiWarps = 8;
constexpr uint32_t kTmemCols = 512;
constexpr int kBN = 256;             // tile columns (interleaved gate/up rows of W1)
constexpr int kHalfBN = kBN / 2;     // weight rows staged by each CTA
constexpr int kPairRows = 2 * kBM;   // pool rows of a pair tile
constexpr int kTBufs = 2;
constexpr int kStages = 3;
constexpr int kPanels = 2;                          // 128-K blocks per stage
constexpr uint32_t kAPanel = kBM * kBK;             // this CTA's 128 pool rows, one block
constexpr uint32_t kBPanel = kHalfBN * kBK;         // this CTA's 128 weight rows, one block
constexpr uint32_t kABytes = kPanels * kAPanel;
constexpr uint32_t kBBytes = kPanels * kBPanel;
constexpr uint32_t kStageBytes = kABytes + kBBytes;
constexpr uint16_t kPairMask = 3;

struct alignas(8) PairCtrl {
    uint64_t full[kStages];
    uint64_t empty[kStages];
    uint64_t tfull[kTBufs];
    uint64_t tempty[kTBufs];
    uint32_t tmem_base;
    int abort;
};
constexpr size_t kCtrlBytes = 512;
static_assert(sizeof(PairCtrl) <= kCtrlBytes, "ctrl block");
// L1 output staging: per epilogue warp 32 rows x 64 FP8 codes (one TMA store
// box, 64-byte swizzled, 2 KB).
constexpr uint32_t kOutBytes = 32 * 64;
constexpr size_t kSmemBytes = 1024 + (size_t)kStages * kStageBytes + (size_t)kEpiWarps * kOutBytes + kCtrlBytes;

struct PairTile {
    int e, row0, rows, nb, nmb;   // rows: valid rows of the 256-row block
};

// Tile `tile` of the pair schedule: like decode_tile with 256-row blocks.
__device__ __forceinline__ PairTile decode_pair_tile(int tile, int NB, const int32_t *__restrict__ offset,
                                                     const int32_t *__restrict__ mb2_prefix,
                                                     const int32_t *__restrict__ mblk2_expert) {
    PairTile t;
    const int mbi = tile / NB;
    const int e = __ldg(mblk2_expert + mbi);
    const int first = __ldg(mb2_prefix + e);
    const int nmb = __ldg(mb2_prefix + e + 1) - first;
    const int off = __ldg(offset + e);
    const int cnt = __ldg(offset + e + 1) - off;
    const int local = tile - first * NB;
    int mb, nb;
    if (nmb > 1) {   // several blocks share each weight tile: walk N-major
        mb = local % nmb;
        nb = local / nmb;
    } else {
        mb = 0;
        nb = local;
    }
    t.e = e;
    t.row0 = off + mb * kPairRows;
    t.rows = min(kPairRows, cnt - mb * kPairRows);
    t.nb = nb;
    t.nmb = nmb;
    return t;
}

// Release accumulator b to the even CTA's MMA issuer (one arrival per warp).
__device__ __forceinline__ void release_pair(uint32_t tempty_c, uint32_t lane) {
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive_remote(tempty_c);
}

// acc (64 pairs = 128 FP32 columns) += the warp's 128 TMEM columns, gate
// columns (0-7 of every 16) scaled by s_lo, up columns by s_hi; the buffer is
// released once the last piece is in registers.
__device__ __forceinline__ void promote_pair(float2 (&acc)[64], uint32_t tcol, float s_lo, float s_hi,
                                             uint32_t tempty_c, uint32_t lane) {
    const float2 sl = make_float2(s_lo, s_lo), sh = make_float2(s_hi, s_hi);
#pragma unroll
    for (int c = 0; c < 8; ++c) {
        float v[16];
        tmem_ld16(tcol + 16 * c, v);
        tmem_ld_wait();
        if (c == 7) release_pair(tempty_c, lane);
#pragma unroll
        for (int i = 0; i < 4; ++i)
            acc[8 * c + i] = __ffma2_rn(make_float2(v[2 * i], v[2 * i + 1]), sl, acc[8 * c + i]);
#pragma unroll
        for (int i = 4; i < 8; ++i)
            acc[8 * c + i] = __ffma2_rn(make_float2(v[2 * i], v[2 * i + 1]), sh, acc[8 * c + i]);
    }
}

__device__ __forceinline__ float acc_at(const float2 (&acc)[64], int i) {
    return (i & 1) ? acc[i >> 1].y : acc[i >> 1].x;
}

// Bytes one CTA's A copy delivers for `rows` valid rows (0: no copy).
template <bool kGatherA>
__device__ __forceinline__ uint32_t a_copy_bytes(int rows) {
    if (rows <= 0) return 0;
    return kGatherA ? (uint32_t)((rows + 3) >> 2) * 4 * kBK : (32u << a_box_index(rows)) * kBK;
}

// tm_a: 2-D maps (gather4 rows of x, or pool boxes of 32/64/128 rows);
// tm_a3: the pool as [K panel][row][128 B] with 128-row x 2-panel boxes;
// tm_w1h: W1i the same way (128 weight rows x 2 panels).  H % 256 == 0.
template <bool kFast, bool kGatherA>
__global__ void __launch_bounds__(kThreads, 1)
    l1_pair_kernel(const __grid_constant__ AMaps tm_a, const __grid_constant__ CUtensorMap tm_a3,
                   const __grid_constant__ CUtensorMap tm_w1h, const __grid_constant__ CUtensorMap tm_acts,
                   const L1Params p) {
    if (forward_aborted(p.err)) return;   // an earlier step of this forward timed out
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = align1024(raw);
    PairCtrl *ctrl = reinterpret_cast<PairCtrl *>(smem_raw + (base - raw) + kStages * kStageBytes +
                                                  kEpiWarps * kOutBytes);
    const int warp = threadIdx.x >> 5;
    const uint32_t lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();
    const bool leader = rank == 0;
    const int pair = blockIdx.x >> 1, npairs = gridDim.x >> 1;

    const int NB = p.I / 128;   // 256-row blocks of the interleaved 2I rows
    const int KB = p.H / kBK;   // 128-K blocks (even)
    const int KS = KB / kPanels; // stages per tile
    const int total = __ldg(p.mb2_prefix + p.E) * NB;

    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tm_a.box[0]);
        tma_prefetch_desc(&tm_a.box[2]);
        tma_prefetch_desc(&tm_a3);
        tma_prefetch_desc(&tm_w1h);
    }
    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(smem_u32(&ctrl->full[s]), 1);
            mbar_init(smem_u32(&ctrl->empty[s]), 1);
        }
        for (int b = 0; b < kTBufs; ++b) {
            mbar_init(smem_u32(&ctrl->tfull[b]), 1);
            mbar_init(smem_u32(&ctrl->tempty[b]), 2 * kEpiWarps);
        }
        ctrl->abort = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc_pair(smem_u32(&ctrl->tmem_base), kTmemCols);
        tmem_relinquish_pair();
    }
    // both CTAs' barriers initialised and TMEM allocated before any copy or arrival
    tc_fence_before();
    cluster_sync();
    tc_fence_after();
    const uint32_t tmem = ctrl->tmem_base;
    volatile int *abort_flag = &ctrl->abort;
    const uint32_t full_c = mapa_shared(smem_u32(&ctrl->full[0]), 0);     // even CTA's full[0]
    const uint32_t tempty_c = mapa_shared(smem_u32(&ctrl->tempty[0]), 0); // even CTA's tempty[0]

    if (warp == 0) {
        // ---------------- TMA producer (both CTAs) ----------------
        const uint64_t pol_once = policy_evict_first();
        const uint64_t pol_shared = policy_evict_normal();
        const uint64_t pol_x = policy_evict_last();
        int it = 0;
        bool ok = true;
        for (int tile = pair; ok && tile < total; tile += npairs) {
            const PairTile t = decode_pair_tile(tile, NB, p.offset, p.mb2_prefix, p.mblk2_expert);
            const int mine = min(max(t.rows - (int)rank * kBM, 0), kBM);
            const int peer = min(max(t.rows - (1 - (int)rank) * kBM, 0), kBM);
            const int my_row0 = t.row0 + (int)rank * kBM;
            const uint64_t pol_w = t.nmb > 1 ? pol_shared : pol_once;
            int tok[4] = {0, 0, 0, 0};
            if (kGatherA) {
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int r = (int)lane * 4 + i;
                    tok[i] = r < mine ? __ldg(p.gather + my_row0 + r) / p.k : 0;
                }
            }
            const int wrow = t.e * 2 * p.I + t.nb * kBN + (int)rank * kHalfBN;
            const int n_g4 = (mine + 3) >> 2;
            const int abox = a_box_index(max(mine, 1));
            const uint32_t tx =
                kPanels * (a_copy_bytes<kGatherA>(mine) + a_copy_bytes<kGatherA>(peer)) + 2 * kBBytes;
            for (int ks = 0; ks < KS; ++ks, ++it) {
                const int s = it % kStages;
                const uint32_t ph = (it / kStages) & 1;
                if (!mbar_wait(smem_u32(&ctrl->empty[s]), ph ^ 1, abort_flag, p.err)) {
                    ok = false;
                    break;
                }
                const uint32_t full = full_c + 8u * s;
                if (leader && lane == 0) mbar_arrive_expect_tx(smem_u32(&ctrl->full[s]), tx);
                __syncwarp();
                const uint32_t dst = base + s * kStageBytes;
                if (mine > 0) {
                    if (kGatherA) {
                        if ((int)lane < n_g4) {
#pragma unroll
                            for (int j = 0; j < kPanels; ++j)
                                tma_gather4_pair(dst + j * kAPanel + lane * 512, &tm_a.box[0],
                                                 (ks * kPanels + j) * kBK, tok[0], tok[1], tok[2], tok[3], full,
                                                 pol_x);
                        }
                    } else if (lane == 0) {
                        if (abox == 2) {   // full rows: both K panels in one 3-D box
                            tma_load_3d_pair(dst, &tm_a3, 0, my_row0, ks * kPanels, full, pol_x);
                        } else {           // panel j of a 32/64-row box at the panel's 16 KB slot
#pragma unroll
                            for (int j = 0; j < kPanels; ++j)
                                tma_load_2d_pair(dst + j * kAPanel, &tm_a.box[abox], (ks * kPanels + j) * kBK,
                                                 my_row0, full, pol_x);
                        }
                    }
                }
                if (lane == 0) tma_load_3d_pair(dst + kABytes, &tm_w1h, 0, wrow, ks * kPanels, full, pol_w);
            }
        }
        // the copies of the last stages must land before the pair tears down
        for (int i = max(0, it - kStages); i < it; ++i)
            drain_wait(smem_u32(&ctrl->empty[i % kStages]), (i / kStages) & 1, p.err);
    } else if (warp == 1) {
        // ---------------- MMA issuer (even CTA) ----------------
        if (leader) {
            constexpr uint32_t idesc = idesc_e4m3_f32(kPairRows, kBN);
            int it = 0, kt = 0;
            bool ok = true;
            for (int tile = pair; ok && tile < total; tile += npairs) {
                for (int ks = 0; ok && ks < KS; ++ks, ++it) {
                    const int s = it % kStages;
                    const uint32_t ph = (it / kStages) & 1;
                    if (!mbar_wait(smem_u32(&ctrl->full[s]), ph, abort_flag, p.err)) {
                        ok = false;
                        break;
                    }
                    // each 128-K block of the stage into its own accumulator
#pragma unroll
                    for (int j = 0; j < kPanels; ++j, ++kt) {
                        const int b = kt % kTBufs;
                        const uint32_t tph = (kt / kTBufs) & 1;
                        if (!mbar_wait(smem_u32(&ctrl->tempty[b]), tph ^ 1, abort_flag, p.err)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        if (lane == 0) {
                            const uint64_t ad = sw128_kmajor_desc(base + s * kStageBytes + j * kAPanel);
                            const uint64_t bd = sw128_kmajor_desc(base + s * kStageBytes + kABytes + j * kBPanel);
#pragma unroll
                            for (int kk = 0; kk < kBK / 32; ++kk)
                                umma_pair_e4m3(tmem + b * kBN, ad + 2 * kk, bd + 2 * kk, idesc, kk > 0);
                            umma_pair_commit(smem_u32(&ctrl->tfull[b]), kPairMask);
                        }
                        __syncwarp();
                    }
                    if (ok && lane == 0) umma_pair_commit(smem_u32(&ctrl->empty[s]), kPairMask);
                    __syncwarp();
                }
            }
            if (it > 0) drain_wait(smem_u32(&ctrl->empty[(it - 1) % kStages]), ((it - 1) / kStages) & 1, p.err);
        }
    } else {
        // ---------------- epilogue (both CTAs, own 128 rows) ----------------
        const int q = warp & 3;
        const int h = (warp - kEpiWarp0) >> 2;   // which 128 of the 256 tile columns
        const int lrow = (int)rank * kBM + q * 32 + (int)lane;   // row inside the pair block
        const uint32_t t_lane = tmem + (static_cast<uint32_t>(q * 32) << 16) + h * 128;
        const uint32_t out_stage = base + kStages * kStageBytes + (warp - kEpiWarp0) * kOutBytes;
        int kt = 0;
        bool ok = true;
        for (int tile = pair; ok && tile < total; tile += npairs) {
            const PairTile t = decode_pair_tile(tile, NB, p.offset, p.mb2_prefix, p.mblk2_expert);
            const bool valid = lrow < t.rows;
            const bool warp_on = (int)rank * kBM + q * 32 < t.rows;
            const int row = t.row0 + lrow;
            const int pair_id = valid ? __ldg(p.gather + row) : 0;
            // the pair's top-k weight, needed only by the tail: load it now
            const float wgt = valid ? __ldg(p.topk_w + pair_id) : 0.0f;
            const int jb = t.nb * 2 + h;
            const float2 *sfb = p.w1_sf + ((size_t)t.e * (2 * NB) + jb) * KB;
            const float *sfa = p.x_sf + (size_t)(pair_id / p.k) * KB;

            float2 acc[64];
#pragma unroll
            for (int i = 0; i < 64; ++i) acc[i] = make_float2(0.0f, 0.0f);

            float sa_n = valid ? __ldg(sfa) : 0.0f;
            float2 sb_n = __ldg(sfb);
            for (int kb = 0; kb < KB; ++kb, ++kt) {
                const int b = kt % kTBufs;
                const uint32_t tph = (kt / kTBufs) & 1;
                const float sa = sa_n;
                const float2 sb = sb_n;
                if (kb + 1 < KB) {
                    sa_n = valid ? __ldg(sfa + kb + 1) : 0.0f;
                    sb_n = __ldg(sfb + kb + 1);
                }
                if (!mbar_wait(smem_u32(&ctrl->tfull[b]), tph, abort_flag, p.err)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                if (warp_on)
                    promote_pair(acc, t_lane + b * kBN, sa * sb.x, sa * sb.y, tempty_c + 8u * b, lane);
                else
                    release_pair(tempty_c + 8u * b, lane);
            }
            if (!ok || !valid) continue;

            const float clampv = p.clamp;
            float amax = 0.0f;
            float act[64];
#pragma unroll
            for (int o = 0; o < 64; ++o) {
                const int gi = 16 * (o >> 3) + (o & 7);
                const float g = fminf(fmaxf(acc_at(acc, gi), -clampv), clampv);
                const float u = fminf(fmaxf(acc_at(acc, gi + 8), -clampv), clampv);
                float silu;
                if (kFast)
                    silu = __fdividef(g, 1.0f + __expf(-g));
                else
                    silu = __fdividef(g, 1.0f + expf(-g));
                const float a = silu * u * wgt;
                act[o] = a;
                amax = fmaxf(amax, fabsf(a));
            }
            // q = e4m3(a / sf) as a times the correctly rounded 1/sf: within
            // one f32 ulp of the quotient, so an E4M3 code can differ only
            // for a quotient within an ulp of a rounding midpoint
            const float sf = amax / 448.0f;
            const float rsf = (sf == 0.0f) ? 0.0f : __frcp_rn(sf);
            uint32_t pk[16];
#pragma unroll
            for (int w4 = 0; w4 < 16; ++w4) {
                float qv[4];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int o = w4 * 4 + j;
                    qv[j] = (sf == 0.0f) ? 0.0f : act[o] * rsf;
                }
                pk[w4] = e4m3x2(qv[0], qv[1]) | (e4m3x2(qv[2], qv[3]) << 16);
            }
            if ((int)rank * kBM + q * 32 + 32 <= t.rows) {
                // all 32 rows of the warp valid: one 32 x 64 box through
                // shared memory and the copy engine (64-byte swizzle)
                if (lane == 0) tma_store_wait_read();   // the previous box has left the buffer
                __syncwarp();
                const uint32_t rowp = out_stage + lane * 64;
#pragma unroll
                for (int v = 0; v < 4; ++v)
                    st_shared_v4(rowp + ((v ^ ((lane >> 1) & 3)) << 4), pk[4 * v], pk[4 * v + 1], pk[4 * v + 2],
                                 pk[4 * v + 3]);
                fence_async_smem();
                __syncwarp();
                if (lane == 0) {
                    tma_store_2d(&tm_acts, jb * 64, t.row0 + (int)rank * kBM + q * 32, out_stage);
                    tma_store_commit();
                }
            } else {
                uint4 *dst = reinterpret_cast<uint4 *>(p.l2_acts + (size_t)row * p.acts_pitch + jb * 64);
#pragma unroll
                for (int v = 0; v < 4; ++v)
                    dst[v] = make_uint4(pk[4 * v], pk[4 * v + 1], pk[4 * v + 2], pk[4 * v + 3]);
            }
            p.l2_sf[(size_t)row * (p.I / 64) + jb] = sf;
        }
        if (lane == 0) tma_store_wait_all();
        __syncwarp();
    }
    // Neither CTA leaves (or frees TMEM) while the pair MMA may still touch it.
    tc_fence_before();
    cluster_sync();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc_pair(tmem, kTmemCols);
    }
}

}  // namespace

template <bool kFast, bool kGatherA>
static cudaError_t launch_pair_t(const AMaps &tm_a, const CUtensorMap &tm_a3, const CUtensorMap &tm_w1h,
                                 const CUtensorMap &tm_acts, const L1Params &p, int num_sms, cudaStream_t s) {
    static std::atomic<int> grids[32];   // per device: the resident-pair grid, 0 until computed
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSmemBytes;
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return cudaErrorInvalidDevice;
    int grid = grids[dev & 31].load(std::memory_order_acquire);
    if (!grid) {
        static std::atomic<uint32_t> smem_set{0};
        cudaError_t e = smem_limit_once(reinterpret_cast<const void *>(l1_pair_kernel<kFast, kGatherA>), kSmemBytes,
                                        smem_set);
        if (e != cudaSuccess) return e;
        // as many pairs as can be resident at once (a persistent grid)
        cfg.gridDim = dim3(num_sms & ~1);
        int clusters = 0;
        e = cudaOccupancyMaxActiveClusters(&clusters, l1_pair_kernel<kFast, kGatherA>, &cfg);
        if (e != cudaSuccess || clusters < 1) return e != cudaSuccess ? e : cudaErrorLaunchOutOfResources;
        grid = 2 * min(clusters, num_sms / 2);
        grids[dev & 31].store(grid, std::memory_order_release);
    }
    cfg.gridDim = dim3(grid);
    return cudaLaunchKernelEx(&cfg, l1_pair_kernel<kFast, kGatherA>, tm_a, tm_a3, tm_w1h, tm_acts, p);
}

cudaError_t launch_l1_pair(const AMaps &tm_a, const CUtensorMap &tm_a3, const CUtensorMap &tm_w1h,
                           const CUtensorMap &tm_acts, const L1Params &p, int fast_math, bool gather_a, int num_sms,
                           cudaStream_t s) {
    if (fast_math)
        return gather_a ? launch_pair_t<true, true>(tm_a, tm_a3, tm_w1h, tm_acts, p, num_sms, s)
                        : launch_pair_t<true, false>(tm_a, tm_a3, tm_w1h, tm_acts, p, num_sms, s);
    return gather_a ? launch_pair_t<false, true>(tm_a, tm_a3, tm_w1h, tm_acts, p, num_sms, s)
                    : launch_pair_t<false, false>(tm_a, tm_a3, tm_w1h, tm_acts, p, num_sms, s);
}

}  // namespace moe
