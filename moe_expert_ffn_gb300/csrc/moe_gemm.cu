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
// on the device from the dispatch counts (design §12: N-major inside experts
// with many rows; the tiles of one-block experts, whose weights are read once
// from HBM, spread evenly among the others).  Warp roles, 10 warps:
//   warp 0     TMA producer: multi-stage smem ring (A: 128 rows x 128 K bytes,
//              token rows gathered from x with tile::gather4 or one 2-D box of
//              the pool; B: weight rows x 128 K bytes);
//   warp 1     TMEM allocation, then MMA issuer: one thread issues
//              tcgen05.mma kind::f8f6f4 (M=128, K=32) into a ring of FP32
//              accumulators in TMEM.  Every scale block gets its own
//              accumulator (L1: one per 128-K block; L2: one per 64-K half, the
//              pages' "dual-half" scaling) so the float scales can be applied
//              exactly;
//   warps 2-9  epilogue, two per TMEM lane quadrant (warp w reads lanes
//              32*(w%4)..+31: one pool row per thread, half of the tile's
//              columns per warp): tcgen05.ld each finished accumulator,
//              release it, and FMA it into FP32 registers with its scale
//              product (the pages' "promotion"); after the last block,
//              SwiGLU/requantise (L1) or BF16 (L2) and store.  Both outputs
//              go through per-warp shared-memory boxes and TMA stores, so
//              each row leaves as whole 64- or 128-byte pieces instead of 32
//              rows' 16-byte pieces per instruction.  A tile's fields stay in
//              its tile-ring slot until the tail, so the K loop holds only
//              the accumulators, the loaded piece and the scale state;
//   warp 10    (stand-alone L1 kernel) tile loader: for each published tile
//              the rows' dependent loads (pool row -> pair -> top-k weight,
//              token scale row -> first scale) into a shared-memory table, so
//              an epilogue warp starts a tile without global-load latency.
// L1: 128 x 256 tiles (128 gate/up pairs = two 64-column output groups), two
// 256-column accumulators, one per 128-K block.  L2: 128 x 256 tiles, two
// 256-column accumulators, one per 64-K half.  Register budget: 168 per
// thread; each epilogue thread keeps 128 accumulators and loads TMEM in
// 16-column pieces.
//
// Besides one kernel per GEMM, the same warp roles make two single-launch
// variants: fused_kernel, the whole forward (dispatch, pool copy, both GEMMs,
// combine) in one cooperative launch, and split_kernel, both GEMMs at the
// same time on disjoint CTA sets; in both, L2 tiles wait on per-M-block
// arrival counters that the L1 epilogues release.
#include "moe_device.cuh"
#include "moe_gemm_common.cuh"
#include "moe_internal.h"
#include "moe_phases.cuh"

namespace moe {
namespace {

constexpr int kEpiWarp0 = 2;                 // warps 2.. run the epilogue
constexpr int kL1EpiWarps = 8;               // L1: two warps per TMEM lane quadrant
constexpr int kL1Threads = 32 * (kEpiWarp0 + kL1EpiWarps + 1);   // + the tile loader (last warp)
constexpr int kL1LoaderWarp = kEpiWarp0 + kL1EpiWarps;
constexpr int kL2EpiWarps = 8;               // L2: two warps per TMEM lane quadrant
constexpr int kL2Threads = 32 * (kEpiWarp0 + kL2EpiWarps);
constexpr uint32_t kTmemCols = 512;
constexpr int kMaxStages = 6;
constexpr int kMaxTBufs = 4;

// L1: 128 x 256 tiles, two 256-column accumulators, 4 stages of 48 KB
constexpr int kL1BN = 256;
constexpr int kL1TBufs = 2;
constexpr int kL1Stages = 4;
constexpr uint32_t kL1ABytes = kBM * kBK;
constexpr uint32_t kL1BBytes = kL1BN * kBK;
constexpr uint32_t kL1StageBytes = kL1ABytes + kL1BBytes;
// L2: 128 x 256 tiles, a ring of two 256-column accumulators (one per 64-K
// half of a stage), 4 stages of 48 KB.  (The wide tile does twice the tensor
// work per stage hand-off and per token-row copy of a 128 x 128 tile; that
// tile, with a four-deep ring of 128-column accumulators, measured slower.)
constexpr int kL2BN = 256;
constexpr int kL2TBufs = 2;
constexpr int kL2Stages = 4;
constexpr uint32_t kL2ABytes = kBM * kBK;
constexpr uint32_t kL2BBytes = kL2BN * kBK;
constexpr uint32_t kL2StageBytes = kL2ABytes + kL2BBytes;
static_assert(kL1TBufs * kL1BN <= (int)kTmemCols && kL2TBufs * kL2BN <= (int)kTmemCols, "TMEM");

// The producer decodes every tile for its copies; it hands the decoded tile
// to the epilogue through a small ring (a decode is three dependent global
// loads, about 1.3 k cycles at a tile start otherwise).
constexpr int kInfoSlots = 4;

struct alignas(16) Ctrl {
    uint64_t full[kMaxStages];
    uint64_t empty[kMaxStages];
    uint64_t tfull[kMaxTBufs];
    uint64_t tempty[kMaxTBufs];
    uint64_t info_full[kInfoSlots];
    uint64_t info_empty[kInfoSlots];
    int4 info[kInfoSlots];   // e, row0, rows | nb << 8, global M block
    uint32_t tmem_base;
    int abort;
    float stash[kL2EpiWarps][32];   // per epilogue warp: a per-row value the tile's tail needs (L1: top-k weight)
    uint64_t rows_full[kInfoSlots];  // L1 tile loader: the slot's per-row table is written
};

// What the L1 tile loader writes per tile-ring slot: for each of the tile's
// 128 rows its top-k weight, the offset of its token's scale row and that
// row's first scale, and the tile's two first weight-scale pairs.
struct alignas(16) L1Rows {
    float wgt[kBM];
    int sfa[kBM];
    float sa0[kBM];
    float2 sb0[2];
};
constexpr size_t kL1RowsBytes = kInfoSlots * sizeof(L1Rows);

constexpr size_t kCtrlBytes = 1536;
static_assert(sizeof(Ctrl) <= kCtrlBytes, "ctrl block");
// L1 output staging: per epilogue warp 32 rows x 64 FP8 codes (one TMA store
// box, 64-byte swizzled, 2 KB).
constexpr uint32_t kL1OutBytes = 32 * 64;
constexpr size_t kL1SmemBytes =
    1024 + (size_t)kL1Stages * kL1StageBytes + (size_t)kL1EpiWarps * kL1OutBytes + kCtrlBytes + kL1RowsBytes;
// L2 output staging: per epilogue warp 32 rows x 64 BF16 columns (one TMA
// store box, 128-byte swizzled), written twice per tile.
constexpr uint32_t kL2OutBytes = 32 * 128;
constexpr size_t kL2SmemBytes =
    1024 + (size_t)kL2Stages * kL2StageBytes + (size_t)kL2EpiWarps * kL2OutBytes + kCtrlBytes;
static_assert(kL2SmemBytes <= 232448, "L2 shared memory");

// Common prologue: barriers, TMEM allocation.  Returns the TMEM base.
__device__ __forceinline__ uint32_t gemm_setup(Ctrl *ctrl, int warp, int stages, int tbufs,
                                               int epi_warps) {
    if (threadIdx.x == 0) {
        for (int s = 0; s < stages; ++s) {
            mbar_init(smem_u32(&ctrl->full[s]), 1);
            mbar_init(smem_u32(&ctrl->empty[s]), 1);
        }
        for (int b = 0; b < tbufs; ++b) {
            mbar_init(smem_u32(&ctrl->tfull[b]), 1);
            mbar_init(smem_u32(&ctrl->tempty[b]), epi_warps);
        }
        for (int i = 0; i < kInfoSlots; ++i) {
            mbar_init(smem_u32(&ctrl->rows_full[i]), 1);
            mbar_init(smem_u32(&ctrl->info_full[i]), 1);
            mbar_init(smem_u32(&ctrl->info_empty[i]), epi_warps);
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

// Producer side of the tile ring: publish tile number tc (one thread).
__device__ __forceinline__ bool put_tile(Ctrl *ctrl, int tc, const Tile &t, volatile int *abort_flag, int *err) {
    const int i = tc % kInfoSlots;
    if (!mbar_wait(smem_u32(&ctrl->info_empty[i]), ((tc / kInfoSlots) & 1) ^ 1, abort_flag, err)) return false;
    ctrl->info[i] = make_int4(t.e, t.row0, t.rows | (t.nb << 8), t.mbi);
    mbar_arrive(smem_u32(&ctrl->info_full[i]));   // release: the slot's contents come first
    return true;
}

__device__ __forceinline__ Tile tile_at(Ctrl *ctrl, int tc) {
    const volatile int *v = reinterpret_cast<const volatile int *>(&ctrl->info[tc % kInfoSlots]);
    Tile t;
    t.e = v[0];
    t.row0 = v[1];
    t.rows = v[2] & 0xff;
    t.nb = v[2] >> 8;
    t.mbi = v[3];
    t.nmb = 0;
    return t;
}

// Epilogue side, in two steps: wait for tile number tc and read it, keeping
// its slot; the tail reads it again (tile_at) and frees it (free_tile), so
// the tile's fields need no registers during the tile.
__device__ __forceinline__ bool peek_tile(Ctrl *ctrl, int tc, Tile &t, volatile int *abort_flag, int *err) {
    const int i = tc % kInfoSlots;
    if (!mbar_wait(smem_u32(&ctrl->info_full[i]), (tc / kInfoSlots) & 1, abort_flag, err)) return false;
    t = tile_at(ctrl, tc);
    return true;
}
__device__ __forceinline__ void free_tile(Ctrl *ctrl, int tc, uint32_t lane) {
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_u32(&ctrl->info_empty[tc % kInfoSlots]));
}

// Release TMEM buffer b to the MMA warp (one arrival per epilogue warp).
__device__ __forceinline__ void release_tbuf(Ctrl *ctrl, int b, uint32_t lane) {
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_u32(&ctrl->tempty[b]));
}

// After a failed wait: let the producer's issued copies land before exit.
__device__ __forceinline__ void drain_producer(Ctrl *ctrl, int it, int stages, const int *err) {
    for (int i = max(0, it - stages); i < it; ++i)
        drain_wait(smem_u32(&ctrl->full[i % stages]), (i / stages) & 1, err);
}

// Promote this warp's 128 columns (TMEM columns tcol..tcol+127 of the
// thread's lane) into 128 FP32 accumulators, held as 64 pairs (acc[i] =
// columns 2i, 2i+1), in 16-column pieces, and release the buffer as soon as
// the last piece has landed.  Columns 0-7 of every 16 take s_lo, columns 8-15
// s_hi (L1: gate and up scales; L2: one scale).  Packed FP32 FMAs: each half
// is an IEEE fma rounded to nearest, the same result as fmaf.
__device__ __forceinline__ void promote128(float2 (&acc)[64], uint32_t tcol, float s_lo, float s_hi,
                                           Ctrl *ctrl, int b, uint32_t lane) {
    const float2 sl = make_float2(s_lo, s_lo), sh = make_float2(s_hi, s_hi);
#pragma unroll
    for (int c = 0; c < 8; ++c) {
        float v[16];
        tmem_ld16(tcol + 16 * c, v);
        tmem_ld_wait();
        if (c == 7) release_tbuf(ctrl, b, lane);
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

// ============================================================================
// Warp roles.  Each role walks its CTA's tiles of one GEMM; the running
// counters live in a Pipe so that one launch can run the L1 tiles and then
// the L2 tiles through the same stage ring, accumulators and tile ring.
// ============================================================================
struct Pipe {
    int it = 0;      // pipeline stages (producer, MMA issuer)
    int kt = 0;      // accumulator uses (MMA issuer, epilogue)
    int tc = 0;      // tiles (tile ring)
    bool ok = true;
};

struct Role {
    Ctrl *ctrl;
    uint32_t base;   // stage ring
    uint32_t tmem;
    volatile int *abort_flag;
    uint32_t lane;
    int warp;
    int cta, ncta;   // this CTA's tiles of the GEMM: cta, cta + ncta, ...
};

// M-block readiness between the GEMMs of one launch: every L1 epilogue warp
// adds one to its tile's M-block counter (the tile's global M block, not its
// place in the tile list, which N-major experts walk column block first)
// after its stores; an L2 tile waits until the counter of its M block holds
// all of that block's L1 tiles (column blocks x epilogue warps).  Bounded
// like the barrier waits.
__device__ __forceinline__ void signal_ready(int *ready, int mbi, uint32_t lane) {
    fence_acq_rel_gpu();   // this lane's stores before the warp's release
    __syncwarp();
    if (lane == 0) red_release_gpu_add(ready + mbi, 1);
}

__device__ __forceinline__ bool wait_ready(const int *ready, int mbi, int target, volatile int *abort_flag,
                                           int *err) {
    if (ld_acquire_gpu(ready + mbi) >= target) return true;
    const int lim_us = reinterpret_cast<volatile int *>(err)[1];
    const uint64_t limit = lim_us > 0 ? 1000ull * (uint64_t)lim_us : kWaitTimeoutNs;
    const uint64_t t0 = globaltimer_ns();
    while (true) {
        __nanosleep(256);
        if (ld_acquire_gpu(ready + mbi) >= target) return true;
        if (*abort_flag) return false;
        if (globaltimer_ns() - t0 > limit) {
            *abort_flag = 1;
            raise_timeout(err);
            return false;
        }
    }
}

// ---------------------------------------------------------------- L1 roles
// kGatherA: A rows gathered from x by token with tile::gather4 (tm_a = x,
// boxes one row high); otherwise A is the pool of gathered rows written by
// the dispatch step (tm_a = pool, 128-row boxes).
template <bool kGatherA>
__device__ __forceinline__ void l1_produce(const AMaps &tm_a, const CUtensorMap &tm_w1, const L1Params &p,
                                           const Role &r, Pipe &st) {
    const int NB = p.I / 128, KB = p.H / kBK;
    const int total = __ldcg(p.mb_prefix + p.E) * NB;
    const uint32_t lane = r.lane;
    Ctrl *ctrl = r.ctrl;
    // weights of an expert with one M block are read once (evict first);
    // with several M blocks the tile is shared by neighbouring CTAs
    const uint64_t pol_once = policy_evict_first();
    const uint64_t pol_shared = policy_evict_normal();
    const uint64_t pol_x = policy_evict_last();
    const bool stall = test_stall(p.err, kStallL1, r.cta);
    const int it0 = st.it;   // this GEMM's first stage
    // the next tile is decoded during this one (its dependent loads would
    // otherwise hold back the copies at every tile start)
    const int kb_fin = min(1, KB - 1);
    int n_tiles, singles;
    tile_counts(p.mb_prefix, p.E, NB, n_tiles, singles);
    TilePrefetch pf;
    if (r.cta < total) {
        pf.begin(tile_at_position(r.cta, n_tiles, singles), NB, p.mblk_expert);
        pf.finish(p.offset, p.mb_prefix);
    }
    for (int tile = r.cta; st.ok && tile < total; tile += r.ncta, ++st.tc) {
        const Tile t = pf.tile(NB);
        const bool has_next = tile + r.ncta < total;
        if (has_next) pf.begin(tile_at_position(tile + r.ncta, n_tiles, singles), NB, p.mblk_expert);
        bool put_ok = true;
        if (lane == 0) put_ok = put_tile(ctrl, st.tc, t, r.abort_flag, p.err);
        if (!__shfl_sync(0xffffffffu, put_ok, 0)) {
            st.ok = false;
            break;
        }
        const uint64_t pol_w = t.nmb > 1 ? pol_shared : pol_once;
        int tok[4] = {0, 0, 0, 0};
        if (kGatherA) {
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int rr = (int)lane * 4 + i;
                tok[i] = rr < t.rows ? __ldcg(p.gather + t.row0 + rr) / p.k : 0;
            }
        }
        const int wrow = t.e * 2 * p.I + t.nb * kL1BN;
        // gather4: only the requests that carry valid rows; the other smem
        // rows keep stale bytes, which reach only masked accumulator rows
        const int n_g4 = (t.rows + 3) >> 2;
        const int abox = a_box_index(t.rows);
        const uint32_t tx = (kGatherA ? (uint32_t)n_g4 * 4 * kBK : (32u << abox) * kBK) + kL1BBytes;
        for (int kb = 0; kb < KB; ++kb, ++st.it) {
            const int s = st.it % kL1Stages;
            const uint32_t ph = (st.it / kL1Stages) & 1;
            if (!mbar_wait(smem_u32(&ctrl->empty[s]), ph ^ 1, r.abort_flag, p.err)) {
                st.ok = false;
                break;
            }
            if (has_next && kb == kb_fin) pf.finish(p.offset, p.mb_prefix);
            if (stall && st.it == it0) continue;   // timeout-path test: never fill the first stage
            const uint32_t full = smem_u32(&ctrl->full[s]);
            if (lane == 0) mbar_arrive_expect_tx(full, tx);
            __syncwarp();
            if (kGatherA) {
                if ((int)lane < n_g4)
                    tma_gather4(r.base + s * kL1StageBytes + lane * 512, &tm_a.box[0], kb * kBK, tok[0], tok[1],
                                tok[2], tok[3], full, pol_x);
            } else if (lane == 0) {
                tma_load_2d(r.base + s * kL1StageBytes, &tm_a.box[abox], kb * kBK, t.row0, full, pol_x);
            }
            if (lane == 0)
                tma_load_2d(r.base + s * kL1StageBytes + kL1ABytes, &tm_w1, kb * kBK, wrow, full, pol_w);
        }
    }
}

// The L1 tile loader (one warp): for each tile the producer publishes, the
// rows' dependent loads (pool row -> pair -> top-k weight and token scale
// row -> first scale) and the first weight scales, into the slot's L1Rows
// table, so that an epilogue warp starts a tile with shared-memory reads
// instead of three dependent global loads.  It reads the slot after the
// producer publishes it and never frees it (the epilogue does, after the
// tail), so a table is rewritten only after its tile's epilogue is done.
__device__ __forceinline__ void l1_load_rows(const L1Params &p, const Role &r, L1Rows *rows) {
    const int NB = p.I / 128, KB = p.H / kBK;
    const int total = __ldcg(p.mb_prefix + p.E) * NB;
    Ctrl *ctrl = r.ctrl;
    int tc = 0;
    for (int tile = r.cta; tile < total; tile += r.ncta, ++tc) {
        const int i = tc % kInfoSlots;
        if (!mbar_wait(smem_u32(&ctrl->info_full[i]), (tc / kInfoSlots) & 1, r.abort_flag, p.err)) return;
        const Tile t = tile_at(ctrl, tc);
        L1Rows &R = rows[i];
        int pr[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int rr = (int)r.lane + 32 * j;
            pr[j] = rr < t.rows ? __ldcg(p.gather + t.row0 + rr) : 0;
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int rr = (int)r.lane + 32 * j;
            const int off = (pr[j] / p.k) * KB;
            R.wgt[rr] = rr < t.rows ? __ldg(p.topk_w + pr[j]) : 0.0f;
            R.sfa[rr] = off;
            R.sa0[rr] = __ldg(p.x_sf + off);
        }
        if (r.lane < 2) R.sb0[r.lane] = __ldg(p.w1_sf + (t.e * (2 * NB) + t.nb * 2 + (int)r.lane) * KB);
        __syncwarp();
        if (r.lane == 0) mbar_arrive(smem_u32(&ctrl->rows_full[i]));
    }
}

__device__ __forceinline__ void l1_issue(const L1Params &p, const Role &r, Pipe &st) {
    const int NB = p.I / 128, KB = p.H / kBK;
    const int total = __ldcg(p.mb_prefix + p.E) * NB;
    Ctrl *ctrl = r.ctrl;
    constexpr uint32_t idesc = idesc_e4m3_f32(kBM, kL1BN);
    for (int tile = r.cta; st.ok && tile < total; tile += r.ncta) {
        for (int kb = 0; kb < KB; ++kb, ++st.it, ++st.kt) {
            const int s = st.it % kL1Stages;
            const uint32_t ph = (st.it / kL1Stages) & 1;
            const int b = st.kt % kL1TBufs;
            const uint32_t tph = (st.kt / kL1TBufs) & 1;
            if (!mbar_wait(smem_u32(&ctrl->full[s]), ph, r.abort_flag, p.err) ||
                !mbar_wait(smem_u32(&ctrl->tempty[b]), tph ^ 1, r.abort_flag, p.err)) {
                st.ok = false;
                break;
            }
            tc_fence_after();
            if (r.lane == 0) {
                const uint64_t ad = sw128_kmajor_desc(r.base + s * kL1StageBytes);
                const uint64_t bd = sw128_kmajor_desc(r.base + s * kL1StageBytes + kL1ABytes);
#pragma unroll
                for (int kk = 0; kk < kBK / 32; ++kk)
                    umma_e4m3(r.tmem + b * kL1BN, ad + 2 * kk, bd + 2 * kk, idesc, kk > 0);
                umma_commit(smem_u32(&ctrl->empty[s]));
                umma_commit(smem_u32(&ctrl->tfull[b]));
            }
            __syncwarp();
        }
    }
}

// kSignal: add this warp's finished tiles to the M-block counters in `ready`.
// out_stage: this warp's 2 KB shared-memory box for the TMA store of its
// 32 rows x 64 codes (tm_acts: l2_acts with 32-row x 64-byte boxes).
template <bool kFast, bool kSignal, bool kRows = false>
__device__ __forceinline__ void l1_epilogue(const CUtensorMap &tm_acts, const L1Params &p, const Role &r, Pipe &st,
                                            uint32_t out_stage, int *ready, const L1Rows *rows = nullptr) {
    const int NB = p.I / 128, KB = p.H / kBK;
    const int total = __ldcg(p.mb_prefix + p.E) * NB;
    const uint32_t lane = r.lane;
    Ctrl *ctrl = r.ctrl;
    const int q = r.warp & 3;                  // TMEM lane quadrant this warp may access
    const int h = (r.warp - kEpiWarp0) >> 2;   // which 128 of the 256 tile columns
    const int lrow = q * 32 + (int)lane;
    const uint32_t t_lane = r.tmem + (static_cast<uint32_t>(q * 32) << 16) + h * 128;
    float *wstash = ctrl->stash[r.warp - kEpiWarp0];
    for (int tile = r.cta; st.ok && tile < total; tile += r.ncta, ++st.tc) {
        // Tile state for the K loop only: offsets of the two scale rows and
        // whether the warp holds any row.  What the tail needs is read again
        // from the tile ring (its slot is held until then) and, for the top-k
        // weight, from shared memory, so none of it occupies registers
        // during the promotion.
        bool warp_on;
        int sfa_off, sfb_off;
        float sa_n;
        float2 sb_n;
        {
            Tile t;
            if (!peek_tile(ctrl, st.tc, t, r.abort_flag, p.err)) {
                st.ok = false;
                break;
            }
            warp_on = q * 32 < t.rows;
            sfb_off = (t.e * (2 * NB) + t.nb * 2 + h) * KB;   // interleaved 128-row block = output 64-group
            if (kRows) {
                const int i = st.tc % kInfoSlots;
                if (!mbar_wait(smem_u32(&ctrl->rows_full[i]), (st.tc / kInfoSlots) & 1, r.abort_flag, p.err)) {
                    st.ok = false;
                    break;
                }
                sfa_off = rows[i].sfa[lrow];
                sa_n = rows[i].sa0[lrow];
                sb_n = rows[i].sb0[h];
            } else {
                const bool valid = lrow < t.rows;
                const int pair = valid ? __ldcg(p.gather + t.row0 + lrow) : 0;
                wstash[lane] = valid ? __ldg(p.topk_w + pair) : 0.0f;
                sfa_off = (pair / p.k) * KB;
                // (an invalid row reads token 0's scales: in bounds, and its
                // outputs are not stored)
                sa_n = __ldg(p.x_sf + sfa_off);
                sb_n = __ldg(p.w1_sf + sfb_off);
            }
        }

        float2 acc[64];
#pragma unroll
        for (int i = 0; i < 64; ++i) acc[i] = make_float2(0.0f, 0.0f);

        // scale factors prefetched one K block ahead
        for (int kb = 0; kb < KB; ++kb, ++st.kt) {
            const int b = st.kt % kL1TBufs;
            const uint32_t tph = (st.kt / kL1TBufs) & 1;
            const float s_lo = sa_n * sb_n.x, s_hi = sa_n * sb_n.y;
            if (kb + 1 < KB) {
                sa_n = __ldg(p.x_sf + sfa_off + kb + 1);
                sb_n = __ldg(p.w1_sf + sfb_off + kb + 1);
            }
            if (!mbar_wait(smem_u32(&ctrl->tfull[b]), tph, r.abort_flag, p.err)) {
                st.ok = false;
                break;
            }
            tc_fence_after();
            if (warp_on)
                promote128(acc, t_lane + b * kL1BN, s_lo, s_hi, ctrl, b, lane);
            else
                release_tbuf(ctrl, b, lane);
        }
        if (!st.ok) break;
        const Tile t = tile_at(ctrl, st.tc);
        const int row = t.row0 + lrow;
        const int jb = t.nb * 2 + h;
        const bool valid = lrow < t.rows;
        if (valid) {
            // SwiGLU * top-k weight (gate columns 0-7, up columns 8-15 of every 16)
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
                const float a = silu * u * (kRows ? rows[st.tc % kInfoSlots].wgt[lrow] : wstash[lane]);
                act[o] = a;
                amax = fmaxf(amax, fabsf(a));
            }
            // per-64 FP8 requantisation: sf = amax / 448, q = e4m3(a / sf)
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
            // this warp's 64 outputs are intermediate columns [64 jb, 64 jb + 64)
            if (q * 32 + 32 <= t.rows) {
                // all 32 rows of the warp valid: one 32 x 64 box through shared
                // memory and the copy engine, so each row leaves as one 64-byte
                // piece instead of 32 rows' 16-byte pieces per instruction
                // (64-byte swizzle: chunk v of row `lane` at chunk v ^ (lane/2 % 4))
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
                    tma_store_2d(&tm_acts, jb * 64, t.row0 + q * 32, out_stage);
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
        free_tile(ctrl, st.tc, lane);
        if (kSignal) {
            // the box's writes complete and ordered before the M block's release
            if (lane == 0) tma_store_wait_all();
            __syncwarp();
            fence_proxy_async_global();
            signal_ready(ready, t.mbi, lane);
        }
    }
    if (lane == 0) tma_store_wait_all();
    __syncwarp();
}

// ---------------------------------------------------------------- L2 roles
// ready (nullable): wait until the tile's M block counter reaches `target`
// before copying its activation rows.
__device__ __forceinline__ void l2_produce(const AMaps &tm_a, const CUtensorMap &tm_w2, const L2Params &p,
                                           const Role &r, Pipe &st, const int *ready, int target) {
    const int NB = (p.H + kL2BN - 1) / kL2BN;   // the last block may be half empty (H % 256 == 128)
    const int KB = p.I / kBK;
    const int total = __ldcg(p.mb_prefix + p.E) * NB;
    Ctrl *ctrl = r.ctrl;
    const uint64_t pol_once = policy_evict_first();
    const uint64_t pol_shared = policy_evict_normal();
    const uint64_t pol_a = policy_evict_last();
    const bool stall = test_stall(p.err, kStallL2, r.cta);
    const int it0 = st.it;   // this GEMM's first stage
    int last_mbi = -1;
    // the next tile is decoded during this one, as in the L1 producer
    const int kb_fin = min(1, KB - 1);
    int n_tiles, singles;
    tile_counts(p.mb_prefix, p.E, NB, n_tiles, singles);
    TilePrefetch pf;
    if (r.cta < total) {
        pf.begin(tile_at_position(r.cta, n_tiles, singles), NB, p.mblk_expert);
        pf.finish(p.offset, p.mb_prefix);
    }
    for (int tile = r.cta; st.ok && tile < total; tile += r.ncta, ++st.tc) {
        const Tile t = pf.tile(NB);
        const bool has_next = tile + r.ncta < total;
        if (has_next) pf.begin(tile_at_position(tile + r.ncta, n_tiles, singles), NB, p.mblk_expert);
        if (!put_tile(ctrl, st.tc, t, r.abort_flag, p.err)) {
            st.ok = false;
            break;
        }
        if (ready && t.mbi != last_mbi) {
            last_mbi = t.mbi;
            if (!wait_ready(ready, last_mbi, target, r.abort_flag, p.err)) {
                st.ok = false;
                break;
            }
            fence_proxy_async_global();   // the rows the acquire made visible, for the copy engine
        }
        const uint64_t pol_w = t.nmb > 1 ? pol_shared : pol_once;
        const int wrow = t.e * p.H + t.nb * kL2BN;
        for (int kb = 0; kb < KB; ++kb, ++st.it) {
            const int s = st.it % kL2Stages;
            const uint32_t ph = (st.it / kL2Stages) & 1;
            if (!mbar_wait(smem_u32(&ctrl->empty[s]), ph ^ 1, r.abort_flag, p.err)) {
                st.ok = false;
                break;
            }
            if (has_next && kb == kb_fin) pf.finish(p.offset, p.mb_prefix);
            if (stall && st.it == it0) continue;   // timeout-path test: never fill the first stage
            const uint32_t full = smem_u32(&ctrl->full[s]);
            const int abox = a_box_index(t.rows);
            mbar_arrive_expect_tx(full, (32u << abox) * kBK + kL2BBytes);
            tma_load_2d(r.base + s * kL2StageBytes, &tm_a.box[abox], kb * kBK, t.row0, full, pol_a);
            tma_load_2d(r.base + s * kL2StageBytes + kL2ABytes, &tm_w2, kb * kBK, wrow, full, pol_w);
        }
    }
}

// Each 128-K stage is two 64-K halves, each into its own accumulator.
// kOneCommit: the second half's MMAs are the stage's last, so the stage's
// empty commit also tells the epilogue that half is done, and the half needs
// no commit of its own (one commit fewer per stage on the issuing thread).
// The one-launch GEMM pair keeps both, because its epilogue counts uses
// across both GEMMs.
template <bool kOneCommit>
__device__ __forceinline__ void l2_issue(const L2Params &p, const Role &r, Pipe &st) {
    const int NB = (p.H + kL2BN - 1) / kL2BN;
    const int KB = p.I / kBK;
    const int total = __ldcg(p.mb_prefix + p.E) * NB;
    Ctrl *ctrl = r.ctrl;
    constexpr uint32_t idesc = idesc_e4m3_f32(kBM, kL2BN);
    for (int tile = r.cta; st.ok && tile < total; tile += r.ncta) {
        for (int kb = 0; st.ok && kb < KB; ++kb, ++st.it) {
            const int s = st.it % kL2Stages;
            const uint32_t ph = (st.it / kL2Stages) & 1;
            if (!mbar_wait(smem_u32(&ctrl->full[s]), ph, r.abort_flag, p.err)) {
                st.ok = false;
                break;
            }
            const uint64_t ad = sw128_kmajor_desc(r.base + s * kL2StageBytes);
            const uint64_t bd = sw128_kmajor_desc(r.base + s * kL2StageBytes + kL2ABytes);
#pragma unroll
            for (int half = 0; half < 2; ++half, ++st.kt) {
                const int b = st.kt % kL2TBufs;
                const uint32_t tph = (st.kt / kL2TBufs) & 1;
                if (!mbar_wait(smem_u32(&ctrl->tempty[b]), tph ^ 1, r.abort_flag, p.err)) {
                    st.ok = false;
                    break;
                }
                tc_fence_after();
                if (r.lane == 0) {
                    umma_e4m3(r.tmem + b * kL2BN, ad + 4 * half, bd + 4 * half, idesc, 0);
                    umma_e4m3(r.tmem + b * kL2BN, ad + 4 * half + 2, bd + 4 * half + 2, idesc, 1);
                    if (!(kOneCommit && half == 1)) umma_commit(smem_u32(&ctrl->tfull[b]));
                }
                __syncwarp();
            }
            if (st.ok && r.lane == 0) umma_commit(smem_u32(&ctrl->empty[s]));
            __syncwarp();
        }
    }
}

// kAcquire: the L1 outputs of this launch are read after the tile's M block
// is ready (an acquire by lane 0, then L2-coherent loads of the scales).
template <bool kAcquire>
__device__ __forceinline__ float2 load_sa(const float2 *p) {
    if (kAcquire) return ld_cg_f32x2(p);
    return __ldg(p);
}

template <bool kAcquire, bool kOneCommit>
__device__ __forceinline__ void l2_epilogue(const CUtensorMap &tm_out, const L2Params &p, const Role &r, Pipe &st,
                                            uint32_t out_stage, const int *ready, int target) {
    const int NB = (p.H + kL2BN - 1) / kL2BN;
    const int KB = p.I / kBK;
    const int total = __ldcg(p.mb_prefix + p.E) * NB;
    const uint32_t lane = r.lane;
    Ctrl *ctrl = r.ctrl;
    const int q = r.warp & 3;
    const int h = (r.warp - kEpiWarp0) >> 2;   // which 128 of the 256 tile columns
    const int lrow = q * 32 + (int)lane;
    const uint32_t t_lane = r.tmem + (static_cast<uint32_t>(q * 32) << 16) + h * 128;
    const int HB = p.H / 128;                  // 128-row weight scale blocks
    for (int tile = r.cta; st.ok && tile < total; tile += r.ncta, ++st.tc) {
        // K-loop state only (the tail reads the tile again from its slot)
        bool warp_on;
        int sfa_off, sfb_off;
        {
            Tile t;
            if (!peek_tile(ctrl, st.tc, t, r.abort_flag, p.err)) {
                st.ok = false;
                break;
            }
            if (kAcquire) {
                bool rd = true;
                if (lane == 0) rd = wait_ready(ready, t.mbi, target, r.abort_flag, p.err);
                if (!__shfl_sync(0xffffffffu, rd, 0)) {
                    st.ok = false;
                    break;
                }
                __syncwarp();   // lane 0's acquire before every lane's loads
            }
            const int cb = t.nb * 2 + h;           // this warp's 128-column block of H
            warp_on = q * 32 < t.rows && cb < HB;
            sfb_off = (t.e * HB + min(cb, HB - 1)) * KB;
            // the row's two 64-K activation scales of 128-K block kb (a row
            // past the tile's end reads the tile's last row: in bounds, and
            // its outputs are not stored)
            sfa_off = (t.row0 + min(lrow, t.rows - 1)) * (p.I / 128);
        }
        const float2 *sfa = reinterpret_cast<const float2 *>(p.l2_sf) + sfa_off;
        const float *sfb = p.w2_sf + sfb_off;

        float2 acc[64];
#pragma unroll
        for (int i = 0; i < 64; ++i) acc[i] = make_float2(0.0f, 0.0f);

        // scales prefetched two 128-K blocks ahead (a far L2 hit takes
        // longer than one block's promotion)
        const float2 z2 = make_float2(0.0f, 0.0f);
        float2 sa0 = load_sa<kAcquire>(sfa);
        float2 sa1 = KB > 1 ? load_sa<kAcquire>(sfa + 1) : z2;
        float sb0 = __ldg(sfb);
        float sb1 = KB > 1 ? __ldg(sfb + 1) : 0.0f;
        for (int kb = 0; st.ok && kb < KB; ++kb) {
            const float2 sa = sa0;
            const float sb = sb0;
            sa0 = sa1;
            sb0 = sb1;
            if (kb + 2 < KB) {
                sa1 = load_sa<kAcquire>(sfa + kb + 2);
                sb1 = __ldg(sfb + kb + 2);
            }
#pragma unroll
            for (int half = 0; half < 2; ++half, ++st.kt) {
                const float sc = (half ? sa.y : sa.x) * sb;
                const int b = st.kt % kL2TBufs;
                // kOneCommit: the second half waits for its stage's empty
                // barrier (use kt of a launch that starts at use 0 is half
                // kt % 2 of stage kt / 2)
                const int js = st.kt >> 1;
                const bool got = (kOneCommit && half == 1)
                                     ? mbar_wait(smem_u32(&ctrl->empty[js % kL2Stages]), (js / kL2Stages) & 1,
                                                 r.abort_flag, p.err)
                                     : mbar_wait(smem_u32(&ctrl->tfull[b]), (st.kt / kL2TBufs) & 1, r.abort_flag,
                                                 p.err);
                if (!got) {
                    st.ok = false;
                    break;
                }
                tc_fence_after();
                if (warp_on)
                    promote128(acc, t_lane + b * kL2BN, sc, sc, ctrl, b, lane);
                else
                    release_tbuf(ctrl, b, lane);
            }
        }
        if (!st.ok) break;
        const Tile t = tile_at(ctrl, st.tc);
        free_tile(ctrl, st.tc, lane);
        if (!warp_on) continue;
        const int cb = t.nb * 2 + h;
        const bool valid = lrow < t.rows;
        if (q * 32 + 32 <= t.rows) {
            // all 32 rows of the warp valid: two 32 x 64 boxes through shared
            // memory and the copy engine (whole 128-byte row pieces)
#pragma unroll
            for (int k = 0; k < 2; ++k) {
                if (lane == 0) tma_store_wait_read();   // the previous box has left the buffer
                __syncwarp();
                const uint32_t rowp = out_stage + lane * 128;
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    const int i = 32 * k + 4 * c;
                    st_shared_v4(rowp + ((c ^ (lane & 7)) << 4), bf16x2(acc[i].x, acc[i].y),
                                 bf16x2(acc[i + 1].x, acc[i + 1].y), bf16x2(acc[i + 2].x, acc[i + 2].y),
                                 bf16x2(acc[i + 3].x, acc[i + 3].y));
                }
                fence_async_smem();
                __syncwarp();
                if (lane == 0) {
                    tma_store_2d(&tm_out, cb * 128 + 64 * k, t.row0 + q * 32, out_stage);
                    tma_store_commit();
                }
            }
        } else if (valid) {
            uint4 *dst = reinterpret_cast<uint4 *>(p.l2_out + (size_t)(t.row0 + lrow) * p.H + cb * 128);
#pragma unroll
            for (int v = 0; v < 16; ++v)
                dst[v] = make_uint4(bf16x2(acc[4 * v].x, acc[4 * v].y), bf16x2(acc[4 * v + 1].x, acc[4 * v + 1].y),
                                    bf16x2(acc[4 * v + 2].x, acc[4 * v + 2].y),
                                    bf16x2(acc[4 * v + 3].x, acc[4 * v + 3].y));
        }
    }
    if (lane == 0) tma_store_wait_all();
    __syncwarp();
}

// ============================================================================
// Kernels
// ============================================================================
// L1: gate/up GEMM + SwiGLU * w + per-64 FP8 requantisation.
template <bool kFast, bool kGatherA>
__global__ void __launch_bounds__(kL1Threads, 1)
    l1_kernel(const __grid_constant__ AMaps tm_a, const __grid_constant__ CUtensorMap tm_w1,
              const __grid_constant__ CUtensorMap tm_acts, const L1Params p) {
    if (forward_aborted(p.err)) return;   // an earlier step of this forward timed out
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = align1024(raw);
    Ctrl *ctrl = reinterpret_cast<Ctrl *>(smem_raw + (base - raw) + kL1Stages * kL1StageBytes +
                                          kL1EpiWarps * kL1OutBytes);
    L1Rows *rows = reinterpret_cast<L1Rows *>(reinterpret_cast<uint8_t *>(ctrl) + kCtrlBytes);
    const int warp = threadIdx.x >> 5;
    const uint32_t lane = threadIdx.x & 31;
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tm_a.box[0]);
        tma_prefetch_desc(&tm_a.box[2]);
        tma_prefetch_desc(&tm_w1);
    }
    const uint32_t tmem = gemm_setup(ctrl, warp, kL1Stages, kL1TBufs, kL1EpiWarps);
    const Role r{ctrl, base, tmem, &ctrl->abort, lane, warp, (int)blockIdx.x, (int)gridDim.x};
    Pipe st;
    if (warp == 0) {
        l1_produce<kGatherA>(tm_a, tm_w1, p, r, st);
        if (!st.ok) drain_producer(ctrl, st.it, kL1Stages, p.err);
    } else if (warp == 1) {
        l1_issue(p, r, st);
        if (!st.ok && st.kt > 0)
            drain_wait(smem_u32(&ctrl->tfull[(st.kt - 1) % kL1TBufs]), ((st.kt - 1) / kL1TBufs) & 1, p.err);
    } else if (warp == kL1LoaderWarp) {
        l1_load_rows(p, r, rows);
    } else {
        l1_epilogue<kFast, false, true>(tm_acts, p, r, st,
                                        base + kL1Stages * kL1StageBytes + (warp - kEpiWarp0) * kL1OutBytes, nullptr,
                                        rows);
    }
    gemm_teardown(tmem, warp);
}

// L2: down GEMM with per-64 activation scales, BF16 output in pool order.
__global__ void __launch_bounds__(kL2Threads, 1)
    l2_kernel(const __grid_constant__ AMaps tm_a, const __grid_constant__ CUtensorMap tm_w2,
              const __grid_constant__ CUtensorMap tm_out, const L2Params p) {
    if (forward_aborted(p.err)) return;   // an earlier step of this forward timed out
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = align1024(raw);
    Ctrl *ctrl = reinterpret_cast<Ctrl *>(smem_raw + (base - raw) + kL2Stages * kL2StageBytes +
                                          kL2EpiWarps * kL2OutBytes);
    const int warp = threadIdx.x >> 5;
    const uint32_t lane = threadIdx.x & 31;
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tm_a.box[0]);
        tma_prefetch_desc(&tm_a.box[2]);
        tma_prefetch_desc(&tm_w2);
    }
    const uint32_t tmem = gemm_setup(ctrl, warp, kL2Stages, kL2TBufs, kL2EpiWarps);
    const Role r{ctrl, base, tmem, &ctrl->abort, lane, warp, (int)blockIdx.x, (int)gridDim.x};
    Pipe st;
    if (warp == 0) {
        if (lane == 0) {
            l2_produce(tm_a, tm_w2, p, r, st, nullptr, 0);
            if (!st.ok) drain_producer(ctrl, st.it, kL2Stages, p.err);
        }
        __syncwarp();
    } else if (warp == 1) {
        l2_issue<true>(p, r, st);
        if (!st.ok && st.kt > 0) {   // the last committed use: a first half (tfull) or a stage (empty)
            const int u = st.kt - 1;
            if (u & 1)
                drain_wait(smem_u32(&ctrl->empty[(u >> 1) % kL2Stages]), ((u >> 1) / kL2Stages) & 1, p.err);
            else
                drain_wait(smem_u32(&ctrl->tfull[u % kL2TBufs]), (u / kL2TBufs) & 1, p.err);
        }
    } else {
        l2_epilogue<false, true>(tm_out, p, r, st, base + kL2Stages * kL2StageBytes + (warp - kEpiWarp0) * kL2OutBytes,
                           nullptr, 0);
    }
    gemm_teardown(tmem, warp);
}

// The whole forward in one persistent launch (every CTA resident: a
// cooperative launch), the pages' fused pipeline (MegaMoE SM90 Implementation
// Design (Final), §3.3): Phase 1 the dispatch over all CTAs with grid-wide
// barriers, then the pool copy of the token rows; Phases 2 and 3 each CTA's
// L1 tiles and then its L2 tiles through the same stage ring, accumulators
// and tile ring, an L2 tile starting once the L1 tiles of its M block (on
// any CTA) have stored their outputs, so L2 work fills the SMs that finish
// L1 early; Phase 4, after a last barrier, the combine.  On one GPU the
// pages' NVLink pull, scatter and barriers are the local pool copy, the
// pool-order outputs and these grid barriers.  The dispatch's scratch lives
// in the stage ring, which the pipeline only uses after it.
template <bool kFast, bool kGatherA>
__global__ void __launch_bounds__(kL2Threads, 1)
    fused_kernel(const __grid_constant__ AMaps tm_a1, const __grid_constant__ CUtensorMap tm_w1,
                 const __grid_constant__ CUtensorMap tm_acts, const __grid_constant__ AMaps tm_a2,
                 const __grid_constant__ CUtensorMap tm_w2, const __grid_constant__ CUtensorMap tm_out,
                 const L1Params p1, const L2Params p2, int *ready, const FusedParams f) {
    if (forward_aborted(p1.err)) return;   // an earlier step of this forward timed out
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = align1024(raw);
    Ctrl *ctrl = reinterpret_cast<Ctrl *>(smem_raw + (base - raw) + kL2Stages * kL2StageBytes +
                                          kL2EpiWarps * kL2OutBytes);
    const int warp = threadIdx.x >> 5;
    const uint32_t lane = threadIdx.x & 31;
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tm_a1.box[0]);
        tma_prefetch_desc(&tm_w1);
        tma_prefetch_desc(&tm_a2.box[2]);
        tma_prefetch_desc(&tm_w2);
    }
    // ---- Phase 1: dispatch, then the pool of token rows
    int bar_target = 0;
    {
        const bool stall = blockIdx.x == 0 && reinterpret_cast<const volatile int *>(p1.err)[2] == kStallDispatch;
        bool ok = dispatch_phase(f.topk_idx, f.T, f.k, p1.E, f.d, f.cta_cnt, f.bar, bar_target,
                                 reinterpret_cast<int32_t *>(smem_raw + (base - raw)), stall);
        if (ok && !kGatherA) {
            pool_phase(f.x, f.d.gather, f.d.offset + p1.E, f.k, p1.H, f.T * f.k, f.pool, f.pool_pitch);
            bar_target += (int)gridDim.x;
            ok = grid_sync(f.bar, bar_target, p1.err);
        }
        if (!ok) return;   // a barrier ran out; no TMEM held yet
        // the generic writes of the dispatch scratch (shared) and of the pool
        // (global) before the copy engine touches either
        fence_async_smem();
        fence_proxy_async_global();
    }
    // ---- Phases 2 and 3: the two GEMMs
    const uint32_t tmem = gemm_setup(ctrl, warp, kL2Stages, kL2TBufs, kL2EpiWarps);
    const Role r{ctrl, base, tmem, &ctrl->abort, lane, warp, (int)blockIdx.x, (int)gridDim.x};
    const int target = (p1.I / 128) * kL1EpiWarps;   // L1 tile-warps per M block
    Pipe st;
    if (warp == 0) {
        l1_produce<kGatherA>(tm_a1, tm_w1, p1, r, st);
        if (lane == 0 && st.ok) l2_produce(tm_a2, tm_w2, p2, r, st, ready, target);
        st.ok = __shfl_sync(0xffffffffu, st.ok, 0);
        st.it = __shfl_sync(0xffffffffu, st.it, 0);
        if (!st.ok && lane == 0) drain_producer(ctrl, st.it, kL2Stages, p1.err);
        __syncwarp();
    } else if (warp == 1) {
        l1_issue(p1, r, st);
        if (st.ok) l2_issue<false>(p2, r, st);
        if (!st.ok && st.kt > 0)
            drain_wait(smem_u32(&ctrl->tfull[(st.kt - 1) % kL2TBufs]), ((st.kt - 1) / kL2TBufs) & 1, p1.err);
    } else {
        // the L1 output box is the first half of the warp's L2 output box
        l1_epilogue<kFast, true>(tm_acts, p1, r, st,
                                 base + kL2Stages * kL2StageBytes + (warp - kEpiWarp0) * kL2OutBytes, ready);
        if (st.ok)
            l2_epilogue<true, false>(tm_out, p2, r, st,
                              base + kL2Stages * kL2StageBytes + (warp - kEpiWarp0) * kL2OutBytes, ready, target);
        // this warp's output stores are complete (the epilogue waited for
        // them); order them before the barrier's release, for the combine
        fence_proxy_async_global();
    }
    gemm_teardown(tmem, warp);
    // ---- Phase 4: the combine, once every CTA's L2 outputs are stored
    bar_target += (int)gridDim.x;
    if (!grid_sync(f.bar, bar_target, p1.err) || forward_aborted(p1.err)) return;
    combine_phase(p2.l2_out, f.d.pair_pool, f.T, f.k, p2.H, f.y);
}

// The overlapped split of the two GEMMs on disjoint SM sets (PR357
// Green-Context Split MegaMoE code review, §5.2 "SM 资源划分" and §6.2 "K2"):
// L1 and L2 run at the same time, each on its own CTAs, and an L2 tile starts
// on an M block as soon as that block's L1 tiles have stored their outputs.
// On one GPU this is one cooperative launch (every CTA resident) whose CTAs
// are partitioned: CTAs [0, n1) walk the L1 tiles, CTAs [n1, grid) the L2
// tiles, through the per-M-block arrival counters of fused_kernel.  Two
// separate launches spinning on each other's counters would rely on both being
// resident at once, which nothing guarantees; one cooperative launch does.
template <bool kFast, bool kGatherA>
__global__ void __launch_bounds__(kL2Threads, 1)
    split_kernel(const __grid_constant__ AMaps tm_a1, const __grid_constant__ CUtensorMap tm_w1,
                 const __grid_constant__ CUtensorMap tm_acts, const __grid_constant__ AMaps tm_a2,
                 const __grid_constant__ CUtensorMap tm_w2, const __grid_constant__ CUtensorMap tm_out,
                 const L1Params p1, const L2Params p2, int *ready, int n1) {
    if (forward_aborted(p1.err)) return;   // an earlier step of this forward timed out
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = align1024(raw);
    Ctrl *ctrl = reinterpret_cast<Ctrl *>(smem_raw + (base - raw) + kL2Stages * kL2StageBytes +
                                          kL2EpiWarps * kL2OutBytes);
    const int warp = threadIdx.x >> 5;
    const uint32_t lane = threadIdx.x & 31;
    const bool is_l1 = (int)blockIdx.x < n1;
    if (warp == 0 && lane == 0) {
        if (is_l1) {
            tma_prefetch_desc(&tm_a1.box[0]);
            tma_prefetch_desc(&tm_w1);
        } else {
            tma_prefetch_desc(&tm_a2.box[2]);
            tma_prefetch_desc(&tm_w2);
        }
    }
    const uint32_t tmem = gemm_setup(ctrl, warp, kL2Stages, kL2TBufs, kL2EpiWarps);
    const Role r{ctrl, base, tmem, &ctrl->abort, lane, warp, is_l1 ? (int)blockIdx.x : (int)blockIdx.x - n1,
                 is_l1 ? n1 : (int)gridDim.x - n1};
    const uint32_t out_stage = base + kL2Stages * kL2StageBytes + (warp - kEpiWarp0) * kL2OutBytes;
    const int target = (p1.I / 128) * kL1EpiWarps;   // L1 tile-warps per M block
    Pipe st;
    if (is_l1) {
        if (warp == 0) {
            l1_produce<kGatherA>(tm_a1, tm_w1, p1, r, st);
            if (!st.ok) drain_producer(ctrl, st.it, kL1Stages, p1.err);
        } else if (warp == 1) {
            l1_issue(p1, r, st);
            if (!st.ok && st.kt > 0)
                drain_wait(smem_u32(&ctrl->tfull[(st.kt - 1) % kL1TBufs]), ((st.kt - 1) / kL1TBufs) & 1, p1.err);
        } else {
            l1_epilogue<kFast, true>(tm_acts, p1, r, st, out_stage, ready);
        }
    } else {
        if (warp == 0) {
            if (lane == 0) {
                l2_produce(tm_a2, tm_w2, p2, r, st, ready, target);
                if (!st.ok) drain_producer(ctrl, st.it, kL2Stages, p2.err);
            }
            __syncwarp();
        } else if (warp == 1) {
            l2_issue<true>(p2, r, st);
            if (!st.ok && st.kt > 0) {   // the last committed use: a first half (tfull) or a stage (empty)
                const int u = st.kt - 1;
                if (u & 1)
                    drain_wait(smem_u32(&ctrl->empty[(u >> 1) % kL2Stages]), ((u >> 1) / kL2Stages) & 1, p2.err);
                else
                    drain_wait(smem_u32(&ctrl->tfull[u % kL2TBufs]), (u / kL2TBufs) & 1, p2.err);
            }
        } else {
            l2_epilogue<true, true>(tm_out, p2, r, st, out_stage, ready, target);
        }
    }
    gemm_teardown(tmem, warp);
}

}  // namespace


template <bool kFast, bool kGatherA>
static void launch_l1_t(const AMaps &tm_a, const CUtensorMap &tm_w1, const CUtensorMap &tm_acts, const L1Params &p,
                        int num_sms, cudaStream_t s) {
    static std::atomic<uint32_t> smem_set{0};
    smem_limit_once(reinterpret_cast<const void *>(l1_kernel<kFast, kGatherA>), kL1SmemBytes, smem_set);
    l1_kernel<kFast, kGatherA><<<num_sms, kL1Threads, kL1SmemBytes, s>>>(tm_a, tm_w1, tm_acts, p);
}

void launch_l1(const AMaps &tm_a, const CUtensorMap &tm_w1, const CUtensorMap &tm_acts, const L1Params &p,
               int fast_math, bool gather_a, int num_sms, cudaStream_t s) {
    if (fast_math) {
        if (gather_a) launch_l1_t<true, true>(tm_a, tm_w1, tm_acts, p, num_sms, s);
        else launch_l1_t<true, false>(tm_a, tm_w1, tm_acts, p, num_sms, s);
    } else {
        if (gather_a) launch_l1_t<false, true>(tm_a, tm_w1, tm_acts, p, num_sms, s);
        else launch_l1_t<false, false>(tm_a, tm_w1, tm_acts, p, num_sms, s);
    }
}

template <bool kFast, bool kGatherA>
static cudaError_t launch_fused_t(const AMaps &tm_a1, const CUtensorMap &tm_w1, const CUtensorMap &tm_acts,
                                  const AMaps &tm_a2, const CUtensorMap &tm_w2, const CUtensorMap &tm_out,
                                  const L1Params &p1, const L2Params &p2, int *ready, const FusedParams &f,
                                  int num_sms, cudaStream_t s) {
    static std::atomic<uint32_t> smem_set{0};
    const cudaError_t e =
        smem_limit_once(reinterpret_cast<const void *>(fused_kernel<kFast, kGatherA>), kL2SmemBytes, smem_set);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;   // every CTA resident: L2 tiles wait on other CTAs' L1 tiles
    attr[0].val.cooperative = 1;
    cfg.gridDim = dim3(num_sms);
    cfg.blockDim = dim3(kL2Threads);
    cfg.dynamicSmemBytes = kL2SmemBytes;
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, fused_kernel<kFast, kGatherA>, tm_a1, tm_w1, tm_acts, tm_a2, tm_w2, tm_out, p1,
                              p2, ready, f);
}

cudaError_t launch_fused(const AMaps &tm_a1, const CUtensorMap &tm_w1, const CUtensorMap &tm_acts, const AMaps &tm_a2,
                         const CUtensorMap &tm_w2, const CUtensorMap &tm_out, const L1Params &p1, const L2Params &p2,
                         int *ready, const FusedParams &f, int fast_math, bool gather_a, int num_sms, cudaStream_t s) {
    if (num_sms > kDispatchMcMaxCtas || p1.E > 1024) return cudaErrorInvalidValue;
    if (fast_math)
        return gather_a ? launch_fused_t<true, true>(tm_a1, tm_w1, tm_acts, tm_a2, tm_w2, tm_out, p1, p2, ready, f,
                                                     num_sms, s)
                        : launch_fused_t<true, false>(tm_a1, tm_w1, tm_acts, tm_a2, tm_w2, tm_out, p1, p2, ready, f,
                                                      num_sms, s);
    return gather_a ? launch_fused_t<false, true>(tm_a1, tm_w1, tm_acts, tm_a2, tm_w2, tm_out, p1, p2, ready, f,
                                                  num_sms, s)
                    : launch_fused_t<false, false>(tm_a1, tm_w1, tm_acts, tm_a2, tm_w2, tm_out, p1, p2, ready, f,
                                                   num_sms, s);
}

template <bool kFast, bool kGatherA>
static cudaError_t launch_split_t(const AMaps &tm_a1, const CUtensorMap &tm_w1, const CUtensorMap &tm_acts,
                                  const AMaps &tm_a2, const CUtensorMap &tm_w2, const CUtensorMap &tm_out,
                                  const L1Params &p1, const L2Params &p2, int *ready, int n1, int num_sms,
                                  cudaStream_t s) {
    static std::atomic<uint32_t> smem_set{0};
    const cudaError_t e =
        smem_limit_once(reinterpret_cast<const void *>(split_kernel<kFast, kGatherA>), kL2SmemBytes, smem_set);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;   // every CTA resident: L2 CTAs wait on the L1 CTAs' counters
    attr[0].val.cooperative = 1;
    cfg.gridDim = dim3(num_sms);
    cfg.blockDim = dim3(kL2Threads);
    cfg.dynamicSmemBytes = kL2SmemBytes;
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, split_kernel<kFast, kGatherA>, tm_a1, tm_w1, tm_acts, tm_a2, tm_w2, tm_out, p1,
                              p2, ready, n1);
}

cudaError_t launch_split(const AMaps &tm_a1, const CUtensorMap &tm_w1, const CUtensorMap &tm_acts, const AMaps &tm_a2,
                         const CUtensorMap &tm_w2, const CUtensorMap &tm_out, const L1Params &p1, const L2Params &p2,
                         int *ready, int n1, int fast_math, bool gather_a, int num_sms, cudaStream_t s) {
    if (n1 < 1 || n1 >= num_sms) return cudaErrorInvalidValue;
    if (fast_math)
        return gather_a ? launch_split_t<true, true>(tm_a1, tm_w1, tm_acts, tm_a2, tm_w2, tm_out, p1, p2, ready, n1,
                                                     num_sms, s)
                        : launch_split_t<true, false>(tm_a1, tm_w1, tm_acts, tm_a2, tm_w2, tm_out, p1, p2, ready, n1,
                                                      num_sms, s);
    return gather_a ? launch_split_t<false, true>(tm_a1, tm_w1, tm_acts, tm_a2, tm_w2, tm_out, p1, p2, ready, n1,
                                                  num_sms, s)
                    : launch_split_t<false, false>(tm_a1, tm_w1, tm_acts, tm_a2, tm_w2, tm_out, p1, p2, ready, n1,
                                                   num_sms, s);
}

void launch_l2(const AMaps &tm_a, const CUtensorMap &tm_w2, const CUtensorMap &tm_out, const L2Params &p,
               int num_sms, cudaStream_t s) {
    static std::atomic<uint32_t> smem_set{0};
    smem_limit_once(reinterpret_cast<const void *>(l2_kernel), kL2SmemBytes, smem_set);
    l2_kernel<<<num_sms, kL2Threads, kL2SmemBytes, s>>>(tm_a, tm_w2, tm_out, p);
}

}  // namespace moe
