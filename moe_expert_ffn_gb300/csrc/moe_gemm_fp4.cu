// moe_gemm_fp4.cu -- the grouped GEMMs of the FP4-weight configuration.
//
// Weights are FP4 E2M1 (two codes per byte, low nibble = even k) with one
// UE8M0 scale per 32 K; activations are FP8 E4M3 with one UE8M0 scale per 32
// K (PR357 Green-Context Split MegaMoE code review, §1 "SM100 FP8/FP4
// MegaMoE", §6.2 "MXF8F6F4 UMMA"; MegaMoE SM90 Implementation Design (Final),
// §2.1 "FP4 Tensor Core (E2M1)", "Scale Factor Format").  Both scale kinds are
// powers of two, so the tensor core applies them itself: tcgen05.mma
// kind::mxf8f6f4 with block_scale, one scale per row per K=32 step, and the
// whole K loop accumulates in one TMEM accumulator (no promotion in the
// epilogue).
//
//   L1: h = x . W1^T, then SwiGLU * w and FP8 requantisation with one UE8M0
//       scale per 32 columns, 2^ceil(log2(amax/448)) (PR357 review §6.1
//       "SwiGLU/quant"; design §10.1);
//   L2: o = q . W2^T rounded to BF16 (design §11.1).
//
// Weight tiles are loaded by TMA straight from the packed codes: the tensor
// map type 16U4_ALIGN16B expands every 16 codes (8 bytes) into a 16-byte slot,
// the layout the f8f6f4 MMA reads for E2M1, so HBM moves half a byte per
// weight.  Such a copy costs an SM about the same time whether its box has
// 128 or 256 rows, so tiles are 128 rows x 256 columns (one 256-row weight
// box per stage), K stages of 128.  Warp roles, 10 warps:
//   warp 0     TMA producer (4 stages: A 16 KB, B 32 KB);
//   warp 1     TMEM allocation, then MMA issuer;
//   warps 2-5  scale writers: for every stage they load the UE8M0 words (four
//              K steps per 32-bit word) of the tile's 128 A rows and 256 B rows
//              and tcgen05.st them into a TMEM slot of the scale ring.  The MMA
//              reads the scale of row r from TMEM lane 32*(m/32) + r%32 (m =
//              the output row being computed), column base + r/32, so each lane
//              quadrant holds a full copy: lane 32q + j, column base + c = row
//              32c + j.  They take a stage slot when the MMA's commit frees it
//              (the producer's empty barrier) and arrive on the slot's full
//              barrier next to the producer, so the MMA issuer waits once per
//              stage and commits once;
//   warps 6-9  epilogue, one per TMEM lane quadrant: each thread moves the
//              first 128 of its row's 256 accumulator columns to a TMEM stash,
//              reads the second 128 into registers and frees the accumulator
//              (so the next tile's MMAs start after two copies, not after the
//              conversion), then converts and stores each half (64 gate/up
//              pairs, or 128 outputs).  One 256-column accumulator, the scale
//              ring and the stash fit in TMEM.
#include "moe_device.cuh"
#include "moe_gemm_common.cuh"
#include "moe_internal.h"

namespace moe {
namespace {

constexpr int kThreads = 320;
constexpr int kBN = 256;
constexpr int kStages = 4;
constexpr uint32_t kABytes = kBM * kBK;
constexpr uint32_t kBBytes = kBN * kBK;                 // E2M1 expanded to one byte per code
constexpr uint32_t kBTxBytes = kBN * kBK / 2;           // a 16U4 load counts the packed bytes
constexpr uint32_t kStageBytes = kABytes + kBBytes;
constexpr uint32_t kTmemCols = 512;
constexpr int kAccs = 1;                                // 256-column accumulators
constexpr uint32_t kSfCol0 = kAccs * kBN;               // scale ring after the accumulators
constexpr uint32_t kSfACols = kBM / 32;                 // A scales: one column per 32 rows
constexpr uint32_t kSfSlotCols = 16;                    // then B scales (8 columns); 16-aligned slots
static_assert(kSfACols + kBN / 32 <= kSfSlotCols, "scale slot");
constexpr uint32_t kStashCol0 = kSfCol0 + kStages * kSfSlotCols;   // 128 columns: the epilogue's first half
constexpr int kNumSfWarps = 4;
constexpr int kNumEpiWarps = 4;
constexpr int kEpiWarp0 = 6;                           // warps 2..5 write scales
static_assert(kStashCol0 + 128 <= kTmemCols, "TMEM budget");

struct alignas(8) Ctrl {
    uint64_t full[kStages];
    uint64_t empty[kStages];
    uint64_t acc_full[kAccs];
    uint64_t acc_empty[kAccs];
    uint32_t tmem_base;
    int abort;
};
constexpr size_t kCtrlBytes = 512;
static_assert(sizeof(Ctrl) <= kCtrlBytes, "ctrl");
// L2 output staging: per epilogue warp 32 rows x 64 BF16 columns (one TMA
// store box, 128-byte swizzled).  L1 has none: its scale writers re-read the
// tile's scale rows from the L1 cache every stage, and every 16 KB taken from
// it for shared memory showed (L1 2.3x slower with it).
constexpr uint32_t kOutBytes = 32 * 128;
template <bool kL1>
constexpr uint32_t out_stage_bytes() { return kL1 ? 0u : (uint32_t)kNumEpiWarps * kOutBytes; }
template <bool kL1>
constexpr size_t smem_bytes() { return 1024 + (size_t)kStages * kStageBytes + out_stage_bytes<kL1>() + kCtrlBytes; }
static_assert(smem_bytes<false>() <= 232448, "shared memory");

__device__ __forceinline__ uint32_t ld_u32(const uint8_t *p) {
    return __ldg(reinterpret_cast<const uint32_t *>(p));
}

// UE8M0 exponent of the smallest power of two 2^e with amax/448 <= 2^e (the
// ratio in binary32), e in [-127, 127]; -127 for an all-zero group.
__device__ __forceinline__ int ue8m0_exponent(float amax) {
    const float r = amax / 448.0f;
    if (!(r > 0.0f)) return -127;
    int ex;
    const float fr = frexpf(r, &ex);
    int e = (fr == 0.5f) ? ex - 1 : ex;
    return min(127, max(-127, e));
}

template <bool kL1, bool kFast, bool kGatherA>
__global__ void __launch_bounds__(kThreads, 1)
    fp4_gemm_kernel(const __grid_constant__ AMaps tm_a, const __grid_constant__ CUtensorMap tm_b,
                    const __grid_constant__ CUtensorMap tm_out, const Fp4Params p) {
    if (forward_aborted(p.err)) return;   // an earlier step of this forward timed out
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = align1024(raw);
    Ctrl *ctrl = reinterpret_cast<Ctrl *>(smem_raw + (base - raw) + kStages * kStageBytes +
                                          out_stage_bytes<kL1>());
    const int warp = threadIdx.x >> 5;
    const uint32_t lane = threadIdx.x & 31;

    // N blocks: L1 covers the 2I interleaved rows exactly; L2's last block is
    // half empty when H % 256 == 128
    const int NB = kL1 ? 2 * p.I / kBN : (p.H + kBN - 1) / kBN;
    const int KB = kL1 ? p.H / kBK : p.I / kBK;
    const int brow0 = kL1 ? 2 * p.I : p.H;          // B rows per expert
    const int sf_row_bytes = (kL1 ? p.H : p.I) / 32; // scale bytes per row of A and B
    int total, singles;
    tile_counts(p.mb_prefix, p.E, NB, total, singles);

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(smem_u32(&ctrl->full[s]), 1 + kNumSfWarps);   // the copies and the scale writers
            mbar_init(smem_u32(&ctrl->empty[s]), 1);
        }
        for (int b = 0; b < kAccs; ++b) {
            mbar_init(smem_u32(&ctrl->acc_full[b]), 1);
            mbar_init(smem_u32(&ctrl->acc_empty[b]), kNumEpiWarps);
        }
        ctrl->abort = 0;
        fence_mbar_init();
        tma_prefetch_desc(&tm_a.box[0]);
        tma_prefetch_desc(&tm_a.box[2]);
        tma_prefetch_desc(&tm_b);
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(&ctrl->tmem_base), kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = ctrl->tmem_base;
    volatile int *abort_flag = &ctrl->abort;

    if (warp == 0) {
        // ---------------- TMA producer ----------------
        const uint64_t pol_once = policy_evict_first();
        const uint64_t pol_shared = policy_evict_normal();
        const uint64_t pol_a = policy_evict_last();
        const bool stall = test_stall(p.err, kL1 ? kStallL1 : kStallL2, blockIdx.x);
        int it = 0;
        bool ok = true;
        for (int tile = blockIdx.x; ok && tile < total; tile += gridDim.x) {
            const Tile t = decode_tile(tile_at_position(tile, total, singles), NB, p.offset, p.mb_prefix, p.mblk_expert);
            const uint64_t pol_w = t.nmb > 1 ? pol_shared : pol_once;
            int tok[4] = {0, 0, 0, 0};
            if (kGatherA) {
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int r = (int)lane * 4 + i;
                    tok[i] = r < t.rows ? __ldg(p.gather + t.row0 + r) / p.k : 0;
                }
            }
            const int n_g4 = (t.rows + 3) >> 2;
            const int abox = a_box_index(t.rows);
            const uint32_t tx = (kGatherA ? (uint32_t)n_g4 * 4 * kBK : (32u << abox) * kBK) + kBTxBytes;
            const int brow = t.e * brow0 + t.nb * kBN;
            for (int kb = 0; kb < KB; ++kb, ++it) {
                const int s = it % kStages;
                const uint32_t ph = (it / kStages) & 1;
                if (!mbar_wait(smem_u32(&ctrl->empty[s]), ph ^ 1, abort_flag, p.err)) {
                    ok = false;
                    break;
                }
                if (stall && it == 0) continue;   // timeout-path test: never fill the first stage
                const uint32_t full = smem_u32(&ctrl->full[s]);
                if (lane == 0) mbar_arrive_expect_tx(full, tx);
                __syncwarp();
                if (kGatherA) {
                    if ((int)lane < n_g4)
                        tma_gather4(base + s * kStageBytes + lane * 512, &tm_a.box[0], kb * kBK, tok[0], tok[1],
                                    tok[2], tok[3], full, pol_a);
                } else if (lane == 0) {
                    tma_load_2d(base + s * kStageBytes, &tm_a.box[abox], kb * kBK, t.row0, full, pol_a);
                }
                if (lane == 0)
                    tma_load_2d(base + s * kStageBytes + kABytes, &tm_b, kb * kBK, brow, full, pol_w);
            }
        }
        if (!ok)
            for (int i = max(0, it - kStages); i < it; ++i)
                drain_wait(smem_u32(&ctrl->full[i % kStages]), (i / kStages) & 1, p.err);
    } else if (warp == 1) {
        // ---------------- MMA issuer ----------------
        int it = 0, tc = 0;
        bool ok = true;
        for (int tile = blockIdx.x; ok && tile < total; tile += gridDim.x, ++tc) {
            const int b = tc % kAccs;
            if (!mbar_wait(smem_u32(&ctrl->acc_empty[b]), ((tc / kAccs) & 1) ^ 1, abort_flag, p.err)) {
                ok = false;
                break;
            }
            for (int kb = 0; kb < KB; ++kb, ++it) {
                const int s = it % kStages;
                const uint32_t ph = (it / kStages) & 1;
                if (!mbar_wait(smem_u32(&ctrl->full[s]), ph, abort_flag, p.err)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                if (lane == 0) {
                    const uint64_t ad = sw128_kmajor_desc(base + s * kStageBytes);
                    const uint64_t bd = sw128_kmajor_desc(base + s * kStageBytes + kABytes);
                    const uint32_t sfa = tmem + kSfCol0 + s * kSfSlotCols;
#pragma unroll
                    for (int kk = 0; kk < kBK / 32; ++kk)
                        umma_mx(tmem + b * kBN, ad + 2 * kk, bd + 2 * kk, idesc_mx_e4m3_e2m1(kBM, kBN, kk),
                                sfa, sfa + kSfACols, (kb | kk) != 0);
                    umma_commit(smem_u32(&ctrl->empty[s]));
                    if (kb == KB - 1) umma_commit(smem_u32(&ctrl->acc_full[b]));
                }
                __syncwarp();
            }
        }
        if (!ok && it > 0)
            drain_wait(smem_u32(&ctrl->empty[(it - 1) % kStages]), ((it - 1) / kStages) & 1, p.err);
    } else if (warp < kEpiWarp0) {
        // ---------------- scale writers ----------------
        const int q = warp & 3;
        const uint32_t t_lane = tmem + (static_cast<uint32_t>(q * 32) << 16) + kSfCol0;
        int it = 0;
        bool ok = true;
        for (int tile = blockIdx.x; ok && tile < total; tile += gridDim.x) {
            const Tile t = decode_tile(tile_at_position(tile, total, singles), NB, p.offset, p.mb_prefix, p.mblk_expert);
            // row c*32 + lane of the tile: A pool rows c = 0..3, B weight rows
            // c = 0..7 (rows past the expert's last weight row, in a half-empty
            // L2 block, reuse that row: their outputs are masked)
            const uint8_t *arow[4];
            const uint8_t *brow[8];
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const int r = 32 * c + (int)lane;
                const int prow = t.row0 + min(r, t.rows - 1);   // masked rows reuse a valid row
                if (kL1)
                    arow[c] = p.a_sf + (size_t)(__ldg(p.gather + prow) / p.k) * sf_row_bytes;
                else
                    arow[c] = p.a_sf + (size_t)prow * sf_row_bytes;
            }
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                const int r = min(t.nb * kBN + 32 * c + (int)lane, brow0 - 1);
                brow[c] = p.b_sf + (size_t)(t.e * brow0 + r) * sf_row_bytes;
            }
            uint32_t wa[4], wb[8];
#pragma unroll
            for (int c = 0; c < 4; ++c) wa[c] = ld_u32(arow[c]);
#pragma unroll
            for (int c = 0; c < 8; ++c) wb[c] = ld_u32(brow[c]);
            for (int kb = 0; kb < KB; ++kb, ++it) {
                const int s = it % kStages;
                const uint32_t ph = (it / kStages) & 1;
                // words of the next K block, loaded while this one is stored
                uint32_t na[4], nbw[8];
                const int kn = min(kb + 1, KB - 1) * 4;
#pragma unroll
                for (int c = 0; c < 4; ++c) na[c] = ld_u32(arow[c] + kn);
#pragma unroll
                for (int c = 0; c < 8; ++c) nbw[c] = ld_u32(brow[c] + kn);
                if (!mbar_wait(smem_u32(&ctrl->empty[s]), ph ^ 1, abort_flag, p.err)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t col = t_lane + s * kSfSlotCols;
                tmem_st4(col, wa[0], wa[1], wa[2], wa[3]);
                tmem_st4(col + kSfACols, wb[0], wb[1], wb[2], wb[3]);
                tmem_st4(col + kSfACols + 4, wb[4], wb[5], wb[6], wb[7]);
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&ctrl->full[s]));
#pragma unroll
                for (int c = 0; c < 4; ++c) wa[c] = na[c];
#pragma unroll
                for (int c = 0; c < 8; ++c) wb[c] = nbw[c];
            }
        }
    } else {
        // ---------------- epilogue ----------------
        const int q = warp & 3;
        const int lrow = q * 32 + (int)lane;
        const uint32_t t_lane = tmem + (static_cast<uint32_t>(q * 32) << 16);
        const uint32_t out_stage = base + kStages * kStageBytes + (warp - kEpiWarp0) * kOutBytes;
        int tc = 0;
        bool ok = true;
        for (int tile = blockIdx.x; ok && tile < total; tile += gridDim.x, ++tc) {
            const Tile t = decode_tile(tile_at_position(tile, total, singles), NB, p.offset, p.mb_prefix, p.mblk_expert);
            const int b = tc % kAccs;
            if (!mbar_wait(smem_u32(&ctrl->acc_full[b]), (tc / kAccs) & 1, abort_flag, p.err)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const bool valid = lrow < t.rows;
            const bool warp_on = q * 32 < t.rows;
            const int row = t.row0 + lrow;
            // first half -> stash, second half -> registers, free the accumulator
            float acc[128];
            if (warp_on) {
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    float v[32];
                    tmem_ld32(t_lane + b * kBN + 32 * c, v);
                    tmem_ld_wait();
                    tmem_st32(t_lane + kStashCol0 + 32 * c, v);
                }
                tmem_st_wait();
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    float v[32];
                    tmem_ld32(t_lane + b * kBN + 128 + 32 * c, v);
                    tmem_ld_wait();
#pragma unroll
                    for (int i = 0; i < 32; ++i) acc[32 * c + i] = v[i];
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&ctrl->acc_empty[b]));
            // convert the second half (in registers), then the first (from the stash)
#pragma unroll 1
            for (int pass = 0; pass < 2; ++pass) {
                const int h = 1 - pass;
                const int cb = t.nb * 2 + h;   // 128-column block of the output
                if (pass == 1 && warp_on) {
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        float v[32];
                        tmem_ld32(t_lane + kStashCol0 + 32 * c, v);
                        tmem_ld_wait();
#pragma unroll
                        for (int i = 0; i < 32; ++i) acc[32 * c + i] = v[i];
                    }
                }
                if (!valid) continue;
                if (kL1) {
                    // SwiGLU * top-k weight (gate columns 0-7, up columns 8-15 of every 16)
                    const float wgt = __ldg(p.topk_w + __ldg(p.gather + row));
                    const float clampv = p.clamp;
#pragma unroll
                    for (int o = 0; o < 64; ++o) {
                        const int gi = 16 * (o >> 3) + (o & 7);
                        const float g = fminf(fmaxf(acc[gi], -clampv), clampv);
                        const float u = fminf(fmaxf(acc[gi + 8], -clampv), clampv);
                        float silu;
                        if (kFast)
                            silu = __fdividef(g, 1.0f + __expf(-g));
                        else
                            silu = __fdividef(g, 1.0f + expf(-g));
                        acc[gi] = silu * u * wgt;
                    }
                    // two 32-column groups, UE8M0 scale 2^ceil(log2(amax/448)) each
                    uint32_t pk[16];
                    uint32_t codes = 0;
#pragma unroll
                    for (int grp = 0; grp < 2; ++grp) {
                        float amax = 0.0f;
#pragma unroll
                        for (int o = 32 * grp; o < 32 * grp + 32; ++o)
                            amax = fmaxf(amax, fabsf(acc[16 * (o >> 3) + (o & 7)]));
                        const int e = ue8m0_exponent(amax);
                        // a / 2^e as a * 2^-e: both exact powers of two, the same rounding
                        const float rsf = ldexpf(1.0f, -e);
                        codes |= static_cast<uint32_t>(e + 127) << (8 * grp);
#pragma unroll
                        for (int w4 = 8 * grp; w4 < 8 * grp + 8; ++w4) {
                            float qv[4];
#pragma unroll
                            for (int j = 0; j < 4; ++j) {
                                const int o = w4 * 4 + j;
                                const float a = acc[16 * (o >> 3) + (o & 7)];
                                qv[j] = (amax == 0.0f) ? 0.0f : a * rsf;
                            }
                            pk[w4] = e4m3x2(qv[0], qv[1]) | (e4m3x2(qv[2], qv[3]) << 16);
                        }
                    }
                    // outputs [64 cb, 64 cb + 64) of the intermediate dimension
                    uint4 *dst = reinterpret_cast<uint4 *>(p.l2_acts + (size_t)row * p.acts_pitch + cb * 64);
#pragma unroll
                    for (int v = 0; v < 4; ++v)
                        dst[v] = make_uint4(pk[4 * v], pk[4 * v + 1], pk[4 * v + 2], pk[4 * v + 3]);
                    *reinterpret_cast<uint16_t *>(p.l2_sf + (size_t)row * (p.I / 32) + 2 * cb) =
                        static_cast<uint16_t>(codes);
                } else if (cb * 128 < p.H && q * 32 + 32 <= t.rows) {
                    // all 32 rows of the warp valid: two 32 x 64 boxes through
                    // shared memory and the copy engine (whole 128-byte row pieces)
#pragma unroll
                    for (int k = 0; k < 2; ++k) {
                        if (lane == 0) tma_store_wait_read();   // the previous box has left the buffer
                        __syncwarp();
                        const uint32_t rowp = out_stage + lane * 128;
#pragma unroll
                        for (int c = 0; c < 8; ++c) {
                            const int i = 64 * k + 8 * c;
                            st_shared_v4(rowp + ((c ^ (lane & 7)) << 4), bf16x2(acc[i], acc[i + 1]),
                                         bf16x2(acc[i + 2], acc[i + 3]), bf16x2(acc[i + 4], acc[i + 5]),
                                         bf16x2(acc[i + 6], acc[i + 7]));
                        }
                        fence_async_smem();
                        __syncwarp();
                        if (lane == 0) {
                            tma_store_2d(&tm_out, cb * 128 + 64 * k, t.row0 + q * 32, out_stage);
                            tma_store_commit();
                        }
                    }
                } else if (cb * 128 < p.H) {
                    uint4 *dst = reinterpret_cast<uint4 *>(p.l2_out + (size_t)row * p.H + cb * 128);
#pragma unroll
                    for (int v = 0; v < 16; ++v)
                        dst[v] = make_uint4(bf16x2(acc[8 * v + 0], acc[8 * v + 1]),
                                            bf16x2(acc[8 * v + 2], acc[8 * v + 3]),
                                            bf16x2(acc[8 * v + 4], acc[8 * v + 5]),
                                            bf16x2(acc[8 * v + 6], acc[8 * v + 7]));
                }
            }
        }
        if (!kL1) {
            if (lane == 0) tma_store_wait_all();
            __syncwarp();
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

template <bool kL1, bool kFast, bool kGatherA>
void launch_t(const AMaps &tm_a, const CUtensorMap &tm_b, const CUtensorMap &tm_out, const Fp4Params &p,
              int num_sms, cudaStream_t s) {
    static std::atomic<uint32_t> smem_set{0};
    smem_limit_once(reinterpret_cast<const void *>(fp4_gemm_kernel<kL1, kFast, kGatherA>), smem_bytes<kL1>(),
                    smem_set);
    fp4_gemm_kernel<kL1, kFast, kGatherA><<<num_sms, kThreads, smem_bytes<kL1>(), s>>>(tm_a, tm_b, tm_out, p);
}

}  // namespace

void launch_fp4_l1(const AMaps &tm_a, const CUtensorMap &tm_w1, const Fp4Params &p,
                   int fast_math, bool gather_a, int num_sms, cudaStream_t s) {
    // (the output map is not used by L1; its codes leave by plain stores)
    if (fast_math) {
        if (gather_a) launch_t<true, true, true>(tm_a, tm_w1, tm_w1, p, num_sms, s);
        else launch_t<true, true, false>(tm_a, tm_w1, tm_w1, p, num_sms, s);
    } else {
        if (gather_a) launch_t<true, false, true>(tm_a, tm_w1, tm_w1, p, num_sms, s);
        else launch_t<true, false, false>(tm_a, tm_w1, tm_w1, p, num_sms, s);
    }
}

void launch_fp4_l2(const AMaps &tm_a, const CUtensorMap &tm_w2, const CUtensorMap &tm_out, const Fp4Params &p,
                   int num_sms, cudaStream_t s) {
    launch_t<false, false, false>(tm_a, tm_w2, tm_out, p, num_sms, s);
}

}  // namespace moe
