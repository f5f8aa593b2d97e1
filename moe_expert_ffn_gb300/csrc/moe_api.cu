// moe_api.cu -- the C ABI declared in include/moe.h: workspace carving, TMA
// tensor maps, argument checks and the launch sequence of one forward
// (dispatch -> L1 GEMM -> L2 GEMM -> combine) on the caller's stream.
#include <math.h>
#include <stdlib.h>
#include <string.h>

#include "moe.h"
#include "moe_device.cuh"
#include "moe_internal.h"

using namespace moe;

namespace {

constexpr size_t kAlign = 1024;

// Row pitch padding of the row-major operands the GEMMs read with TMA: rows
// of a 2^k-byte pitch put every row of a tile (and the same K offset of all
// concurrent tiles) on the same few memory partitions; one extra 256-byte
// segment per row spreads them.  256 bytes, not 128: the tensor maps fill L2
// in 256-byte lines, and with a pitch that is an odd multiple of 128 every
// other row starts in the middle of a line, so its first and last lines are
// half another row's padding (measured: 2.9% more DRAM reads than the
// weight bytes in the decode L2 GEMM, 0.9% in L1).
constexpr size_t kPitchPad = 256;

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

struct Layout {
    size_t pool_pitch, acts_pitch, w1_pitch, w2_pitch;   // bytes per row
    // workspace
    size_t err, count, offset, mb_prefix, mblk_expert, mb2_prefix, mblk2_expert, gather, pair_pool, ready;
    size_t dcnt;   // per-CTA expert counts of the multi-CTA dispatch
    size_t pool, l2_acts, l2_sf, l2_out;
    size_t st_x, st_xsf, st_idx, st_w, st_y;
    size_t ws_total;
    // weights
    size_t w1i, w1i_sf, w2, w2_sf;
    size_t wt_total;
};

bool valid_cfg(const moe_config *c) {
    if (!c) return false;
    if (c->max_tokens < 1 || c->hidden < 128 || c->inter < 128) return false;
    if (c->hidden % 128 || c->inter % 128) return false;
    if (c->num_experts < 1 || c->num_experts > 1024) return false;
    if (c->topk < 1 || c->topk > 32 || c->topk > c->num_experts) return false;
    if (c->wfmt != MOE_W_FP8_BLK128 && c->wfmt != MOE_W_FP4_E2M1_UE8M0_32) return false;
    if (isnan(c->act_clamp) || c->act_clamp <= 0.0f) return false;
    const long long pm = (long long)c->max_tokens * c->topk;
    if (pm > (1ll << 24)) return false;
    if ((long long)c->num_experts * 2 * c->inter >= (1ll << 31)) return false;
    if ((long long)c->num_experts * c->hidden >= (1ll << 31)) return false;
    return true;
}

Layout make_layout(const moe_config *c) {
    Layout L;
    const size_t Tm = c->max_tokens, k = c->topk, E = c->num_experts, H = c->hidden, I = c->inter;
    const size_t Pm = Tm * k;
    const size_t MBmax = Pm / kBM + E + 1;
    const bool fp4 = c->wfmt == MOE_W_FP4_E2M1_UE8M0_32;
    L.pool_pitch = H + kPitchPad;
    L.acts_pitch = I + kPitchPad;
    L.w1_pitch = (fp4 ? H / 2 : H) + kPitchPad;
    L.w2_pitch = (fp4 ? I / 2 : I) + kPitchPad;
    size_t o = 0;
    auto take = [&](size_t bytes, size_t align) {
        o = align_up(o, align);
        const size_t at = o;
        o += bytes;
        return at;
    };
    L.err = take(sizeof(int) * kErrWords, 256);
    L.count = take(4 * E, 256);
    L.offset = take(4 * (E + 1), 256);
    L.mb_prefix = take(4 * (E + 2), 256);
    L.mblk_expert = take(4 * MBmax, 256);
    L.mb2_prefix = take(4 * (E + 1), 256);
    L.mblk2_expert = take(4 * (Pm / (2 * kBM) + E + 1), 256);
    L.ready = take(4 * MBmax, 256);   // M-block arrival counters of the one-launch GEMM pair
    L.dcnt = take(4 * (size_t)kDispatchMcMaxCtas * E, 256);
    L.gather = take(4 * Pm, 256);
    L.pair_pool = take(4 * Pm, 256);
    L.pool = take(Pm * L.pool_pitch, kAlign);
    L.l2_acts = take(Pm * L.acts_pitch, kAlign);
    L.l2_sf = take(4 * (I / 64) * Pm, kAlign);
    L.l2_out = take(2 * Pm * H, kAlign);
    L.st_x = take(Tm * H, kAlign);
    L.st_xsf = take(4 * Tm * (H / 128), 256);
    L.st_idx = take(4 * Tm * k, 256);
    L.st_w = take(4 * Tm * k, 256);
    L.st_y = take(2 * Tm * H, kAlign);
    L.ws_total = align_up(o, kAlign);

    o = 0;
    if (!fp4) {
        L.w1i = take(E * 2 * I * L.w1_pitch, kAlign);
        L.w1i_sf = take(8 * E * (2 * I / 128) * (H / 128), 256);
        L.w2 = take(E * H * L.w2_pitch, kAlign);
        L.w2_sf = take(4 * E * (H / 128) * (I / 128), 256);
    } else {   // packed E2M1 rows and per-32 UE8M0 scale rows
        L.w1i = take(E * 2 * I * L.w1_pitch, kAlign);
        L.w1i_sf = take(E * 2 * I * H / 32, 256);
        L.w2 = take(E * H * L.w2_pitch, kAlign);
        L.w2_sf = take(E * H * I / 32, 256);
    }
    L.wt_total = align_up(o, kAlign);
    return L;
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    if (!fn) {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    }
    return fn;
}

// 2-D tensor [outer, inner] with row stride `stride` bytes, boxes of
// box_inner x box_outer elements, 128-byte swizzle unless asked otherwise.
// Bytes (box_inner 128), 16-bit words, or packed 4-bit codes expanded to one
// byte each in shared memory (16U4_ALIGN16B: inner counts codes, box_inner 128).
bool make_map(CUtensorMap *m, const void *base, uint64_t inner, uint64_t outer, uint64_t stride,
              uint32_t box_inner, uint32_t box_outer,
              CUtensorMapDataType dtype = CU_TENSOR_MAP_DATA_TYPE_UINT8,
              CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_128B) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {inner, outer};
    cuuint64_t strides[1] = {stride};
    cuuint32_t box[2] = {box_inner, box_outer};
    cuuint32_t es[2] = {1, 1};
    return fn(m, dtype, 2, const_cast<void *>(base), dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The same rows as a 3-D tensor [inner/128 panels][outer rows][128 bytes], so
// that one box of box_panels panels x box_outer rows fetches several 128-byte
// K panels of the same rows (each panel a separate 128-byte-swizzled tile).
bool make_map_panels(CUtensorMap *m, const void *base, uint64_t inner, uint64_t outer, uint64_t stride,
                     uint32_t box_outer, uint32_t box_panels) {
    EncodeTiledFn fn = encode_fn();
    if (!fn || inner % 128) return false;
    cuuint64_t dims[3] = {128, outer, inner / 128};
    cuuint64_t strides[2] = {stride, 128};
    cuuint32_t box[3] = {128, box_outer, box_panels};
    cuuint32_t es[3] = {1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void *>(base), dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Bytes of the activation scales of T tokens.
size_t x_sf_bytes(const moe_config &g, int T) {
    return g.wfmt == MOE_W_FP8_BLK128 ? (size_t)T * (g.hidden / 128) * 4 : (size_t)T * (g.hidden / 32);
}

}  // namespace

struct moe_ctx {
    moe_config cfg;
    Layout L;
    int device;
    int num_sms;
    uint8_t *ws;
    uint8_t *wt;
    bool weights_ready;
    int last_T;
    CUtensorMap tm_w1, tm_w2;
    CUtensorMap tm_l2out;   // l2_out [Pmax, H] BF16, 32-row x 64-column boxes (L2 epilogue stores)
    CUtensorMap tm_acts;    // l2_acts [Pmax, I] FP8, 32-row x 64-byte boxes (L1 epilogue stores)
    CUtensorMap tm_w1h;     // FP8 W1i as K panels, 128 rows x 2 panels per box (CTA-pair L1)
    CUtensorMap tm_pool3;   // the pool the same way
    AMaps tm_l2a, tm_pool;
    int l1_a_mode;          // 0 auto, 1 gather4 from x, 2 pool
    int l1_pair_mode;       // 0 auto, 1 CTA pairs, 2 single CTAs
    bool fused;             // both FP8 GEMMs in one cooperative launch (MOE_FUSED=1)
    int split_l1;           // > 0: the two FP8 GEMMs at once on disjoint CTA sets, this many on L1 (MOE_SPLIT)
    int test_hook[2];       // armed timeout test for the next forward: {limit us, stall target}
    bool test_armed;
    cudaEvent_t *prof_ev;   // 5 events per profiled forward
    int prof_max, prof_n;

    template <class T>
    T *w(size_t off) const { return reinterpret_cast<T *>(ws + off); }
    template <class T>
    T *wt_at(size_t off) const { return reinterpret_cast<T *>(wt + off); }
};

extern "C" {

size_t moe_workspace_bytes(const moe_config *cfg) {
    if (!valid_cfg(cfg)) return 0;
    return make_layout(cfg).ws_total;
}

size_t moe_weight_bytes(const moe_config *cfg) {
    if (!valid_cfg(cfg)) return 0;
    return make_layout(cfg).wt_total;
}

int moe_create(moe_ctx **out, const moe_config *cfg, void *d_workspace, void *d_weights) {
    if (!out || !valid_cfg(cfg) || !d_workspace || !d_weights) return MOE_ERR_INVALID_ARG;
    if (!aligned(d_workspace, 256) || !aligned(d_weights, 256)) return MOE_ERR_INVALID_ARG;
    moe_ctx *c = static_cast<moe_ctx *>(calloc(1, sizeof(moe_ctx)));
    if (!c) return MOE_ERR_INVALID_ARG;
    c->cfg = *cfg;
    c->L = make_layout(cfg);
    c->ws = static_cast<uint8_t *>(d_workspace);
    c->wt = static_cast<uint8_t *>(d_weights);
    if (cudaGetDevice(&c->device) != cudaSuccess ||
        cudaDeviceGetAttribute(&c->num_sms, cudaDevAttrMultiProcessorCount, c->device) != cudaSuccess) {
        free(c);
        return MOE_ERR_CUDA;
    }
    const moe_config &g = c->cfg;
    const uint64_t E = g.num_experts, H = g.hidden, I = g.inter;
    const uint64_t Pm = (uint64_t)g.max_tokens * g.topk;
    const bool fp4 = g.wfmt == MOE_W_FP4_E2M1_UE8M0_32;
    const CUtensorMapDataType packed = CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B;
    const Layout &L = c->L;
    bool ok = (fp4 ? make_map(&c->tm_w1, c->wt + L.w1i, H, E * 2 * I, L.w1_pitch, 128, 256, packed) &&
                         make_map(&c->tm_w2, c->wt + L.w2, I, E * H, L.w2_pitch, 128, 256, packed)
                   : make_map(&c->tm_w1, c->wt + L.w1i, H, E * 2 * I, L.w1_pitch, 128, 256) &&
                         make_map_panels(&c->tm_w1h, c->wt + L.w1i, H, E * 2 * I, L.w1_pitch, 128, 2) &&
                         make_map_panels(&c->tm_pool3, c->ws + L.pool, H, Pm, L.pool_pitch, 128, 2) &&
                         make_map(&c->tm_w2, c->wt + L.w2, I, E * H, L.w2_pitch, 128, 256)) &&
              make_map(&c->tm_l2out, c->ws + L.l2_out, H, Pm, H * 2, 64, 32, CU_TENSOR_MAP_DATA_TYPE_UINT16) &&
              make_map(&c->tm_acts, c->ws + L.l2_acts, I, Pm, L.acts_pitch, 64, 32, CU_TENSOR_MAP_DATA_TYPE_UINT8,
                       CU_TENSOR_MAP_SWIZZLE_64B);
    for (int i = 0; ok && i < 3; ++i)
        ok = make_map(&c->tm_l2a.box[i], c->ws + L.l2_acts, I, Pm, L.acts_pitch, 128, 32u << i) &&
             make_map(&c->tm_pool.box[i], c->ws + L.pool, H, Pm, L.pool_pitch, 128, 32u << i);
    if (!ok) {
        free(c);
        return MOE_ERR_CUDA;
    }
    // A operand of the L1 GEMM: MOE_L1_A=gather|pool overrides the automatic choice
    c->l1_a_mode = 0;
    if (const char *m = getenv("MOE_L1_A")) {
        if (!strcmp(m, "gather")) c->l1_a_mode = 1;
        if (!strcmp(m, "pool")) c->l1_a_mode = 2;
    }
    // L1 on CTA pairs: MOE_L1_PAIR=1|0 overrides the automatic choice
    c->l1_pair_mode = 0;
    if (const char *m = getenv("MOE_L1_PAIR")) c->l1_pair_mode = (m[0] == '1') ? 1 : 2;
    // both FP8 GEMMs in one launch, L2 tiles waiting per M block on L1's
    // arrival counters: MOE_FUSED=1 (off by default)
    const char *fz = getenv("MOE_FUSED");
    c->fused = fz && fz[0] == '1';
    // the two GEMMs at the same time on disjoint CTA sets of one launch:
    // MOE_SPLIT=1 (off by default); MOE_SPLIT_L1_SMS sets the L1 share, by
    // default in proportion to the GEMMs' promotion work (L1: one FP32 pass
    // per 128-K block over 2I columns, L2: two per 128-K block over H, so
    // about 2 : 1.4 for equal H and I)
    const char *sp = getenv("MOE_SPLIT");
    c->split_l1 = 0;
    if (sp && sp[0] == '1') {
        const double w1 = 2.0 * cfg->inter * cfg->hidden, w2 = 1.4 * cfg->hidden * (double)cfg->inter;
        int n1 = (int)(c->num_sms * w1 / (w1 + w2) + 0.5);
        if (const char *ns = getenv("MOE_SPLIT_L1_SMS")) n1 = atoi(ns);
        c->split_l1 = std::max(1, std::min(c->num_sms - 1, n1));
    }
    // zero the error block and the dispatch tables (a first forward that
    // stops early must not leave later steps uninitialised tables)
    if (cudaMemset(c->ws + c->L.err, 0, sizeof(int) * kErrWords) != cudaSuccess ||
        cudaMemset(c->ws + c->L.count, 0, c->L.pool - c->L.count) != cudaSuccess) {
        free(c);
        return MOE_ERR_CUDA;
    }
    *out = c;
    return MOE_OK;
}

int moe_transform_weights(moe_ctx *c, const void *w1, const void *w1_sf, const void *w2,
                          const void *w2_sf, void *stream) {
    if (!c || !w1 || !w1_sf || !w2 || !w2_sf) return MOE_ERR_INVALID_ARG;
    if (!aligned(w1, 16) || !aligned(w2, 16) || !aligned(w1_sf, 4) || !aligned(w2_sf, 4))
        return MOE_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const moe_config &g = c->cfg;
    const size_t E = g.num_experts, H = g.hidden, I = g.inter;
    if (g.wfmt == MOE_W_FP4_E2M1_UE8M0_32) {
        if (!aligned(w1, 32) || !aligned(w2, 32) || !aligned(w1_sf, 4) || !aligned(w2_sf, 4))
            return MOE_ERR_INVALID_ARG;
        launch_interleave_rows(static_cast<const uint8_t *>(w1), c->wt_at<uint8_t>(c->L.w1i), (int)E,
                               (int)I, (int)(H / 2), (int)c->L.w1_pitch, s);
        launch_interleave_rows(static_cast<const uint8_t *>(w1_sf), c->wt_at<uint8_t>(c->L.w1i_sf), (int)E,
                               (int)I, (int)(H / 32), (int)(H / 32), s);
        if (cudaMemcpy2DAsync(c->wt + c->L.w2, c->L.w2_pitch, w2, I / 2, I / 2, E * H,
                              cudaMemcpyDeviceToDevice, s) != cudaSuccess ||
            cudaMemcpyAsync(c->wt + c->L.w2_sf, w2_sf, E * H * I / 32, cudaMemcpyDeviceToDevice, s) !=
                cudaSuccess)
            return MOE_ERR_CUDA;
        if (cudaGetLastError() != cudaSuccess) return MOE_ERR_CUDA;
        c->weights_ready = true;
        return MOE_OK;
    }
    launch_transform_w1(static_cast<const uint8_t *>(w1), static_cast<const float *>(w1_sf),
                        c->wt_at<uint8_t>(c->L.w1i), (int)c->L.w1_pitch, c->wt_at<float2>(c->L.w1i_sf),
                        (int)E, (int)H, (int)I, s);
    if (cudaMemcpy2DAsync(c->wt + c->L.w2, c->L.w2_pitch, w2, I, I, E * H, cudaMemcpyDeviceToDevice, s) !=
        cudaSuccess)
        return MOE_ERR_CUDA;
    if (cudaMemcpyAsync(c->wt + c->L.w2_sf, w2_sf, 4 * E * (H / 128) * (I / 128),
                        cudaMemcpyDeviceToDevice, s) != cudaSuccess)
        return MOE_ERR_CUDA;
    if (cudaGetLastError() != cudaSuccess) return MOE_ERR_CUDA;
    c->weights_ready = true;
    return MOE_OK;
}

static int forward_launches(moe_ctx *c, int T, const void *x, const void *x_sf, const int32_t *topk_idx,
                            const float *topk_weights, void *y, int32_t *stats, cudaStream_t s);

int moe_forward(moe_ctx *c, int T, const void *x, const void *x_sf, const int32_t *topk_idx,
                const float *topk_weights, void *y, int32_t *stats, void *stream) {
    if (!c) return MOE_ERR_INVALID_ARG;
    const moe_config &g = c->cfg;
    if (T < 0 || T > g.max_tokens) return MOE_ERR_INVALID_ARG;
    if (!c->weights_ready) return MOE_ERR_NOT_READY;
    if (T == 0) return MOE_OK;
    if (!x || !x_sf || !topk_idx || !topk_weights || !y) return MOE_ERR_INVALID_ARG;
    if (!aligned(x, 16) || !aligned(y, 16) || !aligned(x_sf, 4) || !aligned(topk_idx, 4) ||
        !aligned(topk_weights, 4) || (stats && !aligned(stats, 4)))
        return MOE_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const Layout &L = c->L;
    // timeout-path test hook: words 1-2 of the error block for this forward only
    const bool test = c->test_armed;
    c->test_armed = false;
    if (test && cudaMemcpyAsync(c->ws + L.err + sizeof(int), c->test_hook, 2 * sizeof(int),
                                cudaMemcpyHostToDevice, s) != cudaSuccess)
        return MOE_ERR_CUDA;
    const int rc = forward_launches(c, T, x, x_sf, topk_idx, topk_weights, y, stats, s);
    if (test && cudaMemsetAsync(c->ws + L.err + sizeof(int), 0, 2 * sizeof(int), s) != cudaSuccess)
        return MOE_ERR_CUDA;
    return rc;
}

static int forward_launches(moe_ctx *c, int T, const void *x, const void *x_sf, const int32_t *topk_idx,
                            const float *topk_weights, void *y, int32_t *stats, cudaStream_t s) {
    const moe_config &g = c->cfg;
    const int E = g.num_experts, H = g.hidden, I = g.inter, k = g.topk;
    const int Pm = g.max_tokens * k;
    const Layout &L = c->L;
    DispatchOut o;
    o.count = c->w<int32_t>(L.count);
    o.offset = c->w<int32_t>(L.offset);
    o.mb_prefix = c->w<int32_t>(L.mb_prefix);
    o.mblk_expert = c->w<int32_t>(L.mblk_expert);
    o.mb2_prefix = c->w<int32_t>(L.mb2_prefix);
    o.mblk2_expert = c->w<int32_t>(L.mblk2_expert);
    o.gather = c->w<int32_t>(L.gather);
    o.pair_pool = c->w<int32_t>(L.pair_pool);
    o.stats = stats;
    o.err = c->w<int>(L.err);
    cudaEvent_t *ev = (c->prof_ev && c->prof_n < c->prof_max) ? c->prof_ev + 5 * c->prof_n++ : nullptr;
    if (ev) cudaEventRecord(ev[0], s);
    // A operand: gather token rows in the L1 producer (tile::gather4) when the
    // M blocks are sparse, else copy them once into the pool
    const bool gather_a = c->l1_a_mode ? c->l1_a_mode == 1 : (long long)T * k <= 4LL * E;
    AMaps tm_x;
    if (gather_a) {
        if (!make_map(&tm_x.box[0], x, (uint64_t)H, (uint64_t)T, (uint64_t)H, 128, 1)) return MOE_ERR_CUDA;
        tm_x.box[1] = tm_x.box[2] = tm_x.box[0];
    }
    L1Params p1;
    p1.gather = o.gather;
    p1.offset = o.offset;
    p1.mb_prefix = o.mb_prefix;
    p1.mblk_expert = o.mblk_expert;
    p1.mb2_prefix = o.mb2_prefix;
    p1.mblk2_expert = o.mblk2_expert;
    p1.x_sf = static_cast<const float *>(x_sf);
    p1.topk_w = topk_weights;
    p1.w1_sf = c->wt_at<float2>(L.w1i_sf);
    p1.l2_acts = c->w<uint8_t>(L.l2_acts);
    p1.acts_pitch = (int)L.acts_pitch;
    p1.l2_sf = c->w<float>(L.l2_sf);
    p1.err = o.err;
    p1.H = H;
    p1.I = I;
    p1.E = E;
    p1.k = k;
    p1.Pmax = Pm;
    p1.clamp = g.act_clamp;
    // CTA pairs only on request for now (MOE_L1_PAIR=1): single CTAs are
    // faster end to end on every measured workload
    const bool pair = c->l1_pair_mode == 1 && H % 256 == 0;

    L2Params p2;
    p2.offset = o.offset;
    p2.mb_prefix = o.mb_prefix;
    p2.mblk_expert = o.mblk_expert;
    p2.l2_sf = p1.l2_sf;
    p2.w2_sf = c->wt_at<float>(L.w2_sf);
    p2.l2_out = c->w<uint16_t>(L.l2_out);
    p2.err = o.err;
    p2.H = H;
    p2.I = I;
    p2.E = E;
    p2.Pmax = Pm;

    // the whole FP8 forward in one cooperative launch (MOE_FUSED=1); without
    // room for every CTA at once it does not launch and the separate kernels
    // below run instead.  Its time goes to the L1 stage of the profile.
    if (c->fused && !pair && g.wfmt == MOE_W_FP8_BLK128) {
        int *ready = c->w<int>(L.ready);
        const size_t ready_bytes = 4 * ((size_t)Pm / kBM + E + 1);
        // the ready counters, and the grid-barrier counter with the forward's
        // abort word (error block words 3 and 4)
        if (cudaMemsetAsync(ready, 0, ready_bytes, s) != cudaSuccess ||
            cudaMemsetAsync(o.err + 3, 0, 2 * sizeof(int), s) != cudaSuccess)
            return MOE_ERR_CUDA;
        FusedParams f;
        f.topk_idx = topk_idx;
        f.T = T;
        f.k = k;
        f.d = o;
        f.d.mb2_prefix = nullptr;
        f.d.mblk2_expert = nullptr;
        f.cta_cnt = c->w<int32_t>(L.dcnt);
        f.bar = o.err + 3;
        f.x = static_cast<const uint8_t *>(x);
        f.pool = c->w<uint8_t>(L.pool);
        f.pool_pitch = (int)L.pool_pitch;
        f.y = static_cast<uint16_t *>(y);
        if (ev) cudaEventRecord(ev[1], s);
        if (launch_fused(gather_a ? tm_x : c->tm_pool, c->tm_w1, c->tm_acts, c->tm_l2a, c->tm_w2, c->tm_l2out, p1, p2,
                         ready, f, g.fast_math, gather_a, c->num_sms, s) == cudaSuccess) {
            if (ev) {
                cudaEventRecord(ev[2], s);
                cudaEventRecord(ev[3], s);
                cudaEventRecord(ev[4], s);
            }
            if (cudaGetLastError() != cudaSuccess) return MOE_ERR_CUDA;
            c->last_T = T;
            return MOE_OK;
        }
        (void)cudaGetLastError();
    }
    // large batches: the dispatch over several CTAs (one per 1024 pairs, at
    // most one per SM); the single-CTA kernel if that launch is refused
    bool dispatched = false;
    if ((long long)T * k >= kDispatchMcMinPairs) {
        const int ctas = std::min(std::min(c->num_sms, kDispatchMcMaxCtas), (T * k + 1023) / 1024);
        dispatched = launch_dispatch_mc(topk_idx, T, k, E, o, c->w<int32_t>(L.dcnt), c->w<int>(L.err) + 3,
                                        ctas, s) == cudaSuccess;
        if (!dispatched) (void)cudaGetLastError();
    }
    if (!dispatched && launch_dispatch(topk_idx, T, k, E, o, s) != cudaSuccess) return MOE_ERR_CUDA;
    if (ev) cudaEventRecord(ev[1], s);
    if (!gather_a)
        launch_pool_gather(static_cast<const uint8_t *>(x), o.gather, o.offset + E, k, H, T * k,
                           c->w<uint8_t>(L.pool), (int)L.pool_pitch, o.err, s);

    if (g.wfmt == MOE_W_FP4_E2M1_UE8M0_32) {
        Fp4Params f;
        f.gather = o.gather;
        f.offset = o.offset;
        f.mb_prefix = o.mb_prefix;
        f.mblk_expert = o.mblk_expert;
        f.a_sf = static_cast<const uint8_t *>(x_sf);
        f.b_sf = c->wt_at<uint8_t>(L.w1i_sf);
        f.topk_w = topk_weights;
        f.l2_acts = c->w<uint8_t>(L.l2_acts);
        f.acts_pitch = (int)L.acts_pitch;
        f.l2_sf = c->w<uint8_t>(L.l2_sf);
        f.l2_out = c->w<uint16_t>(L.l2_out);
        f.err = o.err;
        f.H = H;
        f.I = I;
        f.E = E;
        f.k = k;
        f.Pmax = Pm;
        f.clamp = g.act_clamp;
        launch_fp4_l1(gather_a ? tm_x : c->tm_pool, c->tm_w1, f, g.fast_math, gather_a, c->num_sms, s);
        if (ev) cudaEventRecord(ev[2], s);
        f.a_sf = f.l2_sf;
        f.b_sf = c->wt_at<uint8_t>(L.w2_sf);
        launch_fp4_l2(c->tm_l2a, c->tm_w2, c->tm_l2out, f, c->num_sms, s);
        if (ev) cudaEventRecord(ev[3], s);
        launch_combine(f.l2_out, o.pair_pool, T, k, H, static_cast<uint16_t *>(y), o.err, s);
        if (ev) cudaEventRecord(ev[4], s);
        if (cudaGetLastError() != cudaSuccess) return MOE_ERR_CUDA;
        c->last_T = T;
        return MOE_OK;
    }

    bool fused_done = false;
    if (c->split_l1 > 0 && !pair) {
        // both GEMMs at once on disjoint CTA sets; without room for every CTA
        // at once it does not launch and the two kernels below run instead
        int *ready = c->w<int>(L.ready);
        const size_t ready_bytes = 4 * ((size_t)Pm / kBM + E + 1);
        if (cudaMemsetAsync(ready, 0, ready_bytes, s) != cudaSuccess) return MOE_ERR_CUDA;
        fused_done = launch_split(gather_a ? tm_x : c->tm_pool, c->tm_w1, c->tm_acts, c->tm_l2a, c->tm_w2, c->tm_l2out,
                                  p1, p2, ready, c->split_l1, g.fast_math, gather_a, c->num_sms, s) == cudaSuccess;
        if (!fused_done) (void)cudaGetLastError();
    }
    if (!fused_done) {
        if (pair) {
            if (launch_l1_pair(gather_a ? tm_x : c->tm_pool, c->tm_pool3, c->tm_w1h, c->tm_acts, p1, g.fast_math, gather_a,
                               c->num_sms, s) != cudaSuccess)
                return MOE_ERR_CUDA;
        } else {
            launch_l1(gather_a ? tm_x : c->tm_pool, c->tm_w1, c->tm_acts, p1, g.fast_math, gather_a, c->num_sms, s);
        }
    }
    if (ev) cudaEventRecord(ev[2], s);
    if (!fused_done) launch_l2(c->tm_l2a, c->tm_w2, c->tm_l2out, p2, c->num_sms, s);
    if (ev) cudaEventRecord(ev[3], s);

    launch_combine(p2.l2_out, o.pair_pool, T, k, H, static_cast<uint16_t *>(y), o.err, s);
    if (ev) cudaEventRecord(ev[4], s);
    if (cudaGetLastError() != cudaSuccess) return MOE_ERR_CUDA;
    c->last_T = T;
    return MOE_OK;
}

// Device address of a page-locked host buffer the kernels may store to, or
// nullptr (pageable memory, no mapping, a misaligned start, or
// MOE_HOST_DIRECT=0: then the output is staged and copied back).
static void *host_y_direct(void *h_y) {
    static const bool off = [] {
        const char *e = getenv("MOE_HOST_DIRECT");
        return e && e[0] == '0';
    }();
    if (off) return nullptr;
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, h_y) != cudaSuccess) {
        cudaGetLastError();   // a pointer the runtime does not know is not an error here
        return nullptr;
    }
    if (a.type != cudaMemoryTypeHost || !a.devicePointer || (reinterpret_cast<uintptr_t>(a.devicePointer) & 15))
        return nullptr;
    return a.devicePointer;
}

int moe_forward_host(moe_ctx *c, int T, const void *h_x, const void *h_x_sf,
                     const int32_t *h_topk_idx, const float *h_topk_weights, void *h_y,
                     void *stream) {
    if (!c) return MOE_ERR_INVALID_ARG;
    const moe_config &g = c->cfg;
    if (T < 0 || T > g.max_tokens) return MOE_ERR_INVALID_ARG;
    if (!c->weights_ready) return MOE_ERR_NOT_READY;
    if (T == 0) return MOE_OK;
    if (!h_x || !h_x_sf || !h_topk_idx || !h_topk_weights || !h_y) return MOE_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const size_t H = g.hidden, k = g.topk;
    const Layout &L = c->L;
    if (cudaMemcpyAsync(c->ws + L.st_x, h_x, (size_t)T * H, cudaMemcpyHostToDevice, s) ||
        cudaMemcpyAsync(c->ws + L.st_xsf, h_x_sf, x_sf_bytes(g, T), cudaMemcpyHostToDevice, s) ||
        cudaMemcpyAsync(c->ws + L.st_idx, h_topk_idx, (size_t)T * k * 4, cudaMemcpyHostToDevice, s) ||
        cudaMemcpyAsync(c->ws + L.st_w, h_topk_weights, (size_t)T * k * 4, cudaMemcpyHostToDevice, s))
        return MOE_ERR_CUDA;
    // A page-locked h_y that the device can address (every pinned allocation
    // under unified addressing) takes the combine's stores directly, over the
    // CPU-GPU link, instead of a staging buffer and a copy back.
    void *y_direct = host_y_direct(h_y);
    int r = moe_forward(c, T, c->ws + L.st_x, c->ws + L.st_xsf, c->w<int32_t>(L.st_idx),
                        c->w<float>(L.st_w), y_direct ? y_direct : c->ws + L.st_y, nullptr, stream);
    if (r != MOE_OK) return r;
    if (!y_direct && cudaMemcpyAsync(h_y, c->ws + L.st_y, (size_t)T * H * 2, cudaMemcpyDeviceToHost, s))
        return MOE_ERR_CUDA;
    if (cudaStreamSynchronize(s)) return MOE_ERR_CUDA;
    return MOE_OK;
}

int moe_get_dispatch(moe_ctx *c, int32_t *counts, int32_t *offsets, int32_t *gather, void *stream) {
    if (!c) return MOE_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const size_t E = c->cfg.num_experts, P = (size_t)c->last_T * c->cfg.topk;
    if (counts && cudaMemcpyAsync(counts, c->ws + c->L.count, 4 * E, cudaMemcpyDeviceToDevice, s))
        return MOE_ERR_CUDA;
    if (offsets && cudaMemcpyAsync(offsets, c->ws + c->L.offset, 4 * (E + 1), cudaMemcpyDeviceToDevice, s))
        return MOE_ERR_CUDA;
    if (gather && P && cudaMemcpyAsync(gather, c->ws + c->L.gather, 4 * P, cudaMemcpyDeviceToDevice, s))
        return MOE_ERR_CUDA;
    return MOE_OK;
}

int moe_get_intermediates(moe_ctx *c, void *l2_acts, void *l2_sf, void *l2_out, void *stream) {
    if (!c) return MOE_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const size_t H = c->cfg.hidden, I = c->cfg.inter;
    const size_t P = (size_t)c->last_T * c->cfg.topk;
    if (!P) return MOE_OK;
    if (l2_acts && cudaMemcpy2DAsync(l2_acts, I, c->ws + c->L.l2_acts, c->L.acts_pitch, I, P,
                                     cudaMemcpyDeviceToDevice, s))
        return MOE_ERR_CUDA;
    if (l2_sf) {
        const cudaError_t e =
            c->cfg.wfmt == MOE_W_FP8_BLK128
                ? cudaMemcpyAsync(l2_sf, c->ws + c->L.l2_sf, P * (I / 64) * 4, cudaMemcpyDeviceToDevice, s)
                : cudaMemcpyAsync(l2_sf, c->ws + c->L.l2_sf, P * (I / 32), cudaMemcpyDeviceToDevice, s);
        if (e != cudaSuccess) return MOE_ERR_CUDA;
    }
    if (l2_out && cudaMemcpyAsync(l2_out, c->ws + c->L.l2_out, P * H * 2, cudaMemcpyDeviceToDevice, s))
        return MOE_ERR_CUDA;
    return MOE_OK;
}

static void profile_release(moe_ctx *c) {
    if (!c->prof_ev) return;
    for (int i = 0; i < 5 * c->prof_max; ++i) cudaEventDestroy(c->prof_ev[i]);
    free(c->prof_ev);
    c->prof_ev = nullptr;
    c->prof_max = c->prof_n = 0;
}

int moe_profile_begin(moe_ctx *c, int max_forwards) {
    if (!c || max_forwards < 1 || max_forwards > 100000) return MOE_ERR_INVALID_ARG;
    profile_release(c);
    c->prof_ev = static_cast<cudaEvent_t *>(calloc(5 * (size_t)max_forwards, sizeof(cudaEvent_t)));
    if (!c->prof_ev) return MOE_ERR_INVALID_ARG;
    for (int i = 0; i < 5 * max_forwards; ++i)
        if (cudaEventCreate(&c->prof_ev[i]) != cudaSuccess) {
            c->prof_max = i / 5 + 1;
            profile_release(c);
            return MOE_ERR_CUDA;
        }
    c->prof_max = max_forwards;
    c->prof_n = 0;
    return MOE_OK;
}

int moe_profile_end(moe_ctx *c, float *stage_ms, int *n_forwards) {
    if (!c || !c->prof_ev) return MOE_ERR_INVALID_ARG;
    float sum[4] = {0, 0, 0, 0};
    int rc = MOE_OK;
    for (int f = 0; f < c->prof_n && rc == MOE_OK; ++f) {
        cudaEvent_t *ev = c->prof_ev + 5 * f;
        if (cudaEventSynchronize(ev[4]) != cudaSuccess) rc = MOE_ERR_CUDA;
        for (int st = 0; st < 4 && rc == MOE_OK; ++st) {
            float ms = 0;
            if (cudaEventElapsedTime(&ms, ev[st], ev[st + 1]) != cudaSuccess) rc = MOE_ERR_CUDA;
            sum[st] += ms;
        }
    }
    if (stage_ms) memcpy(stage_ms, sum, sizeof(sum));
    if (n_forwards) *n_forwards = c->prof_n;
    profile_release(c);
    return rc;
}

int moe_test_arm_timeout(moe_ctx *c, int which, int wait_limit_us) {
    if (!c || (which != kStallL1 && which != kStallL2 && which != kStallDispatch) || wait_limit_us < 1)
        return MOE_ERR_INVALID_ARG;
    c->test_hook[0] = wait_limit_us;
    c->test_hook[1] = which;
    c->test_armed = true;
    return MOE_OK;
}

int moe_device_status(moe_ctx *c) {
    if (!c) return MOE_ERR_INVALID_ARG;
    if (cudaDeviceSynchronize() != cudaSuccess) return MOE_ERR_CUDA;
    int err = 0;
    if (cudaMemcpy(&err, c->ws + c->L.err, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess)
        return MOE_ERR_CUDA;
    if (err && cudaMemset(c->ws + c->L.err, 0, sizeof(int)) != cudaSuccess) return MOE_ERR_CUDA;
    if (err & kErrTimeout) return MOE_ERR_DEVICE_TIMEOUT;
    if (err & kErrBadExpert) return MOE_ERR_BAD_EXPERT;
    return MOE_OK;
}

const char *moe_strerror(int code) {
    switch (code) {
        case MOE_OK: return "ok";
        case MOE_ERR_INVALID_ARG: return "invalid argument";
        case MOE_ERR_UNSUPPORTED: return "unsupported shape or format";
        case MOE_ERR_CUDA: return "CUDA call failed";
        case MOE_ERR_DEVICE_TIMEOUT: return "a device-side wait timed out";
        case MOE_ERR_BAD_EXPERT: return "topk_idx holds an expert id outside [-1, E)";
        case MOE_ERR_NOT_READY: return "weights not transformed yet";
        default: return "unknown error";
    }
}

void moe_destroy(moe_ctx *c) {
    if (!c) return;
    profile_release(c);
    free(c);
}

}  // extern "C"
