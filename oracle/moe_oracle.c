/*
 * moe_oracle.c -- plain, slow CPU oracle of the MegaMoE expert layer.
 *
 * TEST INFRASTRUCTURE. Only the test suite, the smoke check and the CPU
 * baseline leg of the benchmark may load or call this library.  The product
 * path (the CUDA library under moe_expert_ffn_gb300/) never links, imports or
 * calls it, and shares no code, header, table or constant with it.
 *
 * What it computes (MegaMoE SM90 Implementation Design (Final), §3.3 "Fused
 * Kernel Pipeline" and §20.1 "Baseline": dispatch -> dequantised L1 GEMM ->
 * SwiGLU -> FP8 quantise -> dequantised L2 GEMM -> combine), written as the
 * plain definition: every dot product is a sequential double-precision sum,
 * every quantisation step is done element by element, nothing is blocked,
 * fused or reordered.
 *
 * Readings taken where the pages are silent or ambiguous (each is listed in
 * the repository's design notes as well):
 *   - L2-activation scale granularity: one float scale per token row and per
 *     64 consecutive intermediate columns (§1.1 decision 9 "Per-64 dual-half
 *     SF", §5.4, §10.1 step 6), sf = amax / 448 (§10.1 step 5).
 *   - an all-zero 64-group gets sf = 0 and codes 0 (never divides by zero).
 *   - FP8 rounding is round-to-nearest-even with saturation to +-448.
 *   - the top-k weight multiplies the SwiGLU output before quantisation
 *     (§10.1 steps 2-3).
 *   - the L2 output of each (token, slot) pair is rounded to BF16 before the
 *     combine (§11.1 step 1), and the combine sums the active slots in
 *     ascending slot order in FP32, then rounds to BF16 (§11.2).
 *   - dispatch order inside one expert is the stable (token, slot) order.
 *   - topk_idx == -1 marks an inactive slot; any other id outside [0, E) is
 *     an error.
 *   - FP4-weight configuration (PR357 Green-Context Split MegaMoE code review,
 *     §1 and §3.2; design §2.1 "Scale Factor Format"): weights are E2M1 packed
 *     two per byte along K, low nibble = even k, with one UE8M0 scale per 32
 *     K; activations are FP8 E4M3 with one UE8M0 scale per 32 K; the L2
 *     activations are requantised per 32 columns with a UE8M0 scale
 *     2^ceil(log2(amax/448)) (exponent clamped to [-127, 127]).
 *
 * Parity pins: every exported function is checked by tests/test_oracle_*.py
 * against an independent fact (library casts, brute force, closed forms,
 * invariants).  No function here is "parity unpinned".
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_OK 0
#define ORC_EINVAL (-1)
#define ORC_EBADEXPERT (-5)

/* ------------------------------------------------------------------------ */
/* Number formats, written from their definitions.                          */
/* ------------------------------------------------------------------------ */

/* OCP FP8 E4M3 ("e4m3fn"): sign, 4 exponent bits (bias 7), 3 mantissa bits,
 * no infinities, S.1111.111 is NaN, largest finite magnitude 448. */
double orc_e4m3_decode(uint8_t code)
{
    int s = code >> 7, e = (code >> 3) & 15, m = code & 7;
    double v;
    if (e == 15 && m == 7) return NAN;
    if (e == 0) v = ldexp((double)m, -9);            /* (m/8) * 2^-6 */
    else v = ldexp((double)(8 + m), e - 10);         /* (1+m/8) * 2^(e-7) */
    return s ? -v : v;
}

/* float -> E4M3, round to nearest (ties to even code), saturating finite
 * values and infinities to +-448, NaN -> 0x7F.  The nearest code is found
 * by looking at every non-negative finite code. */
uint8_t orc_e4m3_encode(float f)
{
    double a;
    int best = 0, c;
    double best_err;
    uint8_t sign;
    if (isnan(f)) return 0x7F;
    sign = signbit(f) ? 0x80 : 0x00;
    a = fabs((double)f);
    if (a >= 448.0) return (uint8_t)(sign | 0x7E);
    best_err = a;                                     /* code 0 = 0.0 */
    for (c = 1; c <= 0x7E; c++) {
        double err = fabs(orc_e4m3_decode((uint8_t)c) - a);
        if (err < best_err || (err == best_err && (c & 1) == 0 && (best & 1) == 1)) {
            best = c;
            best_err = err;
        }
    }
    return (uint8_t)(sign | best);
}

/* BF16: the upper 16 bits of an IEEE binary32, rounded to nearest even. */
uint16_t orc_bf16_encode(float f)
{
    uint32_t u;
    memcpy(&u, &f, 4);
    if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu)) return 0x7FC0;
    u += 0x7FFFu + ((u >> 16) & 1u);
    return (uint16_t)(u >> 16);
}

float orc_bf16_decode(uint16_t h)
{
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}

/* OCP MX FP4 E2M1: sign, 2 exponent bits (bias 1), 1 mantissa bit. */
double orc_e2m1_decode(uint8_t nib)
{
    int s = (nib >> 3) & 1, e = (nib >> 1) & 3, m = nib & 1;
    double v = (e == 0) ? 0.5 * m : ldexp(1.0 + 0.5 * m, e - 1);
    return s ? -v : v;
}

/* float -> E2M1, nearest with ties to even code, saturating at +-6. */
uint8_t orc_e2m1_encode(float f)
{
    double a = fabs((double)f), best_err;
    int best = 0, c;
    uint8_t sign = signbit(f) ? 8 : 0;
    if (isnan(f)) return 0;
    best_err = a;
    for (c = 1; c < 8; c++) {
        double err = fabs(orc_e2m1_decode((uint8_t)c) - a);
        if (err < best_err || (err == best_err && (c & 1) == 0 && (best & 1) == 1)) {
            best = c;
            best_err = err;
        }
    }
    return (uint8_t)(sign | best);
}

/* UE8M0: an unsigned power of two 2^(code-127); code 255 is NaN. */
double orc_ue8m0_decode(uint8_t code)
{
    if (code == 255) return NAN;
    return ldexp(1.0, (int)code - 127);
}

/* Smallest power of two 2^e with amax / qmax <= 2^e (the ratio is taken in
 * binary32), e clamped to [-127, 127]; returns the UE8M0 code e + 127. */
uint8_t orc_ue8m0_for_amax(float amax, float qmax)
{
    float r = amax / qmax;
    int ex, e;
    double frac;
    if (!(r > 0.0f)) return 0;                        /* zero group: 2^-127 */
    frac = frexp((double)r, &ex);                     /* r = frac * 2^ex, frac in [0.5,1) */
    e = (frac == 0.5) ? ex - 1 : ex;
    if (e < -127) e = -127;
    if (e > 127) e = 127;
    return (uint8_t)(e + 127);
}

/* ------------------------------------------------------------------------ */
/* Quantisers of the L1 output (design §10.1 steps 4-6).                     */
/* ------------------------------------------------------------------------ */

/* One FP8 group with a float scale: sf = amax/448 in binary32, q = e4m3(a/sf)
 * with a binary32 division.  Returns sf. */
float orc_quant_fp8_group(const float *a, int n, uint8_t *q)
{
    float amax = 0.0f, sf;
    int i;
    for (i = 0; i < n; i++) {
        float v = fabsf(a[i]);
        if (v > amax) amax = v;
    }
    sf = amax / 448.0f;
    for (i = 0; i < n; i++) q[i] = (sf == 0.0f) ? 0 : orc_e4m3_encode(a[i] / sf);
    return sf;
}

/* One FP8 group with a UE8M0 scale (FP4-weight configuration).  Returns the
 * UE8M0 code. */
uint8_t orc_quant_fp8_ue8m0_group(const float *a, int n, uint8_t *q)
{
    float amax = 0.0f, sf;
    uint8_t code;
    int i;
    for (i = 0; i < n; i++) {
        float v = fabsf(a[i]);
        if (v > amax) amax = v;
    }
    code = orc_ue8m0_for_amax(amax, 448.0f);
    sf = (float)orc_ue8m0_decode(code);
    for (i = 0; i < n; i++) q[i] = (amax == 0.0f) ? 0 : orc_e4m3_encode(a[i] / sf);
    return code;
}

/* ------------------------------------------------------------------------ */
/* Dispatch (design §9.2, PR357 review §6.1): per-expert count, exclusive     */
/* prefix and the gather map of (token, slot) pairs in stable order.          */
/* ------------------------------------------------------------------------ */

int orc_dispatch(int T, int k, int E, const int32_t *topk_idx,
                 int32_t *count, int32_t *offset, int32_t *gather)
{
    int t, j, e, status = ORC_OK;
    int32_t *fill;
    if (T < 0 || k <= 0 || E <= 0) return ORC_EINVAL;
    for (e = 0; e < E; e++) count[e] = 0;
    for (t = 0; t < T; t++)
        for (j = 0; j < k; j++) {
            int32_t id = topk_idx[(size_t)t * k + j];
            if (id >= 0 && id < E) count[id]++;
            else if (id != -1) status = ORC_EBADEXPERT;
        }
    offset[0] = 0;
    for (e = 0; e < E; e++) offset[e + 1] = offset[e] + count[e];
    fill = (int32_t *)calloc((size_t)E, sizeof(int32_t));
    if (!fill) return ORC_EINVAL;
    for (t = 0; t < T; t++)
        for (j = 0; j < k; j++) {
            int32_t id = topk_idx[(size_t)t * k + j];
            if (id >= 0 && id < E) gather[offset[id] + fill[id]++] = t * k + j;
        }
    free(fill);
    return status;
}

/* ------------------------------------------------------------------------ */
/* The expert layer.                                                          */
/* ------------------------------------------------------------------------ */

typedef struct {
    int T, H, I, E, k;
    int wfmt;          /* 0: FP8 weights, 128x128 f32 scales, acts 1x128 f32 scales
                          1: FP4 E2M1 weights, 1x32 UE8M0 scales, acts FP8 1x32 UE8M0 */
    float act_clamp;   /* symmetric clamp of gate and up; +inf = off */
} orc_cfg;

typedef struct {
    const orc_cfg *c;
    const uint8_t *x;      /* [T,H] e4m3 */
    const void *x_sf;      /* wfmt 0: f32 [T,H/128]; wfmt 1: u8 [T,H/32] */
    const uint8_t *w1;     /* wfmt 0: e4m3 [E,2I,H]; wfmt 1: packed e2m1 [E,2I,H/2] */
    const void *w1_sf;     /* wfmt 0: f32 [E,2I/128,H/128]; wfmt 1: u8 [E,2I,H/32] */
    const uint8_t *w2;     /* wfmt 0: e4m3 [E,H,I]; wfmt 1: packed e2m1 [E,H,I/2] */
    const void *w2_sf;     /* wfmt 0: f32 [E,H/128,I/128]; wfmt 1: u8 [E,H,I/32] */
} orc_layer;

/* Dequantised weight element W[e][n][kk] of a matrix with N rows and K
 * columns (W1: N=2I, K=H; W2: N=H, K=I). */
static double weight_at(const orc_layer *L, const uint8_t *w, const void *sf,
                        int N, int K, int e, int n, int kk)
{
    if (L->c->wfmt == 0) {
        const float *s = (const float *)sf;
        double v = orc_e4m3_decode(w[((size_t)e * N + n) * K + kk]);
        return v * (double)s[((size_t)e * (N / 128) + n / 128) * (K / 128) + kk / 128];
    } else {
        const uint8_t *s = (const uint8_t *)sf;
        uint8_t byte = w[((size_t)e * N + n) * (K / 2) + kk / 2];
        uint8_t nib = (kk & 1) ? (uint8_t)(byte >> 4) : (uint8_t)(byte & 15);
        return orc_e2m1_decode(nib) * orc_ue8m0_decode(s[((size_t)e * N + n) * (K / 32) + kk / 32]);
    }
}

static double act_at(const orc_layer *L, int t, int h)
{
    int H = L->c->H;
    double v = orc_e4m3_decode(L->x[(size_t)t * H + h]);
    if (L->c->wfmt == 0)
        return v * (double)((const float *)L->x_sf)[(size_t)t * (H / 128) + h / 128];
    return v * orc_ue8m0_decode(((const uint8_t *)L->x_sf)[(size_t)t * (H / 32) + h / 32]);
}

/* L1 GEMM + SwiGLU + top-k weight for one (token, expert) pair:
 * a[i] = f32( silu(clamp(g_i)) * clamp(u_i) * w ) with g rows [0,I) and up
 * rows [I,2I) of the canonical W1 (design §10.1 steps 1-3, §15.1). */
static void pair_l1(const orc_layer *L, int t, int e, float w, double *xd, float *a)
{
    const orc_cfg *c = L->c;
    int H = c->H, I = c->I, h, i;
    double clampv = (double)c->act_clamp;
    for (h = 0; h < H; h++) xd[h] = act_at(L, t, h);
    for (i = 0; i < I; i++) {
        double g = 0.0, u = 0.0, silu;
        for (h = 0; h < H; h++) g += xd[h] * weight_at(L, L->w1, L->w1_sf, 2 * I, H, e, i, h);
        for (h = 0; h < H; h++) u += xd[h] * weight_at(L, L->w1, L->w1_sf, 2 * I, H, e, I + i, h);
        if (g > clampv) g = clampv;
        if (g < -clampv) g = -clampv;
        if (u > clampv) u = clampv;
        if (u < -clampv) u = -clampv;
        silu = g / (1.0 + exp(-g));
        a[i] = (float)(silu * u * (double)w);
    }
}

/* Requantise the L1 output: FP8 codes q[I] and dequantised values ad[I].
 * Scales: wfmt 0 -> f32 per 64 columns (sf_out[I/64]); wfmt 1 -> UE8M0 per 32
 * columns (code stored as float in sf_out[I/32]). */
static void pair_requant(const orc_cfg *c, const float *a, uint8_t *q, float *sf_out, double *ad)
{
    int I = c->I, g, i;
    if (c->wfmt == 0) {
        for (g = 0; g < I / 64; g++) {
            float sf = orc_quant_fp8_group(a + g * 64, 64, q + g * 64);
            sf_out[g] = sf;
            for (i = g * 64; i < g * 64 + 64; i++) ad[i] = orc_e4m3_decode(q[i]) * (double)sf;
        }
    } else {
        for (g = 0; g < I / 32; g++) {
            uint8_t code = orc_quant_fp8_ue8m0_group(a + g * 32, 32, q + g * 32);
            double sf = orc_ue8m0_decode(code);
            sf_out[g] = (float)code;
            for (i = g * 32; i < g * 32 + 32; i++) ad[i] = orc_e4m3_decode(q[i]) * sf;
        }
    }
}

/* L2 GEMM for one pair: o[h] = sum_i ad[i] * W2[e][h][i] in double. */
static void pair_l2(const orc_layer *L, int e, const double *ad, double *o)
{
    int H = L->c->H, I = L->c->I, h, i;
    for (h = 0; h < H; h++) {
        double s = 0.0;
        for (i = 0; i < I; i++) s += ad[i] * weight_at(L, L->w2, L->w2_sf, H, I, e, h, i);
        o[h] = s;
    }
}

static int check_cfg(const orc_cfg *c)
{
    if (!c || c->T < 0 || c->H <= 0 || c->I <= 0 || c->E <= 0 || c->k <= 0) return ORC_EINVAL;
    if (c->H % 128 || c->I % 128) return ORC_EINVAL;
    if (c->wfmt != 0 && c->wfmt != 1) return ORC_EINVAL;
    return ORC_OK;
}

/* Output rows y[s][H] (BF16 bits) of the selected tokens sel[s]. */
int orc_forward(const orc_cfg *c, const uint8_t *x, const void *x_sf,
                const int32_t *topk_idx, const float *topk_w,
                const uint8_t *w1, const void *w1_sf, const uint8_t *w2, const void *w2_sf,
                int n_sel, const int32_t *sel, uint16_t *y)
{
    orc_layer L;
    int s, status;
    status = check_cfg(c);
    if (status) return status;
    L.c = c; L.x = x; L.x_sf = x_sf; L.w1 = w1; L.w1_sf = w1_sf; L.w2 = w2; L.w2_sf = w2_sf;
    for (s = 0; s < n_sel; s++) {
        int t = sel[s], j;
        for (j = 0; j < c->k; j++) {
            int32_t id = topk_idx[(size_t)t * c->k + j];
            if (id != -1 && (id < 0 || id >= c->E)) status = ORC_EBADEXPERT;
        }
        if (t < 0 || t >= c->T) return ORC_EINVAL;
    }
#pragma omp parallel for schedule(dynamic, 1)
    for (s = 0; s < n_sel; s++) {
        int H = c->H, I = c->I, t = sel[s], j, h;
        double *xd = (double *)malloc(sizeof(double) * H);
        float *a = (float *)malloc(sizeof(float) * I);
        uint8_t *q = (uint8_t *)malloc(I);
        float *sf = (float *)malloc(sizeof(float) * (I / 32));
        double *ad = (double *)malloc(sizeof(double) * I);
        double *o = (double *)malloc(sizeof(double) * H);
        float *acc = (float *)malloc(sizeof(float) * H);
        for (h = 0; h < H; h++) acc[h] = 0.0f;
        for (j = 0; j < c->k; j++) {
            int32_t e = topk_idx[(size_t)t * c->k + j];
            if (e < 0 || e >= c->E) continue;
            pair_l1(&L, t, e, topk_w[(size_t)t * c->k + j], xd, a);
            pair_requant(c, a, q, sf, ad);
            pair_l2(&L, e, ad, o);
            for (h = 0; h < H; h++) acc[h] += orc_bf16_decode(orc_bf16_encode((float)o[h]));
        }
        for (h = 0; h < H; h++) y[(size_t)s * H + h] = orc_bf16_encode(acc[h]);
        free(xd); free(a); free(q); free(sf); free(ad); free(o); free(acc);
    }
    return status;
}

/* Intermediates of one (token, expert, weight) pair, for stage-by-stage
 * checks: a[I] (SwiGLU * weight, binary32), q[I] (FP8 codes), sf[I/64] or
 * [I/32] (scales, UE8M0 codes as floats for wfmt 1), o[H] (L2 output, double),
 * ob[H] (L2 output rounded to BF16, bits). */
int orc_pair(const orc_cfg *c, const uint8_t *x, const void *x_sf,
             const uint8_t *w1, const void *w1_sf, const uint8_t *w2, const void *w2_sf,
             int t, int e, float w, float *a, uint8_t *q, float *sf, double *o, uint16_t *ob)
{
    orc_layer L;
    double *xd, *ad;
    int h, status = check_cfg(c);
    if (status) return status;
    if (t < 0 || t >= c->T || e < 0 || e >= c->E) return ORC_EINVAL;
    L.c = c; L.x = x; L.x_sf = x_sf; L.w1 = w1; L.w1_sf = w1_sf; L.w2 = w2; L.w2_sf = w2_sf;
    xd = (double *)malloc(sizeof(double) * c->H);
    ad = (double *)malloc(sizeof(double) * c->I);
    pair_l1(&L, t, e, w, xd, a);
    pair_requant(c, a, q, sf, ad);
    pair_l2(&L, e, ad, o);
    for (h = 0; h < c->H; h++) ob[h] = orc_bf16_encode((float)o[h]);
    free(xd);
    free(ad);
    return ORC_OK;
}

int orc_num_threads(void)
{
#ifdef _OPENMP
    extern int omp_get_max_threads(void);
    return omp_get_max_threads();
#else
    return 1;
#endif
}
