/*
 * moe.h -- C ABI of the GB300 (sm_103a) MegaMoE expert layer.
 *
 * One call of moe_forward runs, on the caller's CUDA stream, the whole expert
 * layer of a Mixture-of-Experts block on one GPU:
 *
 *   1. dispatch: per-expert counts, exclusive prefix, stable gather map
 *      (MegaMoE SM90 Implementation Design (Final), §9.2; PR357 Green-Context
 *      Split MegaMoE code review, §6.1);
 *   2. L1 grouped GEMM x . W1^T with block scales applied per 128-K block
 *      (design §5.2-§5.3);
 *   3. SwiGLU silu(gate) * up, times the top-k weight (design §10.1 steps 1-3);
 *   4. per-row, per-64-column FP8 E4M3 requantisation, sf = amax / 448
 *      (design §10.1 steps 4-6, §1.1 decision 9);
 *   5. L2 grouped GEMM with the two per-64 activation scales of every
 *      128-K block (design §5.4);
 *   6. BF16 rounding of each (token, slot) output (design §11.1);
 *   7. top-k combine: FP32 sum over active slots in slot order, BF16 y
 *      (design §11.2; PR357 review §6.3 "K3 combine_reduce").
 *
 * Pointers: every buffer argument of moe_create / moe_transform_weights /
 * moe_forward / moe_get_* is DEVICE memory owned by the caller, except the
 * h_* arguments of moe_forward_host, which are HOST memory.  The library never
 * allocates device memory: the caller passes a workspace of
 * moe_workspace_bytes() bytes and a weight store of moe_weight_bytes() bytes,
 * both 256-byte aligned, which must outlive the context.  A moe_ctx holds
 * host state only.
 *
 * Streams: `stream` is a cudaStream_t (NULL = the legacy default stream).
 * Calls are stream-ordered and asynchronous unless stated otherwise; two
 * forwards of one context must not run concurrently (they share the
 * workspace).  Back-to-back forwards need no reset by the caller.
 *
 * Errors: every int-returning call returns MOE_OK (0) or a negative MOE_ERR_*
 * code; nothing is thrown across the ABI.  Argument and shape errors are
 * detected on the host before anything is launched.  Faults found on the
 * device (an expert id outside [-1, E), a pipeline wait that timed out) are
 * recorded in a device error word that moe_device_status() reads.
 */
#ifndef MOE_GB300_H
#define MOE_GB300_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define MOE_API __attribute__((visibility("default")))
#else
#define MOE_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

#define MOE_OK 0
#define MOE_ERR_INVALID_ARG (-1)    /* null pointer, bad size, misaligned buffer */
#define MOE_ERR_UNSUPPORTED (-2)    /* shape or format this library does not run */
#define MOE_ERR_CUDA (-3)           /* a CUDA runtime/driver call failed */
#define MOE_ERR_DEVICE_TIMEOUT (-4) /* a bounded device-side wait gave up */
#define MOE_ERR_BAD_EXPERT (-5)     /* topk_idx held an id outside [-1, E) */
#define MOE_ERR_NOT_READY (-6)      /* moe_forward before moe_transform_weights */

typedef struct moe_ctx moe_ctx;

/* Weight formats.
 * MOE_W_FP8_BLK128: W1/W2 FP8 E4M3 with one f32 scale per 128x128 block,
 *   activations x FP8 E4M3 with one f32 scale per 1x128 (recipe (1,1,128),
 *   design §16.1 and §15.2).
 * MOE_W_FP4_E2M1_UE8M0_32: W1/W2 FP4 E2M1 (two codes per byte, low nibble =
 *   even k) with one UE8M0 scale per 1x32; activations FP8 E4M3 with one UE8M0
 *   scale per 1x32; the L2 activations are requantised per 1x32 with UE8M0
 *   scales 2^ceil(log2(amax/448)) (design §2.1, PR357 review §1, §6.1). */
typedef enum { MOE_W_FP8_BLK128 = 0, MOE_W_FP4_E2M1_UE8M0_32 = 1 } moe_wfmt;

typedef struct {
    int max_tokens;   /* T_max: largest num_tokens a forward may pass (>= 1) */
    int hidden;       /* H, multiple of 128 */
    int inter;        /* I (intermediate size per expert), multiple of 128 */
    int num_experts;  /* E, 1..1024 */
    int topk;         /* k, 1..32 */
    int wfmt;         /* moe_wfmt */
    float act_clamp;  /* symmetric clamp of gate and up before SwiGLU; +INFINITY = off
                         (design §10.1 step 3, §1.1 decision 16) */
    int fast_math;    /* SwiGLU exponential: 0 expf (accurate), 1 __expf; the
                         division is the fast one (<= 2 ulp) either way */
} moe_config;

/* Bytes of device workspace for `cfg` (0 if `cfg` is invalid).  The pages
 * size the layer's one buffer with a call of its own (MegaMoE SM90
 * Implementation Design (Final), §16.1 "get_symm_buffer_size_for_sm90_mega_moe";
 * PR357 Green-Context Split MegaMoE code review, §3.1 "Split symmetric
 * buffer"); on one GPU the symmetric buffer is a plain device buffer holding
 * the dispatch tables, the token pool, the L2 activations and their scales,
 * the BF16 pair outputs and the staging of moe_forward_host.  The pages'
 * token-alignment query (design §16.1 "get_token_alignment_for_sm90_mega_moe")
 * has no counterpart: any num_tokens in [0, max_tokens] is accepted. */
MOE_API size_t moe_workspace_bytes(const moe_config *cfg);

/* Bytes of the transformed-weight store for `cfg` (0 if `cfg` is invalid):
 * what moe_transform_weights writes (design §16.1
 * "transform_weights_for_mega_moe_sm90", §15; PR357 review §3.2 "Weight
 * transform"). */
MOE_API size_t moe_weight_bytes(const moe_config *cfg);

/* Create a context bound to the current CUDA device.  The configuration
 * carries the arguments the pages' entry point takes besides its tensors
 * (design §16.1 fp8_mega_moe: num_max_tokens_per_rank, num_experts,
 * num_topk, the (1, 1, 128) recipe, activation_clamp, fast_math), minus the
 * rank and symmetric-buffer arguments.  d_workspace and d_weights are
 * caller-owned device buffers of the sizes above (256-byte aligned).  Writes
 * *out on success. */
MOE_API int moe_create(moe_ctx **out, const moe_config *cfg, void *d_workspace, void *d_weights);

/* Read the canonical weights and write the kernel layout into d_weights
 * (design §15: gate/up rows interleaved in groups of 8 along N).
 * Canonical layouts, all row-major, rows [0, I) of w1 = gate, [I, 2I) = up.
 * MOE_W_FP8_BLK128:
 *   w1    u8 (E4M3) [E, 2I, H],   w1_sf f32 [E, 2I/128, H/128]
 *   w2    u8 (E4M3) [E, H, I],    w2_sf f32 [E, H/128, I/128]
 * MOE_W_FP4_E2M1_UE8M0_32 (32-byte aligned code arrays):
 *   w1    u8 (2 x E2M1) [E, 2I, H/2],  w1_sf u8 (UE8M0) [E, 2I, H/32]
 *   w2    u8 (2 x E2M1) [E, H, I/2],   w2_sf u8 (UE8M0) [E, H, I/32]
 * The inputs may be freed once the stream has passed this call. */
MOE_API int moe_transform_weights(moe_ctx *ctx, const void *w1, const void *w1_sf,
                          const void *w2, const void *w2_sf, void *stream);

/* One forward pass (design §3.3).
 *   num_tokens T, 0 <= T <= max_tokens (T = 0 returns at once)
 *   x             u8 (E4M3) [T, H] row-major, rows 16-byte aligned
 *   x_sf          f32 [T, H/128] (FP8 weights) or u8 UE8M0 [T, H/32] (FP4 weights)
 *   topk_idx      int32 [T, k]; -1 marks an inactive slot
 *   topk_weights  f32 [T, k]
 *   y             bf16 [T, H] (written)
 *   cumulative_expert_counts  int32 [E] or NULL: the per-expert counts of
 *                 this call are added to it (design §16.1
 *                 "cumulative_local_expert_recv_stats")
 * Asynchronous on `stream`.  A call may be captured into a CUDA graph once
 * the same shape has run eagerly on the context (the first call sets kernel
 * attributes, once per process); replays read and write the buffers that
 * were passed at capture, with whatever they hold at replay. */
MOE_API int moe_forward(moe_ctx *ctx, int num_tokens, const void *x, const void *x_sf,
                const int32_t *topk_idx, const float *topk_weights, void *y,
                int32_t *cumulative_expert_counts, void *stream);

/* moe_forward with HOST inputs and output (the pages define no such call:
 * their layer reads inputs already in the symmetric buffer): copies h_x, h_x_sf, h_topk_idx,
 * h_topk_weights into the workspace, runs the forward and copies y back to
 * h_y, then synchronises `stream`.  Host buffers may be pageable or pinned
 * (pinned is faster).  When h_y is page-locked memory the device can
 * address (cudaHostAlloc / cudaHostRegister under unified addressing) and
 * 16-byte aligned, the combine stores y into it directly over the CPU-GPU
 * link and no copy back is made (environment MOE_HOST_DIRECT=0 turns that
 * off). */
MOE_API int moe_forward_host(moe_ctx *ctx, int num_tokens, const void *h_x, const void *h_x_sf,
                     const int32_t *h_topk_idx, const float *h_topk_weights, void *h_y,
                     void *stream);

/* Test export (the pages define no such call): copy the dispatch result of
 * the last forward (T tokens) into caller device
 * buffers: counts int32 [E], offsets int32 [E+1] (exclusive prefix of
 * counts), gather int32 [T*k] whose first offsets[E] entries are the pair ids
 * t*k + j of each expert's pairs in (token, slot) order, experts ascending
 * (later entries unspecified).  Any pointer may be NULL. */
MOE_API int moe_get_dispatch(moe_ctx *ctx, int32_t *counts, int32_t *offsets, int32_t *gather,
                     void *stream);

/* Test export (the pages define no such call): copy intermediates of the
 * last forward (T tokens; row r belongs to pair
 * gather[r], rows r >= offsets[E] unspecified), P = T*k:
 * l2_acts u8 (E4M3) [P, I], l2_sf = the L2 activation scales (f32 [P, I/64]
 * with FP8 weights, u8 UE8M0 [P, I/32] with FP4 weights),
 * l2_out bf16 [P, H] (the rounded L2 outputs).  Any pointer may be NULL.
 * For stage-by-stage tests. */
MOE_API int moe_get_intermediates(moe_ctx *ctx, void *l2_acts, void *l2_sf, void *l2_out,
                          void *stream);

/* Largest problem moe_dispatch_noalloc accepts. */
#define MOE_NOALLOC_MAX_PAIRS 65536   /* num_tokens * topk */
#define MOE_NOALLOC_MAX_EXPERTS 1024

/* The dispatch step alone, for callers that cannot allocate device memory
 * and cannot hand this library a workspace: code that runs inside a host
 * application or serving runtime which plans every device byte itself and
 * offers its plugins no workspace hook, or a path where a cudaMalloc would
 * stall the device or break the runtime's memory budget.  The pages have no
 * counterpart of this entry point.
 *
 * Computes what moe_forward's dispatch computes (counts int32 [E], offsets
 * int32 [E+1], gather int32 [T*k] with the first offsets[E] entries valid)
 * from topk_idx int32 [T,k] (device), into caller device buffers, on
 * `stream`.  It allocates nothing: the kernel's other scratch (pair -> row
 * map, M-block tables, error word) lives in one fixed device array of about
 * 270 KB inside this library, which every GPU that loads the library keeps
 * until the process exits.
 *  - Sizes: returns MOE_ERR_INVALID_ARG, launching nothing, when
 *    num_tokens * topk > MOE_NOALLOC_MAX_PAIRS, num_experts >
 *    MOE_NOALLOC_MAX_EXPERTS, topk outside [1, 32], or a pointer is NULL.
 *  - The first call on a device looks up that array's device address (with
 *    that device current); make this first call before any stream capture.
 *    The address is kept per device and context: after cudaDeviceReset the
 *    next call looks it up again in the new context.
 *  - Every call shares the one array and it keeps the last call's contents;
 *    the call clears what must start at zero.  Calls that overlap on the GPU
 *    (two streams, or two host threads) race on it and must not be issued.
 *  - Expert ids outside [-1, E) are skipped but not reported here. */
MOE_API int moe_dispatch_noalloc(const int32_t *topk_idx, int num_tokens, int topk,
                                 int num_experts, int32_t *counts, int32_t *offsets,
                                 int32_t *gather, void *stream);

/* Measurement plumbing (the pages define no such call).
 * Per-stage timing of the next `max_forwards` forwards: moe_profile_begin
 * creates CUDA events (no device memory) and every following moe_forward
 * records one event before its dispatch and one after each of its four
 * stages (dispatch, L1 GEMM, L2 GEMM, combine) on its stream.
 * moe_profile_end synchronises those events, writes the summed milliseconds
 * of each stage to stage_ms[4] and the number of recorded forwards to
 * *n_forwards, and releases the events. */
MOE_API int moe_profile_begin(moe_ctx *ctx, int max_forwards);
MOE_API int moe_profile_end(moe_ctx *ctx, float *stage_ms, int *n_forwards);

/* Test of the device-side timeout path (the pages have no counterpart; it
 * exists so that failure detection can be tested without faulting a GPU).
 * Arms the next moe_forward of `ctx`: every wait of that forward gives up
 * after `wait_limit_us` microseconds instead of 2 s, and
 *   which = 1 or 2: CTA 0's copy producer in GEMM `which` (1 = L1, 2 = L2)
 *           never fills its first pipeline stage, so the MMA's wait for it
 *           runs out (both weight formats);
 *   which = 3: CTA 0 of the multi-CTA dispatch (batches of 8192 routed pairs
 *           or more) never arrives at the grid-wide barrier, so the other
 *           CTAs' waits run out.
 * A step of a forward that times out makes that forward's later steps skip
 * (they check a per-forward abort word at entry) rather than read tables it
 * left incomplete.  That forward returns MOE_OK; its output is undefined;
 * moe_device_status() then returns MOE_ERR_DEVICE_TIMEOUT, and later forwards
 * run normally whether or not the status was read.  The hook disarms itself
 * after one forward.  Returns MOE_ERR_INVALID_ARG for another `which` or a
 * limit below 1 us. */
MOE_API int moe_test_arm_timeout(moe_ctx *ctx, int which, int wait_limit_us);

/* ABI plumbing (the pages define no such call): synchronise the device,
 * read and clear the device error word: MOE_OK, MOE_ERR_BAD_EXPERT,
 * MOE_ERR_DEVICE_TIMEOUT or MOE_ERR_CUDA. */
MOE_API int moe_device_status(moe_ctx *ctx);

/* ABI plumbing (no counterpart in the pages): static description of an
 * error code. */
MOE_API const char *moe_strerror(int code);

/* ABI plumbing (no counterpart in the pages): free the host state (never
 * the caller's buffers).  NULL is allowed. */
MOE_API void moe_destroy(moe_ctx *ctx);

#ifdef __cplusplus
}
#endif

#endif /* MOE_GB300_H */
