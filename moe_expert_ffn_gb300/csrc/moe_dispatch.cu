// moe_dispatch.cu -- dispatch of routed (token, slot) pairs to experts.
//
// Per-expert counts, their exclusive prefix and the gather map that lists
// each expert's pairs in (token, slot) order (MegaMoE SM90 Implementation
// Design (Final), §9.2 "Dispatch Pull Path" and §21 Phase 2; PR357
// Green-Context Split MegaMoE code review, §6.1 "Dispatch metadata").  On one
// GPU the pages' cross-rank pull becomes this local map: the L1 GEMM then
// reads token rows straight from x through it.
//
// One CTA of 1024 threads.  Each warp owns a contiguous segment of the pairs:
// pass 1 builds a per-warp histogram, a scan over (expert, warp) gives every
// warp its first slot inside each expert, pass 2 walks the segment in order
// and ranks equal experts inside each 32-pair batch with __match_any_sync, so
// the map is the stable order without any sort.
#include <mutex>

#include "moe.h"
#include "moe_device.cuh"
#include "moe_internal.h"

namespace moe {
namespace {

constexpr int kThreads = 1024;
constexpr int kWarps = kThreads / 32;

// Exclusive block-wide scan of one value per thread (blockDim = 1024).
__device__ __forceinline__ int block_exclusive_scan(int v, int *warp_tot, int *total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int x = v;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        int y = __shfl_up_sync(0xffffffffu, x, d);
        if (lane >= d) x += y;
    }
    if (lane == 31) warp_tot[warp] = x;
    __syncthreads();
    if (warp == 0) {
        int w = warp_tot[lane];
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            int y = __shfl_up_sync(0xffffffffu, w, d);
            if (lane >= d) w += y;
        }
        warp_tot[lane] = w;  // inclusive over warps
        if (lane == 31) *total = w;
    }
    __syncthreads();
    const int before = warp ? warp_tot[warp - 1] : 0;
    const int r = before + x - v;
    __syncthreads();
    return r;
}

__global__ void __launch_bounds__(kThreads, 1)
    dispatch_kernel(const int32_t *__restrict__ idx, int T, int k, int E, DispatchOut o) {
    extern __shared__ int32_t sm[];
    int32_t *hist = sm;                 // [kWarps][E]: count, then first slot of the warp
    int32_t *off_s = sm + kWarps * E;   // [E+1]
    __shared__ int warp_tot[kWarps];
    __shared__ int tot_a, tot_b, tot_c, tot_s, bad;

    const int P = T * k;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    for (int i = threadIdx.x; i < kWarps * E; i += kThreads) hist[i] = 0;
    if (threadIdx.x == 0) {
        bad = 0;
        reinterpret_cast<volatile int *>(o.err)[kAbortWord] = 0;   // a new forward
    }
    __syncthreads();

    const int seg = (P + kWarps - 1) / kWarps;
    const int p0 = min(P, warp * seg), p1 = min(P, p0 + seg);

    // pass 1: per-warp histogram
    for (int p = p0 + lane; p < p1; p += 32) {
        const int e = __ldg(idx + p);
        if (e >= 0 && e < E)
            atomicAdd(&hist[warp * E + e], 1);
        else if (e != -1)
            bad = 1;
    }
    __syncthreads();

    // per expert: first slot of each warp inside the expert, and the count
    int cnt = 0;
    if (threadIdx.x < E) {
        const int e = threadIdx.x;
        for (int w = 0; w < kWarps; ++w) {
            const int h = hist[w * E + e];
            hist[w * E + e] = cnt;
            cnt += h;
        }
    }
    // E <= kThreads: one expert per thread for both prefix scans
    const int nmb = (cnt + kBM - 1) / kBM;
    const int nmb2 = (cnt + 2 * kBM - 1) / (2 * kBM);
    const int off = block_exclusive_scan(cnt, warp_tot, &tot_a);
    // 128-row blocks: those of experts with several blocks first, then the
    // one-block experts (the tile walk spreads the latter among the former)
    const int mbo_m = block_exclusive_scan(nmb >= 2 ? nmb : 0, warp_tot, &tot_b);
    const int mbo_s = block_exclusive_scan(nmb == 1 ? 1 : 0, warp_tot, &tot_s);
    const int mbo = nmb >= 2 ? mbo_m : tot_b + mbo_s;
    const int mbo2 = block_exclusive_scan(nmb2, warp_tot, &tot_c);
    if (threadIdx.x < E) {
        off_s[threadIdx.x] = off;
        o.count[threadIdx.x] = cnt;
        o.offset[threadIdx.x] = off;
        o.mb_prefix[threadIdx.x] = mbo;
        if (o.stats) o.stats[threadIdx.x] += cnt;
        for (int b = 0; b < nmb; ++b) o.mblk_expert[mbo + b] = threadIdx.x;
        if (o.mb2_prefix) {
            o.mb2_prefix[threadIdx.x] = mbo2;
            for (int b = 0; b < nmb2; ++b) o.mblk2_expert[mbo2 + b] = threadIdx.x;
        }
    }
    if (threadIdx.x == 0) {
        off_s[E] = tot_a;
        o.offset[E] = tot_a;
        o.mb_prefix[E] = tot_b + tot_s;
        o.mb_prefix[E + 1] = tot_b;
        if (o.mb2_prefix) o.mb2_prefix[E] = tot_c;
        if (bad) atomicOr(o.err, kErrBadExpert);
    }
    __syncthreads();

    // pass 2: stable positions, batch by batch in pair order
    const uint32_t lt_mask = (1u << lane) - 1u;
    for (int base = p0; base < p1; base += 32) {
        const int p = base + lane;
        const int e = (p < p1) ? __ldg(idx + p) : -1;
        const bool ok = e >= 0 && e < E;
        const uint32_t grp = __match_any_sync(0xffffffffu, ok ? e : -1);
        int rank = 0;
        if (ok) {
            rank = __popc(grp & lt_mask);
            const int pos = off_s[e] + hist[warp * E + e] + rank;
            o.gather[pos] = p;
            o.pair_pool[p] = pos;
        } else if (p < p1) {
            o.pair_pool[p] = -1;
        }
        __syncwarp();
        if (ok && rank == __popc(grp) - 1) hist[warp * E + e] += __popc(grp);
        __syncwarp();
    }
}

// The same dispatch over G CTAs, for large batches (one CTA's 32 warps would
// walk dozens of 32-pair batches each, one dependent memory round trip after
// another).  A cooperative launch (every CTA resident).  CTA c takes the
// pairs [c*chunk, (c+1)*chunk) and runs the per-warp passes of
// dispatch_kernel on them; between the passes one grid-wide barrier (bounded)
// separates writing the CTA's per-expert counts from reading every CTA's:
// each CTA then knows the expert offsets and its own first slot inside each
// expert, so the stable (token, slot) order holds across CTAs.  CTA 0 writes
// the per-expert tables.  `bar` and the forward's abort word are zero before
// the launch; if the barrier runs out, the CTAs return without writing their
// part and the abort word makes the forward's later kernels skip.
__global__ void __launch_bounds__(kThreads, 1)
    dispatch_mc_kernel(const int32_t *__restrict__ idx, int T, int k, int E, DispatchOut o,
                       int32_t *__restrict__ cta_cnt, int *bar) {
    extern __shared__ int32_t sm[];
    int32_t *hist = sm;                 // [kWarps][E]: count, then first slot of the warp
    int32_t *off_s = sm + kWarps * E;   // [E+1]
    __shared__ int warp_tot[kWarps];
    __shared__ int tot_a, tot_b, tot_c, tot_s, bad, go;

    const int P = T * k;
    const int chunk = (P + (int)gridDim.x - 1) / (int)gridDim.x;
    const int c0 = min(P, (int)blockIdx.x * chunk), c1 = min(P, c0 + chunk);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    for (int i = threadIdx.x; i < kWarps * E; i += kThreads) hist[i] = 0;
    if (threadIdx.x == 0) bad = 0;
    __syncthreads();

    const int seg = (c1 - c0 + kWarps - 1) / kWarps;
    const int p0 = min(c1, c0 + warp * seg), p1 = min(c1, p0 + seg);

    // pass 1: per-warp histogram of this CTA's pairs
    for (int p = p0 + lane; p < p1; p += 32) {
        const int e = __ldg(idx + p);
        if (e >= 0 && e < E)
            atomicAdd(&hist[warp * E + e], 1);
        else if (e != -1)
            bad = 1;
    }
    __syncthreads();
    int cnt = 0;
    if (threadIdx.x < E) {
        const int e = threadIdx.x;
        for (int w = 0; w < kWarps; ++w) {
            const int h = hist[w * E + e];
            hist[w * E + e] = cnt;
            cnt += h;
        }
        cta_cnt[(size_t)blockIdx.x * E + e] = cnt;
        __threadfence();
    }
    if (threadIdx.x == 0 && bad) atomicOr(o.err, kErrBadExpert);

    // every CTA's counts written before any is read
    __syncthreads();
    if (threadIdx.x == 0) {
        const volatile int *ev = o.err;
        // timeout-path test: CTA 0 withholds its arrival, so the wait runs out
        const bool stall = blockIdx.x == 0 && ev[2] == kStallDispatch;
        if (!stall) red_release_gpu_add(bar, 1);
        const int lim_us = ev[1];
        const uint64_t limit = lim_us > 0 ? 1000ull * (uint64_t)lim_us : kWaitTimeoutNs;
        bool ok = true;
        const uint64_t t0 = globaltimer_ns();
        while (ld_acquire_gpu(bar) < (int)gridDim.x) {
            __nanosleep(64);
            if (globaltimer_ns() - t0 > limit) {
                raise_timeout(o.err);
                ok = false;
                break;
            }
        }
        go = ok;
    }
    __syncthreads();
    if (!go) return;

    // the expert totals and this CTA's first slot inside each expert
    int total = 0, before = 0;
    if (threadIdx.x < E) {
        for (int c = 0; c < (int)gridDim.x; ++c) {
            const int v = __ldcg(cta_cnt + (size_t)c * E + threadIdx.x);
            total += v;
            if (c < (int)blockIdx.x) before += v;
        }
    }
    const int off = block_exclusive_scan(total, warp_tot, &tot_a);
    if (threadIdx.x < E) off_s[threadIdx.x] = off + before;
    if (blockIdx.x == 0) {
        const int nmb = (total + kBM - 1) / kBM;
        const int nmb2 = (total + 2 * kBM - 1) / (2 * kBM);
        const int mbo_m = block_exclusive_scan(nmb >= 2 ? nmb : 0, warp_tot, &tot_b);
        const int mbo_s = block_exclusive_scan(nmb == 1 ? 1 : 0, warp_tot, &tot_s);
        const int mbo = nmb >= 2 ? mbo_m : tot_b + mbo_s;
        const int mbo2 = block_exclusive_scan(nmb2, warp_tot, &tot_c);
        if (threadIdx.x < E) {
            o.count[threadIdx.x] = total;
            o.offset[threadIdx.x] = off;
            o.mb_prefix[threadIdx.x] = mbo;
            if (o.stats) o.stats[threadIdx.x] += total;
            for (int b = 0; b < nmb; ++b) o.mblk_expert[mbo + b] = threadIdx.x;
            if (o.mb2_prefix) {
                o.mb2_prefix[threadIdx.x] = mbo2;
                for (int b = 0; b < nmb2; ++b) o.mblk2_expert[mbo2 + b] = threadIdx.x;
            }
        }
        if (threadIdx.x == 0) {
            o.offset[E] = tot_a;
            o.mb_prefix[E] = tot_b + tot_s;
            o.mb_prefix[E + 1] = tot_b;
            if (o.mb2_prefix) o.mb2_prefix[E] = tot_c;
        }
    }
    __syncthreads();

    // pass 2: stable positions, batch by batch in pair order
    const uint32_t lt_mask = (1u << lane) - 1u;
    for (int base = p0; base < p1; base += 32) {
        const int p = base + lane;
        const int e = (p < p1) ? __ldg(idx + p) : -1;
        const bool ok = e >= 0 && e < E;
        const uint32_t grp = __match_any_sync(0xffffffffu, ok ? e : -1);
        int rank = 0;
        if (ok) {
            rank = __popc(grp & lt_mask);
            const int pos = off_s[e] + hist[warp * E + e] + rank;
            o.gather[pos] = p;
            o.pair_pool[p] = pos;
        } else if (p < p1) {
            o.pair_pool[p] = -1;
        }
        __syncwarp();
        if (ok && rank == __popc(grp) - 1) hist[warp * E + e] += __popc(grp);
        __syncwarp();
    }
}

// The pages' "pull into the L1 pool" on one GPU (design §9.2): the FP8 row of
// the token of every pool row, in dispatch order.  One warp per row.
__global__ void __launch_bounds__(256)
    pool_gather_kernel(const uint8_t *__restrict__ x, const int32_t *__restrict__ gather,
                       const int32_t *__restrict__ offset_E, int k, int H, int rows_bound,
                       uint8_t *__restrict__ pool, int pool_pitch, const int *err) {
    if (forward_aborted(err)) return;   // the dispatch did not finish its tables
    const int P = min(__ldg(offset_E), rows_bound);
    const int lane = threadIdx.x & 31;
    const int vecs = H / 16;
    for (int r = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; r < P; r += (gridDim.x * blockDim.x) >> 5) {
        const int pair = __ldg(gather + r);
        if ((unsigned)pair >= (unsigned)rows_bound) continue;   // never a pair of this batch
        const int t = pair / k;
        const uint4 *src = reinterpret_cast<const uint4 *>(x + (size_t)t * H);
        uint4 *dst = reinterpret_cast<uint4 *>(pool + (size_t)r * pool_pitch);
        for (int v = lane; v < vecs; v += 32) dst[v] = __ldg(src + v);
    }
}

}  // namespace

void launch_pool_gather(const uint8_t *x, const int32_t *gather, const int32_t *offset_E, int k,
                        int H, int rows_bound, uint8_t *pool, int pool_pitch, const int *err, cudaStream_t s) {
    const int warps = 8;
    const int blocks = max(1, min((rows_bound + warps - 1) / warps, 65535));
    pool_gather_kernel<<<blocks, warps * 32, 0, s>>>(x, gather, offset_E, k, H, rows_bound, pool,
                                                      pool_pitch, err);
}

cudaError_t launch_dispatch(const int32_t *topk_idx, int T, int k, int E, const DispatchOut &o,
                            cudaStream_t s) {
    const size_t smem = sizeof(int32_t) * (size_t)(kWarps * E + E + 1);
    static std::atomic<uint32_t> smem_set{0};
    cudaError_t e = smem_limit_once(reinterpret_cast<const void *>(dispatch_kernel),
                                    sizeof(int32_t) * (kWarps * 1024 + 1025), smem_set);
    if (e != cudaSuccess) return e;
    // launched through cudaLaunchKernelEx so that the result is this launch's
    // own, not an error an earlier, unrelated call left behind
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(1);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    return cudaLaunchKernelEx(&cfg, dispatch_kernel, topk_idx, T, k, E, o);
}

cudaError_t launch_dispatch_mc(const int32_t *topk_idx, int T, int k, int E, const DispatchOut &o,
                               int32_t *cta_cnt, int *bar, int ctas, cudaStream_t s) {
    const size_t smem = sizeof(int32_t) * (size_t)(kWarps * E + E + 1);
    static std::atomic<uint32_t> smem_set{0};
    cudaError_t e = smem_limit_once(reinterpret_cast<const void *>(dispatch_mc_kernel),
                                    sizeof(int32_t) * (kWarps * 1024 + 1025), smem_set);
    if (e != cudaSuccess) return e;
    // the barrier counter and, next to it, the forward's abort word
    if ((e = cudaMemsetAsync(bar, 0, 2 * sizeof(int), s)) != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;   // the grid-wide barrier needs every CTA resident
    attr[0].val.cooperative = 1;
    cfg.gridDim = dim3(ctas);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, dispatch_mc_kernel, topk_idx, T, k, E, o, cta_cnt, bar);
}

}  // namespace moe

// ---------------------------------------------------------------------------
// moe_dispatch_noalloc: the same kernel with its scratch in a fixed device
// array, for callers that cannot allocate (see include/moe.h).
// ---------------------------------------------------------------------------
namespace {

constexpr int kNaPairs = MOE_NOALLOC_MAX_PAIRS;
constexpr int kNaExperts = MOE_NOALLOC_MAX_EXPERTS;
constexpr int kNaPairPool = 0;                                   // [kNaPairs]
constexpr int kNaMbPrefix = kNaPairPool + kNaPairs;              // [kNaExperts + 1]
constexpr int kNaMblk = kNaMbPrefix + kNaExperts + 64;           // [kNaPairs/128 + kNaExperts + 1]
constexpr int kNaErr = kNaMblk + kNaPairs / moe::kBM + kNaExperts + 64;
constexpr int kNaInts = kNaErr + 64;

// Shared by every call on a device; holds the last call's tables.
static __device__ __align__(256) int32_t g_noalloc_scratch[kNaInts];

constexpr int kNaMaxDevices = 64;
std::mutex g_noalloc_mu;

// The array's device address, looked up once per device and context.  The
// context's ID is kept beside it: after cudaDeviceReset the runtime makes a
// new primary context (a new ID) in which the library's module, and with it
// the array, may sit elsewhere, so the address is looked up again.
struct NoallocSlot {
    unsigned long long ctx_id;
    int32_t *ptr;
};
NoallocSlot g_noalloc_slot[kNaMaxDevices];

typedef CUresult (*CtxGetCurrentFn)(CUcontext *);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long *);

template <class Fn>
Fn driver_fn(const char *name, int version) {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion(name, &p, version, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
        return nullptr;
    return reinterpret_cast<Fn>(p);
}

// ID of the calling thread's current context, 0 when there is none yet (the
// runtime binds the primary context on its first call that needs one).
unsigned long long current_ctx_id() {
    static const CtxGetCurrentFn get_ctx = driver_fn<CtxGetCurrentFn>("cuCtxGetCurrent", 4000);
    static const CtxGetIdFn get_id = driver_fn<CtxGetIdFn>("cuCtxGetId", 12000);
    CUcontext ctx = nullptr;
    unsigned long long id = 0;
    if (!get_ctx || !get_id || get_ctx(&ctx) != CUDA_SUCCESS || !ctx || get_id(ctx, &id) != CUDA_SUCCESS) return 0;
    return id;
}

// Device address of g_noalloc_scratch on the current device (host code may
// not use the symbol itself: on the host it names a stand-in, not the array).
int noalloc_scratch(int32_t **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kNaMaxDevices) return MOE_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    NoallocSlot &sl = g_noalloc_slot[dev];
    const unsigned long long id = current_ctx_id();
    if (!sl.ptr || id == 0 || id != sl.ctx_id) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return MOE_ERR_CUDA;
        sl.ptr = static_cast<int32_t *>(p);
        sl.ctx_id = current_ctx_id();   // the lookup has bound a context if there was none
    }
    *out = sl.ptr;
    return MOE_OK;
}

}  // namespace

extern "C" MOE_API int moe_dispatch_noalloc(const int32_t *topk_idx, int num_tokens, int topk,
                                            int num_experts, int32_t *counts, int32_t *offsets,
                                            int32_t *gather, void *stream) {
    if (!topk_idx || !counts || !offsets || !gather) return MOE_ERR_INVALID_ARG;
    if (num_tokens < 0 || topk < 1 || topk > 32 || num_experts < 1 || num_experts > kNaExperts)
        return MOE_ERR_INVALID_ARG;
    if ((long long)num_tokens * topk > kNaPairs) return MOE_ERR_INVALID_ARG;
    int32_t *scratch = nullptr;
    const int rc = noalloc_scratch(&scratch);
    if (rc != MOE_OK) return rc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    moe::DispatchOut o;
    o.count = counts;
    o.offset = offsets;
    o.gather = gather;
    o.pair_pool = scratch + kNaPairPool;
    o.mb_prefix = scratch + kNaMbPrefix;
    o.mblk_expert = scratch + kNaMblk;
    o.mb2_prefix = nullptr;
    o.mblk2_expert = nullptr;
    o.stats = nullptr;
    o.err = scratch + kNaErr;
    // the error word is only ever OR-ed into: start it at zero
    if (cudaMemsetAsync(o.err, 0, sizeof(int32_t), s) != cudaSuccess) return MOE_ERR_CUDA;
    return moe::launch_dispatch(topk_idx, num_tokens, topk, num_experts, o, s) == cudaSuccess ? MOE_OK
                                                                                               : MOE_ERR_CUDA;
}
