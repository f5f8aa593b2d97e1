// moe_phases.cuh -- the non-GEMM phases of the one-launch forward: a bounded
// grid-wide barrier, the multi-CTA dispatch written for any CTA size, the
// pool copy and the combine, as device functions that every CTA of one
// cooperative launch runs in turn (MegaMoE SM90 Implementation Design
// (Final), §3.3 "Fused Kernel Pipeline": Phase 1 dispatch with a grid sync,
// Phase 4 combine reduce after a barrier).  Data written earlier in the same
// launch by other CTAs is read with L2-coherent loads (ld.global.cg).
#pragma once

#include "moe_device.cuh"
#include "moe_internal.h"

namespace moe {

// Every CTA of the launch arrives once; returns once `target` arrivals are
// in (targets grow by gridDim.x per barrier on one counter that is zero
// before the launch).  Bounded like the pipeline waits: on a timeout it
// records kErrTimeout, sets the forward's abort word and returns false.
// `stall`: a timeout-path test, the CTA does not arrive.
__device__ __forceinline__ bool grid_sync(int *bar, int target, int *err, bool stall = false) {
    __shared__ int go;
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();
        if (!stall) red_release_gpu_add(bar, 1);
        const int lim_us = reinterpret_cast<volatile int *>(err)[1];
        const uint64_t limit = lim_us > 0 ? 1000ull * (uint64_t)lim_us : kWaitTimeoutNs;
        const uint64_t t0 = globaltimer_ns();
        bool ok = true;
        while (ld_acquire_gpu(bar) < target) {
            __nanosleep(64);
            if (globaltimer_ns() - t0 > limit) {
                raise_timeout(err);
                ok = false;
                break;
            }
        }
        go = ok;
    }
    __syncthreads();
    return go != 0;
}

// Exclusive prefix sum, in place, of n ints in shared memory by the whole
// CTA (any blockDim); returns the total.  Each thread sums a contiguous run,
// the runs are scanned by one warp, and each thread then writes its run.
__device__ __forceinline__ int cta_exclusive_scan(int *a, int n, int *scratch /* [33] */) {
    const int nt = blockDim.x, tid = threadIdx.x;
    const int per = (n + nt - 1) / nt;
    const int lo = min(n, tid * per), hi = min(n, lo + per);
    int s = 0;
    for (int i = lo; i < hi; ++i) s += a[i];
    // scan of the per-thread sums: warp-level, then over warps
    const int lane = tid & 31, warp = tid >> 5, nw = (nt + 31) / 32;
    int x = s;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, d);
        if (lane >= d) x += y;
    }
    if (lane == 31) scratch[warp] = x;
    __syncthreads();
    if (tid == 0) {
        int run = 0;
        for (int w = 0; w < nw; ++w) {
            const int v = scratch[w];
            scratch[w] = run;
            run += v;
        }
        scratch[32] = run;
    }
    __syncthreads();
    int base = scratch[warp] + x - s;
    for (int i = lo; i < hi; ++i) {
        const int v = a[i];
        a[i] = base;
        base += v;
    }
    const int total = scratch[32];
    __syncthreads();
    return total;
}

// The dispatch (counts, offsets, M-block tables, the stable gather map and
// the pair -> pool-row map) over all CTAs of the launch: CTA c takes the
// pairs [c*chunk, (c+1)*chunk); per-warp histograms and ranks as in the
// dispatch kernels, one grid barrier between writing the CTA's per-expert
// counts (cta_cnt [grid, E]) and reading every CTA's.  smem: at least
// (warps * E + 2 * E + 1) ints.  Returns false if a barrier timed out.
// The CTA-pair tables (mb2) are not written: the one-launch forward does
// not use CTA pairs.
__device__ __forceinline__ bool dispatch_phase(const int32_t *__restrict__ idx, int T, int k, int E,
                                               const DispatchOut &o, int32_t *cta_cnt, int *bar,
                                               int &bar_target, int32_t *smem, bool stall) {
    __shared__ int scratch[33];
    __shared__ int bad;
    const int nt = blockDim.x, nw = nt / 32;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    int32_t *hist = smem;                  // [nw][E]: count, then first slot of the warp
    int32_t *tot = smem + nw * E;          // [E]: expert totals, then their offsets
    int32_t *off_s = tot + E;              // [E]: this CTA's first slot of each expert
    const int P = T * k;
    const int chunk = (P + (int)gridDim.x - 1) / (int)gridDim.x;
    const int c0 = min(P, (int)blockIdx.x * chunk), c1 = min(P, c0 + chunk);
    for (int i = tid; i < nw * E; i += nt) hist[i] = 0;
    if (tid == 0) bad = 0;
    __syncthreads();
    const int seg = (c1 - c0 + nw - 1) / nw;
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
    for (int e = tid; e < E; e += nt) {
        int cnt = 0;
        for (int w = 0; w < nw; ++w) {
            const int h = hist[w * E + e];
            hist[w * E + e] = cnt;
            cnt += h;
        }
        cta_cnt[(size_t)blockIdx.x * E + e] = cnt;
    }
    if (tid == 0 && bad) atomicOr(o.err, kErrBadExpert);
    bar_target += (int)gridDim.x;
    if (!grid_sync(bar, bar_target, o.err, stall)) return false;

    // expert totals, and this CTA's first slot inside each expert (before
    // the expert offset is added)
    for (int e = tid; e < E; e += nt) {
        int total = 0, before = 0;
        for (int c = 0; c < (int)gridDim.x; ++c) {
            const int v = __ldcg(cta_cnt + (size_t)c * E + e);
            total += v;
            if (c < (int)blockIdx.x) before += v;
        }
        tot[e] = total;
        off_s[e] = before;
    }
    __syncthreads();
    if (blockIdx.x == 0)
        for (int e = tid; e < E; e += nt) {
            o.count[e] = tot[e];
            if (o.stats) o.stats[e] += tot[e];
        }
    const int P_act = cta_exclusive_scan(tot, E, scratch);   // tot -> expert offsets
    for (int e = tid; e < E; e += nt) off_s[e] += tot[e];
    if (blockIdx.x == 0) {
        for (int e = tid; e < E; e += nt) o.offset[e] = tot[e];
        if (tid == 0) o.offset[E] = P_act;
        // M blocks of 128 rows: the expert's first block and the block -> expert table
        __syncthreads();
        // (experts with several blocks first, then the one-block experts)
        for (int e = tid; e < E; e += nt) {
            const int next = (e + 1 < E) ? tot[e + 1] : P_act;
            const int nmb = (next - tot[e] + kBM - 1) / kBM;
            hist[e] = nmb >= 2 ? nmb : 0;   // hist is free again
            hist[E + e] = nmb == 1 ? 1 : 0;
        }
        __syncthreads();
        const int multi_total = cta_exclusive_scan(hist, E, scratch);
        const int single_total = cta_exclusive_scan(hist + E, E, scratch);
        for (int e = tid; e < E; e += nt) {
            const int next = (e + 1 < E) ? tot[e + 1] : P_act;
            const int nmb = (next - tot[e] + kBM - 1) / kBM;
            const int first = nmb >= 2 ? hist[e] : multi_total + hist[E + e];
            o.mb_prefix[e] = first;
            for (int b = 0; b < nmb; ++b) o.mblk_expert[first + b] = e;
        }
        if (tid == 0) {
            o.mb_prefix[E] = multi_total + single_total;
            o.mb_prefix[E + 1] = multi_total;
        }
        __syncthreads();
        // restore this CTA's per-warp first slots (pass 2 needs them): recompute
        for (int i = tid; i < nw * E; i += nt) hist[i] = 0;
        __syncthreads();
        for (int p = p0 + lane; p < p1; p += 32) {
            const int e = __ldg(idx + p);
            if (e >= 0 && e < E) atomicAdd(&hist[warp * E + e], 1);
        }
        __syncthreads();
        for (int e = tid; e < E; e += nt) {
            int cnt = 0;
            for (int w = 0; w < nw; ++w) {
                const int h = hist[w * E + e];
                hist[w * E + e] = cnt;
                cnt += h;
            }
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
    bar_target += (int)gridDim.x;
    return grid_sync(bar, bar_target, o.err);
}

// pool[r] = x[gather[r] / k] for the first offset[E] rows, one warp per row,
// rows spread over every warp of the launch.
__device__ __forceinline__ void pool_phase(const uint8_t *__restrict__ x, const int32_t *gather,
                                           const int32_t *offset_E, int k, int H, int rows_bound,
                                           uint8_t *__restrict__ pool, int pool_pitch) {
    const int P = min(__ldcg(offset_E), rows_bound);
    const int lane = threadIdx.x & 31;
    const int gw = (int)blockIdx.x * ((int)blockDim.x >> 5) + ((int)threadIdx.x >> 5);
    const int nwarps = (int)gridDim.x * ((int)blockDim.x >> 5);
    const int vecs = H / 16;
    for (int r = gw; r < P; r += nwarps) {
        const int pair = __ldcg(gather + r);
        if ((unsigned)pair >= (unsigned)rows_bound) continue;
        const uint4 *src = reinterpret_cast<const uint4 *>(x + (size_t)(pair / k) * H);
        uint4 *dst = reinterpret_cast<uint4 *>(pool + (size_t)r * pool_pitch);
        for (int v = lane; v < vecs; v += 32) dst[v] = __ldg(src + v);
    }
}

// y[t] = bf16( sum over active slots, in slot order from +0, of the BF16
// pair outputs ), tokens spread over the CTAs, 8 columns per thread.
__device__ __forceinline__ void combine_phase(const uint16_t *l2_out, const int32_t *pair_pool, int T, int k,
                                              int H, uint16_t *__restrict__ y) {
    for (int t = blockIdx.x; t < T; t += gridDim.x) {
        for (int h0 = threadIdx.x * 8; h0 < H; h0 += blockDim.x * 8) {
            float acc[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) acc[i] = 0.0f;
            for (int j = 0; j < k; ++j) {
                const int row = __ldcg(pair_pool + (size_t)t * k + j);
                if (row < 0) continue;
                const uint4 v = __ldcg(reinterpret_cast<const uint4 *>(l2_out + (size_t)row * H + h0));
                const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    acc[2 * i] += __uint_as_float(w[i] << 16);
                    acc[2 * i + 1] += __uint_as_float(w[i] & 0xFFFF0000u);
                }
            }
            uint4 out;
            out.x = bf16x2(acc[0], acc[1]);
            out.y = bf16x2(acc[2], acc[3]);
            out.z = bf16x2(acc[4], acc[5]);
            out.w = bf16x2(acc[6], acc[7]);
            *reinterpret_cast<uint4 *>(y + (size_t)t * H + h0) = out;
        }
    }
}

}  // namespace moe
