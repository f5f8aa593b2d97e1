// moe_gemm_common.cuh -- tile scheduler and small helpers shared by the
// grouped-GEMM kernels (FP8 block-scaled-in-software and FP4 block-scaled).
#pragma once

#include "moe_device.cuh"
#include "moe_internal.h"

namespace moe {

struct Tile {
    int e, row0, rows, nb, nmb;   // nmb: M blocks of expert e
    int mbi;                      // global index of the tile's M block (mb_prefix[e] + its block in e)
};

// Tile `tile` of a grouped GEMM with NB column blocks: experts in ascending
// order, each expert's M blocks x NB column blocks walked N-major when the
// expert has at least kNMajorMinRows pairs (weight tile reused across
// consecutive CTAs), M-major otherwise (design §12.2 "Auto N-Major").
__device__ __forceinline__ Tile make_tile(int tile, int NB, int e, int first, int nmb, int off, int cnt) {
    Tile t;
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
    t.mbi = first + mb;
    return t;
}

__device__ __forceinline__ Tile decode_tile(int tile, int NB, const int32_t *__restrict__ offset,
                                            const int32_t *__restrict__ mb_prefix,
                                            const int32_t *__restrict__ mblk_expert) {
    const int e = __ldg(mblk_expert + tile / NB);
    const int first = __ldg(mb_prefix + e);
    const int off = __ldg(offset + e);
    const int cnt = __ldg(offset + e + 1) - off;
    return make_tile(tile, NB, e, first, (cnt + kBM - 1) / kBM, off, cnt);
}

// Position p of a CTA's tile walk -> tile index.  Tiles are numbered expert
// by expert with the one-block experts' tiles last (`singles` of `total`);
// the walk spreads those evenly among the others (position p takes the next
// one-block tile when floor((p + 1) s / n) > floor(p s / n)), so that at any
// time the CTAs streaming once-read weights from HBM are the same share of
// all CTAs, next to CTAs on weight tiles that several M blocks share.  Each
// kind keeps its own order, so the N-major walk of a large expert still
// reaches neighbouring CTAs together.
__device__ __forceinline__ int tile_at_position(int p, int total, int singles) {
    const int s0 = (int)((long long)p * singles / total);
    const int s1 = (int)((long long)(p + 1) * singles / total);
    return s1 > s0 ? total - singles + s0 : p - s0;
}

// Tiles of a grouped GEMM with NB column blocks, and how many of them belong
// to one-block experts (from the block table's last two words).
__device__ __forceinline__ void tile_counts(const int32_t *mb_prefix, int E, int NB, int &total, int &singles) {
    const int all = __ldcg(mb_prefix + E);
    total = all * NB;
    singles = (all - __ldcg(mb_prefix + E + 1)) * NB;
}

// The same decode in two steps, for a producer that must not stall on it:
// begin() loads the tile's expert, finish() (once that has arrived, a stage
// or so later) the expert's offsets; tile() then needs no load.
struct TilePrefetch {
    int tl, e, first, off, off1;
    // L2-coherent loads: the one-launch forward writes these tables earlier
    // in the same launch
    __device__ __forceinline__ void begin(int tile, int NB, const int32_t *mblk_expert) {
        tl = tile;
        e = __ldcg(mblk_expert + tile / NB);
    }
    __device__ __forceinline__ void finish(const int32_t *offset, const int32_t *mb_prefix) {
        first = __ldcg(mb_prefix + e);
        off = __ldcg(offset + e);
        off1 = __ldcg(offset + e + 1);
    }
    __device__ __forceinline__ Tile tile(int NB) const {
        return make_tile(tl, NB, e, first, (off1 - off + kBM - 1) / kBM, off, off1 - off);
    }
};

__device__ __forceinline__ uint32_t align1024(uint32_t a) { return (a + 1023u) & ~1023u; }

// Index of the smallest A box (32, 64 or 128 rows) covering `rows` rows.
__device__ __forceinline__ int a_box_index(int rows) { return rows <= 32 ? 0 : (rows <= 64 ? 1 : 2); }

// Bounded wait used only on the abort path (does not look at the abort flag;
// same limit as mbar_wait).
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity, const int *err) {
    const int lim_us = reinterpret_cast<const volatile int *>(err)[1];
    const uint64_t limit = lim_us > 0 ? 1000ull * (uint64_t)lim_us : kWaitTimeoutNs;
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(bar, parity))
        if (globaltimer_ns() - t0 > limit) return;
}

// Test of the timeout path: whether the producer of the first CTA of GEMM
// `which` (cta: the CTA's index among the CTAs that run that GEMM) withholds
// the copies of its first stage (so the MMA's wait for them runs out).
__device__ __forceinline__ bool test_stall(const int *err, int which, int cta) {
    return cta == 0 && reinterpret_cast<const volatile int *>(err)[2] == which;
}


}  // namespace moe
