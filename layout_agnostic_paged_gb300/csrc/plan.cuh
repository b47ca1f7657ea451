// plan.cuh -- the split plan (K1), computed by every decode CTA in its prologue.
//
// The plan balances ragged requests across the persistent decode grid: all requests'
// 128-token tiles are concatenated and cut into at most G' near-equal ranges, one per
// CTA group (fewer when a range would hold only a few tiles); a request cut across
// several groups yields one partial per group, combined by K3 with the same
// log-sum-exp merge K4 exposes.  The cut depends only on the context lengths and the
// token ranges, never on physical page ids, so results are identical under any page
// permutation.
//
// Every CTA scans the requests itself (two block-wide prefix sums over the tile and
// partial-slot counts), keeps only where its own group starts, and walks its requests
// from there, recomputing each request's span on the way.  CTA 0 also writes every
// request's plan and the header into the workspace for the combine kernel and for the
// caller.  No kernel runs before the decode grid.
//
// Method context: "SPLASH: Switching Parallel Layouts of Attention with Seamless
// Handoff for LLM Serving", Appendix, Table 2 (busiest-rank load of each layout: balance
// is what the layouts trade; CP reads an equal token share under ideal token
// partitioning, which is the partial + log-sum-exp merge implemented here).
#pragma once

#include "common.cuh"
#include "kernels.h"

namespace splash {

// Largest tiles-per-group count for which the plan uses fewer CTA groups than it may.
constexpr int64_t kRegroupMaxTiles = 4;

// Clipped token range and tile span of one request (everything but its place in the
// concatenated tile sequence).
__device__ __forceinline__ ReqPlan request_span(int L, int64_t tok_lo, int64_t tok_hi) {
    const int64_t lo = tok_lo;
    const int64_t hi = tok_hi < 0 ? int64_t(L) : min(tok_hi, int64_t(L));
    ReqPlan p;
    p.ctx_len = L;
    if (hi <= lo) {
        p.lo = p.hi = 0;
        p.tile0 = 0;
        p.ntiles = 0;
    } else {
        p.lo = int32_t(lo);
        p.hi = int32_t(hi);
        p.tile0 = int32_t(lo / kTileTokens);
        p.ntiles = int32_t((hi + kTileTokens - 1) / kTileTokens - lo / kTileTokens);
    }
    p.tile_begin = 0;
    p.first_grp = 0;
    p.nsplit = 0;
    p.slot_base = -1;
    p.row = -1;
    p.pad = 0;
    return p;
}

// Request r of the call: its storage row (rows[r], else r), its context length and its
// token range (lo_arr[r] / hi_arr[r], else the call's scalars), clipped.  A row outside
// [0, num_rows), a length outside [0, max_ctx] or a negative range start is bad input
// (flagged; the row is skipped, the length clamped, the start taken as 0).
__device__ __forceinline__ ReqPlan span_of(const DecodeArgs& a, int r, bool& bad) {
    int row = a.rows ? a.rows[r] : r;
    int L = 0;
    if (row < 0 || row >= a.num_rows) {
        bad = true;
        row = -1;
    } else {
        L = a.ctx_lens[row];
        if (L < 0 || L > a.max_ctx) {
            bad = true;
            L = min(max(L, 0), a.max_ctx);
        }
    }
    int64_t lo = a.tok_lo, hi = a.tok_hi;
    if (a.lo_arr) {
        lo = a.lo_arr[r];
        if (lo < 0) {
            bad = true;
            lo = 0;
        }
    }
    if (a.hi_arr) hi = a.hi_arr[r];
    ReqPlan p = request_span(L, lo, hi);
    if (row < 0) p = request_span(0, 0, 0);
    p.row = row;
    return p;
}

// Groups in use for T tiles over num_groups CTA groups.  The busiest group gets
// k = ceil(T / num_groups) tiles whatever the cut.  When k is small, ceil(T / k) groups
// keep that critical path while giving every group k or k - 1 tiles: fewer requests are
// split (fewer partial rows to merge) and the spare SMs are free for concurrent work.
// For long runs of tiles the extra tile on the average group costs more than it saves,
// so every group is used.  G <= T makes every group range non-empty, so a request's
// pieces are exactly the groups its tiles fall in.
__host__ __device__ inline int64_t plan_groups(int64_t T, int64_t num_groups) {
    const int64_t k = T > 0 ? (T + num_groups - 1) / num_groups : 0;
    return k == 0 ? 0 : (k <= kRegroupMaxTiles ? (T + k - 1) / k : min(num_groups, T));
}

// Inclusive prefix sum of one int64 per thread over a block of nthreads (a multiple of
// 32, at most 1024); warp_sums holds 32 int64 of shared memory.
__device__ __forceinline__ int64_t block_inclusive_scan(int64_t v, int64_t* warp_sums, int nthreads) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int64_t n = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += n;
    }
    if (lane == 31) warp_sums[warp] = v;
    __syncthreads();
    if (warp == 0) {
        int64_t s = lane < nthreads / 32 ? warp_sums[lane] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int64_t n = __shfl_up_sync(0xffffffffu, s, o);
            if (lane >= o) s += n;
        }
        warp_sums[lane] = s;
    }
    __syncthreads();
    const int64_t add = warp > 0 ? warp_sums[warp - 1] : 0;
    __syncthreads();
    return v + add;
}

// Where CTA group j's walk starts: its first request, that request's first tile in the
// concatenated sequence and the first partial slot at or after it.
struct PlanStart {
    int64_t T;        // tiles over all requests
    int64_t G;        // CTA groups in use
    int64_t tb;       // tile_begin of the first request
    int32_t r;        // first request with a tile at or after the group's start (B: none)
    int32_t slot;     // partial slots of all requests before r
};

// The CTA-wide plan scan.  Every thread of the block calls it (nthreads of them); it
// returns the same PlanStart in every thread.  When `writer` is set the block also writes
// every request's ReqPlan and the header (status bits of the scan into *cta_status).
__device__ PlanStart plan_prologue(const DecodeArgs& a, int j, bool writer, int nthreads,
                                   int64_t* scratch /* 32 + 4 int64 of shared memory */,
                                   uint32_t* cta_status) {
    int64_t* warp_sums = scratch;
    int64_t* bcast = scratch + 32;
    const int B = a.B;
    const int per = (B + nthreads - 1) / nthreads;
    const int r0 = min(B, int(threadIdx.x) * per);
    const int r1 = min(B, r0 + per);
    bool bad = false;
    int64_t my_tiles = 0;
    for (int r = r0; r < r1; ++r) my_tiles += span_of(a, r, bad).ntiles;
    const int64_t incl = block_inclusive_scan(my_tiles, warp_sums, nthreads);
    if (threadIdx.x == nthreads - 1) bcast[0] = incl;
    __syncthreads();
    PlanStart s;
    s.T = bcast[0];
    s.G = plan_groups(s.T, a.num_groups);
    const int64_t T = s.T, G = s.G;
    // partial-slot counts
    int64_t my_slots = 0;
    {
        int64_t tb = incl - my_tiles;
        bool unused = false;
        for (int r = r0; r < r1; ++r) {
            const ReqPlan p = span_of(a, r, unused);
            if (p.ntiles > 0) {
                const int64_t ns = group_of_tile(tb + p.ntiles - 1, T, G) - group_of_tile(tb, T, G) + 1;
                if (ns > 1) my_slots += ns;
            }
            tb += p.ntiles;
        }
    }
    const int64_t sincl = block_inclusive_scan(my_slots, warp_sums, nthreads);
    // the thread whose run holds tile a_j finds the group's first request
    if (threadIdx.x == 0) {
        bcast[1] = B;
        bcast[2] = 0;
        bcast[3] = 0;
    }
    __syncthreads();
    const int64_t aj = (T > 0 && j < G) ? group_start(j, T, G) : T;
    const int64_t run0 = incl - my_tiles;
    if (aj < T && run0 <= aj && aj < incl) {
        int64_t tb = run0, slot = sincl - my_slots;
        bool unused = false;
        for (int r = r0; r < r1; ++r) {
            const ReqPlan p = span_of(a, r, unused);
            if (tb + p.ntiles > aj) {
                bcast[1] = r;
                bcast[2] = tb;
                bcast[3] = slot;
                break;
            }
            if (p.ntiles > 0) {
                const int64_t ns = group_of_tile(tb + p.ntiles - 1, T, G) - group_of_tile(tb, T, G) + 1;
                if (ns > 1) slot += ns;
            }
            tb += p.ntiles;
        }
    }
    if (writer) {
        // every request's plan and the header, for the combine kernel and the caller
        const WorkspaceLayout lay(a.B, a.Hs, a.num_groups, a.sts_cap);
        uint8_t* ws = static_cast<uint8_t*>(a.ws);
        ReqPlan* req = reinterpret_cast<ReqPlan*>(ws + lay.req_off);
        int64_t tb = run0, slot = sincl - my_slots;
        bool unused = false;
        for (int r = r0; r < r1; ++r) {
            ReqPlan p = span_of(a, r, unused);
            p.tile_begin = tb;
            if (p.ntiles > 0) {
                const int64_t g0 = group_of_tile(tb, T, G), g1 = group_of_tile(tb + p.ntiles - 1, T, G);
                p.first_grp = int32_t(g0);
                p.nsplit = int32_t(g1 - g0 + 1);
                if (p.nsplit > 1) {
                    p.slot_base = int32_t(slot);
                    slot += p.nsplit;
                }
            }
            req[r] = p;
            tb += p.ntiles;
        }
        if (threadIdx.x == nthreads - 1) {
            PlanHeader* hdr = reinterpret_cast<PlanHeader*>(ws);
            hdr->num_groups = int32_t(G);
            hdr->total_tiles = T;
            hdr->num_reqs = B;
            hdr->heads = a.Hs;
            hdr->max_slots = lay.max_slots;
            hdr->slots_used = int32_t(sincl);
        }
        if (bad) atomicOr(cta_status, uint32_t(SPLASH_DEVICE_BAD_INPUT));
    }
    __syncthreads();
    s.r = int32_t(bcast[1]);
    s.tb = bcast[2];
    s.slot = int32_t(bcast[3]);
    return s;
}

// Iterates the pieces (request, tile range) of CTA group j, identically in every role,
// from the group's PlanStart: each request's span is recomputed from the inputs, its
// place in the tile sequence and its partial slots from running sums.
struct PieceIter {
    const DecodeArgs* a;
    int64_t T, G, aj, bj, tb;
    int r;
    int32_t slot;
    int j;
    __device__ PieceIter(const DecodeArgs& a_, const PlanStart& s, int64_t aj_, int64_t bj_, int j_)
        : a(&a_), T(s.T), G(s.G), aj(aj_), bj(bj_), tb(s.tb), r(aj_ < bj_ ? s.r : a_.B),
          slot(s.slot), j(j_) {}
    __device__ bool next(Piece& pc, ReqPlan& p) {
        while (r < a->B && tb < bj) {
            bool unused = false;
            p = span_of(*a, r, unused);
            p.tile_begin = tb;
            const int cur = r++;
            tb += p.ntiles;
            if (p.ntiles == 0) continue;
            const int64_t g0 = group_of_tile(p.tile_begin, T, G);
            const int64_t g1 = group_of_tile(p.tile_begin + p.ntiles - 1, T, G);
            p.first_grp = int32_t(g0);
            p.nsplit = int32_t(g1 - g0 + 1);
            if (p.nsplit > 1) {
                p.slot_base = slot;
                slot += p.nsplit;
            }
            pc.r = cur;
            pc.row = p.row;
            pc.t_lo = int(max(aj, p.tile_begin) - p.tile_begin);
            pc.t_hi = int(min(bj, p.tile_begin + p.ntiles) - p.tile_begin);
            pc.split = j - p.first_grp;
            pc.valid = true;
            return true;
        }
        return false;
    }
};

}  // namespace splash
