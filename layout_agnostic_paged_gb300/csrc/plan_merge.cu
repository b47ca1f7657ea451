// plan_merge.cu -- split-KV plan (K1), intra-call combine of split partials (K3)
// and the public log-sum-exp merge (K4).
//
// The plan balances ragged requests across the persistent decode grid: all
// requests' 128-token tiles are concatenated and cut into at most G' near-equal
// ranges, one per CTA group (fewer when a range would hold only a few tiles); a
// request cut across several groups yields one partial per group, combined by K3
// with the same log-sum-exp merge K4 exposes.  The cut
// depends only on the context lengths and the token range, never on physical
// page ids, so results are identical under any page permutation.
//
// Method context: "SPLASH: Switching Parallel Layouts of Attention with Seamless
// Handoff for LLM Serving", Appendix, Table 2 (busiest-rank load of each layout:
// balance is what the layouts trade; CP reads an equal token share under ideal
// token partitioning, which is the partial + log-sum-exp merge implemented here).
#include <math.h>

#include "common.cuh"
#include "kernels.h"

namespace splash {

namespace {

constexpr int kPlanThreads = 256;

// Optional kernel-boundary trace (compiled in only with -DSPLASH_TRACE): globaltimer
// stamps of the plan and combine kernels, read back with splash_ktrace_read().
#ifdef SPLASH_TRACE
__device__ unsigned long long g_ktrace[8];
#define KTRACE_SET(slot) (g_ktrace[slot] = globaltimer_ns())
#define KTRACE_MIN(slot) atomicMin(&g_ktrace[slot], globaltimer_ns())
#define KTRACE_MAX(slot) atomicMax(&g_ktrace[slot], globaltimer_ns())
#else
#define KTRACE_SET(slot) ((void)0)
#define KTRACE_MIN(slot) ((void)0)
#define KTRACE_MAX(slot) ((void)0)
#endif

// Inclusive block scan of one int64 per thread (kPlanThreads threads).
__device__ int64_t block_inclusive_scan(int64_t v, int64_t* warp_sums) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        int64_t n = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += n;
    }
    if (lane == 31) warp_sums[warp] = v;
    __syncthreads();
    if (warp == 0) {
        int64_t s = lane < kPlanThreads / 32 ? warp_sums[lane] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            int64_t n = __shfl_up_sync(0xffffffffu, s, o);
            if (lane >= o) s += n;
        }
        warp_sums[lane] = s;
    }
    __syncthreads();
    int64_t add = warp > 0 ? warp_sums[warp - 1] : 0;
    __syncthreads();
    return v + add;
}

// Clipped token range and tile span of one request (the plan's per-request part
// that depends on nothing but its context length).
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

// Largest tiles-per-group count for which the plan uses fewer CTA groups than it may.
constexpr int64_t kRegroupMaxTiles = 4;

// Requests whose tile ends the plan keeps in shared memory for the group search;
// larger batches search the plan in global memory.
constexpr int kPlanSmemReqs = 8192;

// One CTA.  Every thread owns a contiguous run of requests; the run is recomputed
// from the inputs in each pass so that nothing written to global memory is read
// back, and the group search runs over shared memory.
__global__ void __launch_bounds__(kPlanThreads) plan_kernel(const int32_t* __restrict__ ctx_lens,
                                                            int B, int64_t tok_lo, int64_t tok_hi,
                                                            const int32_t* __restrict__ lo_arr,
                                                            const int32_t* __restrict__ hi_arr,
                                                            const int32_t* __restrict__ rows,
                                                            int num_rows, int max_ctx, int num_groups,
                                                            int Hs, uint8_t* __restrict__ ws) {
    extern __shared__ int64_t s_end[];  // [B] tile ends, when B <= kPlanSmemReqs
    __shared__ int64_t warp_sums[32];
    __shared__ int64_t s_total;
    if (threadIdx.x == 0) KTRACE_SET(0);
    pdl_wait();
    pdl_trigger();  // the decode grid may start its prologue now
    if (threadIdx.x == 0) KTRACE_SET(1);
    PlanHeader* hdr = reinterpret_cast<PlanHeader*>(ws);
    const WorkspaceLayout lay(B, Hs, num_groups);
    ReqPlan* req = reinterpret_cast<ReqPlan*>(ws + lay.req_off);
    const bool smem_ends = B <= kPlanSmemReqs;

    const int per = (B + kPlanThreads - 1) / kPlanThreads;
    const int r0 = min(B, int(threadIdx.x) * per);
    const int r1 = min(B, r0 + per);
    // Request r of the call: its storage row (rows[r], else r), its context length and
    // its token range (lo_arr[r] / hi_arr[r], else the call's scalars), clipped.  A row
    // outside [0, num_rows), a length outside [0, max_ctx] or a negative range start is
    // bad input (flagged; the row is skipped, the length clamped, the start taken as 0).
    auto span_of = [&](int r, bool& bad) {
        int row = rows ? rows[r] : r;
        int L = 0;
        if (row < 0 || row >= num_rows) {
            bad = true;
            row = -1;
        } else {
            L = ctx_lens[row];
            if (L < 0 || L > max_ctx) {
                bad = true;
                L = min(max(L, 0), max_ctx);
            }
        }
        int64_t lo = tok_lo, hi = tok_hi;
        if (lo_arr) {
            lo = lo_arr[r];
            if (lo < 0) {
                bad = true;
                lo = 0;
            }
        }
        if (hi_arr) hi = hi_arr[r];
        ReqPlan p = request_span(L, lo, hi);
        if (row < 0) p = request_span(0, 0, 0);
        p.row = row;
        return p;
    };

    // Pass 1: tile counts.
    bool bad = false;
    int64_t my_tiles = 0;
    for (int r = r0; r < r1; ++r) my_tiles += span_of(r, bad).ntiles;
    const int64_t incl = block_inclusive_scan(my_tiles, warp_sums);
    if (threadIdx.x == kPlanThreads - 1) s_total = incl;
    __syncthreads();
    const int64_t T = s_total;
    // The busiest group gets k = ceil(T / num_groups) tiles whatever the cut.  When k is
    // small, ceil(T / k) groups keep that critical path while giving every group k or
    // k - 1 tiles: fewer requests are split (fewer partial rows to merge) and the spare
    // SMs are free for concurrent work.  For long runs of tiles the extra tile on the
    // average group costs more than it saves, so every group is used.  G <= T makes
    // every group range non-empty, so a request's pieces are exactly the groups its
    // tiles fall in.
    const int64_t k = T > 0 ? (T + num_groups - 1) / num_groups : 0;
    const int64_t G = k == 0 ? 0 : k <= kRegroupMaxTiles ? (T + k - 1) / k : min(int64_t(num_groups), T);

    // Pass 2: global tile offsets, CTA-group cut and partial-slot counts.
    int64_t my_slots = 0;
    {
        int64_t tb = incl - my_tiles;
        bool unused = false;
        for (int r = r0; r < r1; ++r) {
            const ReqPlan p = span_of(r, unused);
            if (p.ntiles > 0) {
                const int64_t nsplit = group_of_tile(tb + p.ntiles - 1, T, G) - group_of_tile(tb, T, G) + 1;
                if (nsplit > 1) my_slots += nsplit;
            }
            tb += p.ntiles;
        }
    }
    const int64_t sincl = block_inclusive_scan(my_slots, warp_sums);

    // Pass 3: the complete request plans.
    {
        int64_t tb = incl - my_tiles, slot = sincl - my_slots;
        bool unused = false;
        for (int r = r0; r < r1; ++r) {
            ReqPlan p = span_of(r, unused);
            p.tile_begin = tb;
            if (p.ntiles > 0) {
                const int64_t g0 = group_of_tile(tb, T, G);
                const int64_t g1 = group_of_tile(tb + p.ntiles - 1, T, G);
                p.first_grp = int32_t(g0);
                p.nsplit = int32_t(g1 - g0 + 1);
                if (p.nsplit > 1) {
                    p.slot_base = int32_t(slot);
                    slot += p.nsplit;
                }
            }
            req[r] = p;
            tb += p.ntiles;
            if (smem_ends) s_end[r] = tb;
        }
    }
    const bool any_bad = __syncthreads_or(bad);  // also publishes s_end
    // First request of every CTA group: smallest r whose tiles reach past the group start,
    // so a decode CTA finds its first piece with one load instead of a search.
    int32_t* first_req = reinterpret_cast<int32_t*>(ws + lay.grp_off);
    for (int64_t j = threadIdx.x; j < G; j += kPlanThreads) {
        const int64_t x = group_start(j, T, G);
        int lo = 0, hi = B;
        while (lo < hi) {
            const int mid = (lo + hi) >> 1;
            const int64_t end = smem_ends ? s_end[mid] : req[mid].tile_begin + req[mid].ntiles;
            if (end > x) hi = mid;
            else lo = mid + 1;
        }
        first_req[j] = lo;
    }
    if (threadIdx.x == kPlanThreads - 1) {
        hdr->status = any_bad ? uint32_t(SPLASH_DEVICE_BAD_INPUT) : 0u;
        hdr->num_groups = int32_t(G);
        hdr->total_tiles = T;
        hdr->num_reqs = B;
        hdr->heads = Hs;
        hdr->max_slots = lay.max_slots;
        hdr->slots_used = int32_t(sincl);
        KTRACE_SET(2);
    }
}

// Merge `S` partial rows (out at stride `ostride` floats, lse at stride `lstride`)
// into one output row; one warp.  Lane s < 32 owns split s's weight (broadcast by
// shuffles, the lse column read once); lanes cover d_v in float4 steps with the
// loads of up to 4 splits (16 float4 per lane) in flight.  Splits are added in
// index order on every path.
__device__ __forceinline__ void warp_lse_merge(const float* __restrict__ pout, int64_t ostride,
                                               const float* __restrict__ plse, int64_t lstride,
                                               int S, int d_v, float* __restrict__ out,
                                               float* __restrict__ lse) {
    const int lane = threadIdx.x & 31;
    // For 512-wide rows (one pass) the first four splits' rows are loaded together with
    // the lse column, so the row loads do not wait for the weights.
    float4 pre[4][4];
    const bool one_pass = d_v == 512;
    if (one_pass) {
#pragma unroll
        for (int t = 0; t < 4; ++t)
            if (t < S)
#pragma unroll
                for (int c = 0; c < 4; ++c)
                    pre[t][c] = *reinterpret_cast<const float4*>(pout + t * ostride + lane * 4 + c * 128);
    }
    // up to 32 splits: one load of the lse column, kept in a register for all passes
    const float l0 = (lane < S) ? plse[lane * lstride] : -INFINITY;
    float m = l0;
    for (int s0 = 32; s0 < S; s0 += 32)
        if (s0 + lane < S) m = fmaxf(m, plse[(s0 + lane) * lstride]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    if (m == -INFINITY) {
        for (int j = lane * 4; j < d_v; j += 128)
            *reinterpret_cast<float4*>(out + j) = make_float4(0.f, 0.f, 0.f, 0.f);
        if (lane == 0) *lse = -INFINITY;
        return;
    }
    float wsum = (lane < S) ? expf(l0 - m) : 0.f;
    for (int s0 = 32; s0 < S; s0 += 32)
        if (s0 + lane < S) wsum += expf(plse[(s0 + lane) * lstride] - m);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) wsum += __shfl_xor_sync(0xffffffffu, wsum, o);
    const float inv = 1.0f / wsum;
    if (one_pass) {
        const float myw = (lane < S) ? expf(l0 - m) : 0.f;
        float4 acc[4];
#pragma unroll
        for (int c = 0; c < 4; ++c) acc[c] = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int t = 0; t < 4; ++t) {
            if (t < S) {
                const float w = __shfl_sync(0xffffffffu, myw, t);
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    acc[c].x += w * pre[t][c].x;
                    acc[c].y += w * pre[t][c].y;
                    acc[c].z += w * pre[t][c].z;
                    acc[c].w += w * pre[t][c].w;
                }
            }
        }
        for (int s0 = 0; s0 < S; s0 += 32) {      // splits 4.. in the same order
            const float w_s = s0 == 0 ? myw
                                      : ((s0 + lane < S) ? expf(plse[(s0 + lane) * lstride] - m) : 0.f);
            const int n = min(32, S - s0);
#pragma unroll 4
            for (int t = (s0 == 0 ? 4 : 0); t < n; ++t) {
                const float w = __shfl_sync(0xffffffffu, w_s, t);
                const float* src = pout + (s0 + t) * ostride + lane * 4;
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const float4 o = *reinterpret_cast<const float4*>(src + c * 128);
                    acc[c].x += w * o.x;
                    acc[c].y += w * o.y;
                    acc[c].z += w * o.z;
                    acc[c].w += w * o.w;
                }
            }
        }
#pragma unroll
        for (int c = 0; c < 4; ++c)
            *reinterpret_cast<float4*>(out + lane * 4 + c * 128) =
                make_float4(acc[c].x * inv, acc[c].y * inv, acc[c].z * inv, acc[c].w * inv);
        if (lane == 0) *lse = m + logf(wsum);
        return;
    }
    for (int j0 = 0; j0 < d_v; j0 += 512) {       // 512 floats per pass: 4 float4 per lane
        float4 acc[4];
#pragma unroll
        for (int c = 0; c < 4; ++c) acc[c] = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int s0 = 0; s0 < S; s0 += 32) {
            const float myw = s0 == 0 ? ((lane < S) ? expf(l0 - m) : 0.f)
                                      : ((s0 + lane < S) ? expf(plse[(s0 + lane) * lstride] - m) : 0.f);
            const int n = min(32, S - s0);
#pragma unroll 4
            for (int t = 0; t < n; ++t) {
                const float w = __shfl_sync(0xffffffffu, myw, t);
                const float* src = pout + (s0 + t) * ostride + j0 + lane * 4;
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    if (j0 + lane * 4 + c * 128 < d_v) {
                        const float4 o = *reinterpret_cast<const float4*>(src + c * 128);
                        acc[c].x += w * o.x;
                        acc[c].y += w * o.y;
                        acc[c].z += w * o.z;
                        acc[c].w += w * o.w;
                    }
                }
            }
        }
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            const int jj = j0 + lane * 4 + c * 128;
            if (jj < d_v)
                *reinterpret_cast<float4*>(out + jj) =
                    make_float4(acc[c].x * inv, acc[c].y * inv, acc[c].z * inv, acc[c].w * inv);
        }
    }
    if (lane == 0) *lse = m + logf(wsum);
}

// K3: one warp per (request, head) of the call's slice.  Requests cut across
// several CTA groups are merged from the workspace; empty requests get the
// empty-set result; single-piece requests were written by the decode kernel.
__global__ void __launch_bounds__(256) combine_kernel(const uint8_t* __restrict__ ws, int B, int H,
                                                      int head_lo, int Hs, int num_groups,
                                                      float* __restrict__ out,
                                                      float* __restrict__ lse) {
    if (threadIdx.x == 0) KTRACE_MIN(3);
    pdl_wait();
    if (threadIdx.x == 0) KTRACE_MIN(4);
    if (threadIdx.x == 0) KTRACE_MAX(5);
    const int64_t row = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    if (row >= int64_t(B) * Hs) return;
    const int r = int(row / Hs), hh = int(row % Hs);
    const WorkspaceLayout lay(B, Hs, num_groups);
    const ReqPlan p = reinterpret_cast<const ReqPlan*>(ws + lay.req_off)[r];
    if (p.nsplit == 1 || p.row < 0) return;
    float* o = out + (int64_t(p.row) * H + head_lo + hh) * kDv;
    float* l = lse + int64_t(p.row) * H + head_lo + hh;
    if (p.nsplit == 0) {
        const int lane = threadIdx.x & 31;
        for (int j = lane * 4; j < kDv; j += 128)
            *reinterpret_cast<float4*>(o + j) = make_float4(0.f, 0.f, 0.f, 0.f);
        if (lane == 0) *l = -INFINITY;
        return;
    }
    const float* pout = reinterpret_cast<const float*>(ws + lay.pout_off) +
                        (int64_t(p.slot_base) * Hs + hh) * kDv;
    const float* plse = reinterpret_cast<const float*>(ws + lay.plse_off) +
                        int64_t(p.slot_base) * Hs + hh;
    warp_lse_merge(pout, int64_t(Hs) * kDv, plse, Hs, p.nsplit, kDv, o, l);
}

// K4: the public merge, one warp per (b, h) row.
__global__ void __launch_bounds__(256) lse_merge_kernel(const float* __restrict__ part_out,
                                                        const float* __restrict__ part_lse, int S,
                                                        int64_t rows, int d_v,
                                                        float* __restrict__ out,
                                                        float* __restrict__ lse) {
    pdl_wait();
    const int64_t row = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    if (row >= rows) return;
    warp_lse_merge(part_out + row * d_v, rows * d_v, part_lse + row, rows, S, d_v,
                   out + row * d_v, lse + row);
}

}  // namespace

#ifdef SPLASH_TRACE
extern "C" __attribute__((visibility("default"))) int splash_ktrace_read(void* host_dst) {
    return cudaMemcpyFromSymbol(host_dst, g_ktrace, sizeof(g_ktrace)) == cudaSuccess ? 0 : -1;
}
extern "C" __attribute__((visibility("default"))) int splash_ktrace_clear() {
    const unsigned long long init[8] = {0, 0, 0, ~0ull, ~0ull, 0, 0, 0};
    return cudaMemcpyToSymbol(g_ktrace, init, sizeof(init)) == cudaSuccess ? 0 : -1;
}
#endif

cudaError_t launch_plan(const int32_t* ctx_lens, int B, int64_t tok_lo, int64_t tok_hi,
                        const int32_t* lo_arr, const int32_t* hi_arr, const int32_t* rows,
                        int num_rows, int max_ctx, int num_groups, int Hs, void* ws,
                        cudaStream_t stream) {
    const int smem = B <= kPlanSmemReqs ? B * int(sizeof(int64_t)) : 0;
    if (smem > 48 * 1024) {
        cudaError_t e = ensure_smem_optin(reinterpret_cast<const void*>(plan_kernel), smem);
        if (e != cudaSuccess) return e;
    }
    return launch_pdl(plan_kernel, dim3(1), dim3(kPlanThreads), size_t(smem), stream, ctx_lens, B,
                      tok_lo, tok_hi, lo_arr, hi_arr, rows, num_rows, max_ctx, num_groups, Hs,
                      static_cast<uint8_t*>(ws));
}

cudaError_t launch_combine(const void* ws, int B, int H, int head_lo, int Hs, int num_groups,
                           float* out, float* lse, cudaStream_t stream) {
    const int64_t threads = int64_t(B) * Hs * 32;
    const int blocks = int((threads + 255) / 256);
    if (blocks == 0) return cudaSuccess;
    return launch_pdl(combine_kernel, dim3(blocks), dim3(256), 0, stream,
                      static_cast<const uint8_t*>(ws), B, H, head_lo, Hs, num_groups, out, lse);
}

cudaError_t launch_lse_merge(const float* part_out, const float* part_lse, int S, int64_t rows,
                             int d_v, float* out, float* lse, cudaStream_t stream) {
    const int64_t threads = rows * 32;
    const int64_t blocks = (threads + 255) / 256;
    if (blocks == 0) return cudaSuccess;
    return launch_pdl(lse_merge_kernel, dim3(unsigned(blocks)), dim3(256), 0, stream, part_out,
                      part_lse, S, rows, d_v, out, lse);
}

}  // namespace splash
