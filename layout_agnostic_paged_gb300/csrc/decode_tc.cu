// decode_tc.cu -- tensor-core (tcgen05 / TMEM / TMA) paged MLA decode kernel for sm_103a.
//
// Method: "SPLASH: Switching Parallel Layouts of Attention with Seamless Handoff
// for LLM Serving".  Abstract: with one shared latent KV head, every query head
// of a request reads the same KV stream, so decode attention over a head share,
// a token share or whole requests is one contraction over the same paged cache
// (Appendix, Table 2 gives which share each layout owns).
//
// Shape of the contraction per 128-token tile (swap-AB: tokens are the MMA M):
//   S^T [128 tok x N heads] = K_tile [128 x 576] . Q^T          (36 MMAs, K-major A and B)
//   softmax over tokens per head (fp32, exp2 domain, lazily rescaled running max)
//   O^T [512 dv x N heads] += V_tile^T [512 x 128] . P^T [128 x N]  (4 dv blocks x 8 MMAs,
//                                                                   MN-major A and B)
// N = heads of the CTA's head group padded to 16/32/64, so S^T (N columns) and
// O^T (4N columns) fit in the 512 TMEM columns of one SM.  V is the latent
// prefix of the key: the same shared-memory tile feeds both contractions.
//
// Roles (one CTA per SM, persistent over the split plan's pieces; 256 threads, or
// 384 at N = 64 where two softmax warpgroups each own half of the heads):
//   warp 0 and  TMA producers: Q of the piece, then per tile four 32 KB "pairs"
//   the last    (latent column blocks 2j, 2j+1) and the 16 KB rope block (first, where
//   two warps   there are two rope slots), each page fetched through the block table
//               (2D tiled loads, 128-byte swizzle); the boxes are dealt round-robin to
//               the three warps
//   warp 1      TMEM allocation; its lane 0 alone walks the schedule and issues every
//               MMA (no warp-wide votes or syncs on the path from a landed tile to
//               its MMAs)
//   warps 2-5   softmax (S^T from TMEM -> P^T bf16 into the rope slot), zeroing of
//   (6-9)       V rows past the context (poisoned tails never reach the tensor
//               core), O rescale, and the epilogue (O^T / l -> out or a partial)
// At N = 64, Q and one tile fill shared memory, so a tile's last pair and its rope
// block are fetched only after the previous tile's PV has released their slots.
// Every wait is bounded (see common.cuh); a timeout sets the workspace status
// bit and the CTA unwinds.
#include <math.h>

#include "common.cuh"
#include "kernels.h"
#include "plan.cuh"

namespace splash {
namespace {

constexpr int kSoftmaxThreads = 128;           // threads of one softmax warpgroup
constexpr int kSoftmaxBarrier = 1;             // named barrier id of the first warpgroup
constexpr int kColBlockBytes = kTileTokens * 128;  // one 64-column block of a tile: 16 KB
constexpr int kPairBytes = 2 * kColBlockBytes;
constexpr float kTau = 8.0f;                   // rescale only when a score beats the max by 2^8
// One warp's TMA issue stream moves ~40 GB/s into an SM; the loads are spread over
// kProducerWarps warps so that one SM can ingest a tile at ~3x that rate.
constexpr int kProducerWarps = 3;
#ifndef SPLASH_TRACE_TILE0
#define SPLASH_TRACE_TILE0 0
#endif
constexpr int kTraceTile0 = SPLASH_TRACE_TILE0;  // first tile of a piece the trace stamps

// Whether producer warp pw issues any of the boxes g0 .. g0 + n - 1 (box b belongs to
// warp b % kProducerWarps).
__device__ __forceinline__ bool owns_box(int g0, int n, int pw) {
    return n >= kProducerWarps || (pw - g0 % kProducerWarps + kProducerWarps) % kProducerWarps < n;
}

template <int NPAD>
struct TcConfig {
    static constexpr int kSoftmaxGroups = NPAD == 64 ? 2 : 1;  // warpgroups sharing the heads
    static constexpr int kFirstExtraProducer = 2 + 4 * kSoftmaxGroups;  // warps after the softmax
    static constexpr int kThreads = 32 * (kFirstExtraProducer + kProducerWarps - 1);
    static constexpr int kPairs = NPAD == 64 ? 4 : 5;      // pair slots (ring)
    static constexpr int kRopes = NPAD == 16 ? 2 : 1;      // rope / P^T slots (ring)
    // With two rope slots the next tile's rope slot is free long before its pairs' slots:
    // the rope is then loaded first and contracted first, and only the last pair's MMAs
    // follow the tile's last load.  With one, the slot holds P^T until the PV ends.
    static constexpr bool kRopeFirst = kRopes > 1;
    static constexpr int kQBytes = 9 * NPAD * 128;
    static constexpr int kQOff = 0;
    static constexpr int kPairOff = kQOff + kQBytes;
    static constexpr int kRopeOff = kPairOff + kPairs * kPairBytes;
    static constexpr int kBarOff = kRopeOff + kRopes * kColBlockBytes;
    static constexpr int kNumBars = 2 * kPairs + 2 * kRopes + 7;
    static constexpr int kMiscOff = kBarOff + kNumBars * 8;
    // misc: tmem slot (16 B), abort flag (4 B), CTA status word (4 B), pad, m[NPAD],
    // m_new[NPAD], alpha[NPAD], red[4][NPAD], then the plan scan's 36 int64
    static constexpr int kMiscBytes = 32 + 7 * NPAD * 4;
    static constexpr int kPlanScratchOff = kMiscBytes;
    static constexpr int kPlanScratchBytes = 36 * 8;
    static constexpr int kSmemBytes = kMiscOff + kMiscBytes + kPlanScratchBytes + 1024;  // + alignment slack
    static constexpr int kTmemCols = NPAD == 16 ? 128 : (NPAD == 32 ? 256 : 512);
    static constexpr int kOCol = 0;
    static constexpr int kSCol = 4 * NPAD;
    static_assert(kSmemBytes <= 232448, "shared memory budget");
    static_assert(kSCol + NPAD <= kTmemCols, "TMEM budget");
};

struct TcParams {
    DecodeArgs a;
    float c_log2;        // scale * log2(e): scores in the exp2 domain
    int keep_kv;         // KV loads marked evict-last (a call whose cache fits in L2)
    int group_heads;     // Gs: heads per head group (the last group may have fewer)
    int head_groups;     // NG
};

// Optional phase trace (compiled in only with -DSPLASH_TRACE): globaltimer stamps
// per CTA and event slot, read back with splash_trace_read().
#ifdef SPLASH_TRACE
constexpr int kTraceSlots = 64;
constexpr int kTraceCtas = 1024;
__device__ unsigned long long g_trace[kTraceCtas * kTraceSlots];
#define TRACE(slot)                                                                   \
    do {                                                                              \
        if (blockIdx.x < kTraceCtas && (slot) < kTraceSlots)                          \
            g_trace[blockIdx.x * kTraceSlots + (slot)] = globaltimer_ns();            \
    } while (0)
#else
#define TRACE(slot) \
    do {            \
    } while (0)
#endif

__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Bounded wait by a whole warp; every lane gets the same verdict.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                          uint32_t* status) {
    const bool ok = mbar_wait(bar, parity, abort_flag, status);
    return __all_sync(0xffffffffu, ok);
}

// Reduce-scatter of NV (16 or 32) values per lane across the 32 lanes of a warp:
// afterwards lane L holds the max (or sum) over all lanes of value L for NV = 32,
// and of value (L >> 1) for NV = 16 (lanes 2i and 2i+1 agree).  Each step keeps
// half of the values and trades the other half with the partner lane, so NV = 32
// costs 31 shuffles instead of 32 x 5 for separate all-reduces.
template <int NV, bool MAX>
__device__ __forceinline__ float warp_reduce_scatter(float (&v)[NV], int lane) {
    static_assert(NV == 16 || NV == 32, "16 or 32 values");
#pragma unroll
    for (int step = 0; step < 5; ++step) {
        const int bit = 16 >> step;
        const int k = NV >> (step + 1);
        if (k >= 1) {
            const bool upper = (lane & bit) != 0;
#pragma unroll
            for (int i = 0; i < k; ++i) {
                const float keep = upper ? v[i + k] : v[i];
                const float send = upper ? v[i] : v[i + k];
                const float recv = __shfl_xor_sync(0xffffffffu, send, bit);
                v[i] = MAX ? fmaxf(keep, recv) : keep + recv;
            }
        }
    }
    float r = v[0];
    if (NV == 16) {
        const float o = __shfl_xor_sync(0xffffffffu, r, 1);
        r = MAX ? fmaxf(r, o) : r + o;
    }
    return r;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}

template <int NPAD>
__global__ void __launch_bounds__(TcConfig<NPAD>::kThreads, 1)
    mla_decode_tc_kernel(const __grid_constant__ CUtensorMap map_q,
                         const __grid_constant__ CUtensorMap map_kv, const TcParams prm) {
    using C = TcConfig<NPAD>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~uintptr_t(1023));
    uint8_t* sQ = smem + C::kQOff;
    uint8_t* sPair = smem + C::kPairOff;
    uint8_t* sRope = smem + C::kRopeOff;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kBarOff);
    uint64_t* pair_full = bars;
    uint64_t* pair_empty = bars + C::kPairs;
    uint64_t* rope_full = bars + 2 * C::kPairs;
    uint64_t* rope_empty = rope_full + C::kRopes;
    uint64_t* q_full = rope_empty + C::kRopes;
    uint64_t* q_empty = q_full + 1;
    uint64_t* s_full = q_full + 2;
    uint64_t* p_full = q_full + 3;
    uint64_t* o_full = q_full + 4;
    uint64_t* o_free = q_full + 5;
    uint64_t* drain = q_full + 6;
    uint8_t* misc = smem + C::kMiscOff;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(misc);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(misc + 16);
    uint32_t* cta_status_smem = reinterpret_cast<uint32_t*>(misc + 20);
    int64_t* plan_scratch = reinterpret_cast<int64_t*>(misc + C::kPlanScratchOff);
    float* sm_m = reinterpret_cast<float*>(misc + 32);
    float* sm_mnew = sm_m + NPAD;
    float* sm_alpha = sm_mnew + NPAD;
    float* sm_red = sm_alpha + NPAD;  // [4][NPAD]

    const DecodeArgs& a = prm.a;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    uint8_t* ws = static_cast<uint8_t*>(a.ws);
    const WorkspaceLayout lay(a.B, a.Hs, a.num_groups, a.sts_cap);
    // this CTA's status bits collect in shared memory and go to its own workspace word at
    // the end (the combine kernel ORs the words into the header: no word is shared, so
    // none needs clearing before the call)
    uint32_t* status = cta_status_smem;
    const int NG = prm.head_groups;
    const int j = blockIdx.x / NG, g = blockIdx.x % NG;
    const int hbase = g * prm.group_heads;                  // first head of the group in the slice
    const int nh = min(prm.group_heads, a.Hs - hbase);      // valid heads of the group
    const int P = a.P;
    const int pages_per_tile = kTileTokens / P;
    // the head group lies within one KV head's group of query heads (checked on the
    // host); page p of that KV head starts at row (p * kv_heads + kvh) * P of the pool
    const int kvh = a.kv_heads > 1 ? (a.head_lo + hbase) / a.q_per_kv : 0;

    // Prologue (overlaps the previous kernel on the stream under programmatic dependent
    // launch: nothing here reads global memory).
    if (threadIdx.x == 0) TRACE(0);
    if (threadIdx.x == 0) {
        for (int i = 0; i < C::kPairs; ++i) {
            mbar_init(&pair_full[i], 1);
            mbar_init(&pair_empty[i], 1);
        }
        for (int i = 0; i < C::kRopes; ++i) {
            mbar_init(&rope_full[i], 1);
            mbar_init(&rope_empty[i], 1);
        }
        mbar_init(q_full, 1);
        mbar_init(q_empty, 1);
        mbar_init(s_full, 1);
        mbar_init(p_full, kSoftmaxThreads * C::kSoftmaxGroups);
        mbar_init(o_full, 1);
        mbar_init(o_free, kSoftmaxThreads * C::kSoftmaxGroups);
        mbar_init(drain, 1);
        *abort_flag = 0;
        *cta_status_smem = 0;
        fence_barrier_init();
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, C::kTmemCols);
        tmem_relinquish();
    }
    if (warp == 0 && lane == 0) {
        prefetch_tensormap(&map_q);
        prefetch_tensormap(&map_kv);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (threadIdx.x == 0) TRACE(1);
    pdl_wait();     // every earlier kernel on the stream is complete (inputs are final)
    if (threadIdx.x == 0) TRACE(2);
    // the split plan: every CTA scans the requests; CTA 0 also writes the request plans
    // and the header into the workspace
    const PlanStart plan = plan_prologue(a, j, blockIdx.x == 0, C::kThreads, plan_scratch, status);
    const int64_t T = plan.T;
    const int64_t G = plan.G;       // groups in use (<= a.num_groups, <= T)
    const int64_t aj = (T > 0 && j < G) ? group_start(j, T, G) : 0;
    const int64_t bj = (T > 0 && j < G) ? group_start(j + 1, T, G) : 0;

    if (warp == 0 || warp >= C::kFirstExtraProducer) {
        // ------------------------------------------------------------ TMA producers
        // kProducerWarps warps walk the same schedule (each whole warp, so it stays
        // converged); load slot k of a tile (pairs 0-3, then the rope block) and Q box k
        // belong to producer warp k % kProducerWarps, whose lanes issue them.  A box may
        // complete before its slot's expect-tx (transaction counts may go negative while
        // the expect-tx arrival is pending), so no warp sync separates the two.
        const int pw = warp == 0 ? 0 : warp - C::kFirstExtraProducer + 1;
        if (aj < bj) {
            // a small cache stays in L2 for the next kernels (the sibling head group, a
            // handoff, the next call); a large stream must not push everything else out
            const uint64_t pol_kv = prm.keep_kv ? policy_evict_last() : policy_evict_first();
            const uint64_t pol_q = policy_evict_last();
            int ps = 0, pph = 0, rs = 0, rph = 0, qph = 0;
            PieceIter it(a, plan, aj, bj, j);
            Piece pc;
            ReqPlan p;
            bool ok = true;
            while (ok && it.next(pc, p)) {
                if (!warp_wait(q_empty, qph ^ 1, abort_flag, status)) { ok = false; break; }
                qph ^= 1;
                if (lane == 0) {
                    if (pw == 0) mbar_arrive_expect_tx(q_full, C::kQBytes);
                    const int qrow = pc.row * a.H + a.head_lo + hbase;
                    for (int cb = pw; cb < 9; cb += kProducerWarps)
                        tma_load_2d(sQ + cb * NPAD * 128, &map_q, q_full, cb * 64, qrow, pol_q);
                    if (pw == 0) TRACE(3);
                }
                __syncwarp();
                int ttr = -kTraceTile0;
                const int32_t* bt = a.block_table + int64_t(pc.row) * a.max_pages;
                for (int t = pc.t_lo; t < pc.t_hi && ok; ++t) {
                    const int tok0 = (p.tile0 + t) * kTileTokens;
                    // lane k < pages_per_tile looks up page k of the tile
                    int my_pid = -1;
                    bool bad = false;
                    if (lane < pages_per_tile) {
                        const int ptok = tok0 + lane * P;
                        if (ptok < p.ctx_len) {
                            const int id = bt[ptok / P];
                            if (id >= 0 && id < a.num_pages) my_pid = id;
                            else bad = true;
                        }
                    }
                    const uint32_t present = __ballot_sync(0xffffffffu, my_pid >= 0);
                    if (pw == 0 && __any_sync(0xffffffffu, bad) && lane == 0)
                        atomicOr(status, uint32_t(SPLASH_DEVICE_BAD_INPUT));
                    const uint32_t blk_bytes = uint32_t(__popc(present)) * P * 128;
                    if (pw == 0 && lane == 0 && unsigned(ttr) < 3u) TRACE(4 + ttr * 3);
                    // box b of the tile (pair jj, page k, column block c2: b = jj * bpp + 2k + c2;
                    // rope block of page k: b = 4 * bpp + k) is issued by producer warp
                    // b % kProducerWarps, so the boxes that wait for the last PV of the
                    // previous tile (pair 3 and the rope) spread over all producer warps
                    const int bpp = 2 * pages_per_tile;  // boxes per pair
                    // the rope block of page k is box 4 * bpp + k
                    auto issue_rope = [&]() -> bool {
                        const int g0 = 4 * bpp;
                        if (owns_box(g0, pages_per_tile, pw)) {
                            if (!warp_wait(&rope_empty[rs], rph ^ 1, abort_flag, status)) return false;
                            if (lane == 0 && g0 % kProducerWarps == pw)
                                mbar_arrive_expect_tx(&rope_full[rs], blk_bytes);
                            if (my_pid >= 0 && (g0 + lane) % kProducerWarps == pw)
                                tma_load_2d(sRope + rs * kColBlockBytes + lane * P * 128, &map_kv,
                                            &rope_full[rs], 8 * 64, (my_pid * a.kv_heads + kvh) * P,
                                            pol_kv);
                            if (pw == g0 % kProducerWarps && lane == 0 && unsigned(ttr) < 3u)
                                TRACE(6 + ttr * 3);
                        }
                        return true;
                    };
                    if (C::kRopeFirst && !issue_rope()) { ok = false; break; }
                    for (int jj = 0; jj < 4; ++jj) {
                        const int g0 = jj * bpp;
                        if (owns_box(g0, bpp, pw)) {
                            if (!warp_wait(&pair_empty[ps], pph ^ 1, abort_flag, status)) { ok = false; break; }
                            if (lane == 0 && g0 % kProducerWarps == pw) {
                                mbar_arrive_expect_tx(&pair_full[ps], 2 * blk_bytes);
                                if (ttr == 1) TRACE(55 + jj);
                            }
                            uint8_t* slot = sPair + ps * kPairBytes;
                            if (my_pid >= 0)
                                for (int c2 = 0; c2 < 2; ++c2)
                                    if ((g0 + 2 * lane + c2) % kProducerWarps == pw)
                                        tma_load_2d(slot + c2 * kColBlockBytes + lane * P * 128, &map_kv,
                                                    &pair_full[ps], (2 * jj + c2) * 64,
                                                    (my_pid * a.kv_heads + kvh) * P, pol_kv);
                        }
                        if (++ps == C::kPairs) { ps = 0; pph ^= 1; }
                    }
                    if (!ok) break;
                    if (pw == 0 && lane == 0 && unsigned(ttr) < 3u) TRACE(5 + ttr * 3);
                    if (!C::kRopeFirst && !issue_rope()) { ok = false; break; }
                    ++ttr;
                    if (++rs == C::kRopes) { rs = 0; rph ^= 1; }
                }
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        // Lane 0 alone walks the schedule and issues every tcgen05 instruction (the
        // other lanes go straight to the teardown barrier).
        if (lane == 0 && aj < bj) {
            constexpr uint32_t idesc_qk = idesc_bf16_f32(128, NPAD, false, false);
            constexpr uint32_t idesc_pv = idesc_bf16_f32(128, NPAD, true, true);
            const uint32_t s_tmem = tmem + C::kSCol;
            const uint32_t o_tmem = tmem + C::kOCol;
            // Descriptor bases, computed once: a descriptor for a given start address is the
            // base plus (byte offset >> 4) in its low field (shared addresses < 256 KB), which
            // keeps the issue loop to one add per operand.
            const uint64_t dq0 = smem_desc(smem_u32(sQ), 16, 1024, 2);               // Q, K-major
            const uint64_t dk0 = smem_desc(smem_u32(sPair), 16, 1024, 2);            // K tile, K-major
            const uint64_t dr0 = smem_desc(smem_u32(sRope), 16, 1024, 2);            // rope, K-major
            const uint64_t dv0 = smem_desc(smem_u32(sPair), kColBlockBytes, 1024, 2); // V^T, MN-major
            const uint64_t dp0 = smem_desc(smem_u32(sRope), 1024, 1024, 2);          // P^T, MN-major
            int ps = 0, pph = 0, rs = 0, rph = 0, qph = 0, pfph = 0, ofph = 0;
            PieceIter it(a, plan, aj, bj, j);
            Piece pc;
            ReqPlan p;
            bool ok = true;
            while (ok && it.next(pc, p)) {
                if (!mbar_wait(q_full, qph, abort_flag, status)) { ok = false; break; }
                qph ^= 1;
                int ttr = -kTraceTile0;
                for (int t = pc.t_lo; t < pc.t_hi; ++t) {
                    const bool first = (t == pc.t_lo), last = (t + 1 == pc.t_hi);
                    const int ps0 = ps;
                    if (lane == 0 && unsigned(ttr) < 3u) TRACE(13 + ttr * 5);
                    // S^T = K_tile . Q^T over the 64 rope dims (first, when the rope is
                    // loaded first) and the 512 latent dims (pairs)
                    auto rope_mmas = [&](bool overwrite) -> bool {
                        if (!mbar_wait(&rope_full[rs], rph, abort_flag, status)) return false;
                        if (lane == 0 && unsigned(ttr) < 3u) TRACE(14 + ttr * 5);
                        tc_fence_after();
                        if (lane == 0) {
                            const uint64_t da_r = dr0 + uint64_t(rs) * (kColBlockBytes >> 4);
#pragma unroll
                            for (int k4 = 0; k4 < 4; ++k4)
                                mma_bf16_ss(s_tmem, da_r + ((k4 * 32) >> 4),
                                            dq0 + ((8 * NPAD * 128 + k4 * 32) >> 4), idesc_qk,
                                            (!overwrite || k4 > 0) ? 1u : 0u);
                        }
                        return true;
                    };
                    if (C::kRopeFirst && !rope_mmas(true)) { ok = false; break; }
                    for (int jj = 0; jj < 4; ++jj) {
                        if (!mbar_wait(&pair_full[ps], pph, abort_flag, status)) { ok = false; break; }
                        if (lane == 0 && ttr == 1) TRACE(51 + jj);
                        tc_fence_after();
                        if (lane == 0) {
                            const uint64_t da_s = dk0 + uint64_t(ps) * (kPairBytes >> 4);
                            const uint64_t db_s = dq0 + uint64_t(jj) * (2 * NPAD * 128 >> 4);
#pragma unroll
                            for (int c2 = 0; c2 < 2; ++c2)
#pragma unroll
                                for (int k4 = 0; k4 < 4; ++k4)
                                    mma_bf16_ss(s_tmem, da_s + ((c2 * kColBlockBytes + k4 * 32) >> 4),
                                                db_s + ((c2 * NPAD * 128 + k4 * 32) >> 4), idesc_qk,
                                                (C::kRopeFirst || (jj | c2 | k4) != 0) ? 1u : 0u);
                        }
                        if (++ps == C::kPairs) { ps = 0; pph ^= 1; }
                    }
                    if (!ok) break;
                    if (!C::kRopeFirst && !rope_mmas(false)) { ok = false; break; }
                    if (lane == 0) {
                        tc_commit(s_full);
                        if (last) tc_commit(q_empty);
                        if (unsigned(ttr) < 3u) TRACE(15 + ttr * 5);
                    }
                    // O^T += V^T . P^T once the softmax has written P^T into the rope slot
                    if (!mbar_wait(p_full, pfph, abort_flag, status)) { ok = false; break; }
                    pfph ^= 1;
                    if (lane == 0 && unsigned(ttr) < 3u) TRACE(16 + ttr * 5);
                    if (first) {
                        if (!mbar_wait(o_free, ofph ^ 1, abort_flag, status)) { ok = false; break; }
                        ofph ^= 1;
                    }
                    tc_fence_after();
                    if (lane == 0) {
                        const uint64_t db_p = dp0 + uint64_t(rs) * (kColBlockBytes >> 4);
                        // kept rolled: the 8-MMA body is fetched once, not 4 times cold
#pragma unroll 1
                        for (int jj = 0; jj < 4; ++jj) {
                            const int pslot = (ps0 + jj) % C::kPairs;
                            const uint64_t da_v = dv0 + uint64_t(pslot) * (kPairBytes >> 4);
#pragma unroll
                            for (int kk = 0; kk < 8; ++kk) {
                                mma_bf16_ss(o_tmem + jj * NPAD, da_v + ((kk * 2048) >> 4),
                                            db_p + ((kk * 2048) >> 4), idesc_pv,
                                            (!first || kk > 0) ? 1u : 0u);
                                if (jj == 0 && kk == 0 && unsigned(ttr) < 2u) TRACE(43 + ttr * 4);
                            }
                            tc_commit(&pair_empty[pslot]);
                            if (jj == 0 && unsigned(ttr) < 2u) TRACE(44 + ttr * 4);
                            if (jj == 1 && unsigned(ttr) < 2u) TRACE(45 + ttr * 4);
                            if (jj == 2 && unsigned(ttr) < 2u) TRACE(46 + ttr * 4);

                        }
                        tc_commit(&rope_empty[rs]);
                        if (last) tc_commit(o_full);
                        if (unsigned(ttr) < 3u) TRACE(17 + ttr * 5);
                    }
                    ++ttr;
                    if (++rs == C::kRopes) { rs = 0; rph ^= 1; }
                }
            }
            // drain: every MMA issued so far has completed before TMEM is released.  The
            // wait is bounded like every other; if it gives up, the status word already
            // says SPLASH_DEVICE_TIMEOUT (the call's outputs are invalid) and the CTA still
            // deallocates at the teardown: an allocation must not outlive its CTA, and a
            // tensor pipe that has not finished 2 s after its last issue is the fault the
            // status word reports, not a state the kernel can wait out.
            tc_commit(drain);
            volatile int never = 0;
            mbar_wait(drain, 0, &never, status);
        }
        __syncwarp();   // warp 1 reconverges before the teardown barrier and dealloc
    } else {
        // ------------------------------------------------------------ softmax + epilogue
        // SWG softmax warpgroups; group wg owns heads [hw0, hw0 + HW) of the head group
        constexpr int SWG = C::kSoftmaxGroups;
        constexpr int HW = NPAD / SWG;
        const int st = (threadIdx.x - 64) & 127;      // 0..127 within the warpgroup
        const int wg = (threadIdx.x - 64) >> 7;
        const int hw0 = wg * HW;
        const int bar = kSoftmaxBarrier + wg;         // named barrier of this warpgroup
        const int quad = warp & 3;                    // TMEM lane quadrant of this warp
        const int row = quad * 32 + lane;             // token row of S^T, dv row of O^T
        const uint32_t lane_off = uint32_t(quad * 32) << 16;
        const uint32_t s_tmem = tmem + C::kSCol + lane_off;
        const uint32_t o_tmem = tmem + C::kOCol + lane_off;
        const float cl = prm.c_log2;
        float* pout = reinterpret_cast<float*>(ws + lay.pout_off);
        float* plse = reinterpret_cast<float*>(ws + lay.plse_off);
        int sph = 0, ofl = 0, rs = 0;
        int ps_base = 0;      // pair slot of the tile's pair 0 (mirrors the MMA ring)
        PieceIter it(a, plan, aj, bj, j);
        Piece pc;
        ReqPlan p;
        bool ok = aj < bj;
        while (ok && it.next(pc, p)) {
            named_barrier_sync(bar, kSoftmaxThreads);
            if (st < HW) sm_m[hw0 + st] = -INFINITY;
            named_barrier_sync(bar, kSoftmaxThreads);
            float lpart[HW];
#pragma unroll
            for (int h = 0; h < HW; ++h) lpart[h] = 0.f;
            const int32_t* bt = a.block_table + int64_t(pc.row) * a.max_pages;
            for (int t = pc.t_lo; t < pc.t_hi; ++t) {
                const bool first = (t == pc.t_lo);
                const int tok = (p.tile0 + t) * kTileTokens + row;
                bool in_ctx = tok < p.ctx_len;
                if (in_ctx) {
                    const int id = bt[tok / P];
                    in_ctx = id >= 0 && id < a.num_pages;
                }
                // a token of an unreadable page (bad id) is left out of the attention: its
                // key rows in shared memory are whatever the slot held before
                const bool valid = tok >= p.lo && tok < p.hi && in_ctx;
                bool w = mbar_wait(s_full, sph, abort_flag, status);
                if (named_barrier_or(bar, kSoftmaxThreads, !w)) { ok = false; break; }
                sph ^= 1;
                tc_fence_after();
                const int ttr = t - pc.t_lo - kTraceTile0;
                if (threadIdx.x == 64 && unsigned(ttr) < 3u) TRACE(28 + ttr * 4);
                // the tile's scores of this thread's token for the group's heads, read once
                float sv[HW / 16][16];
#pragma unroll
                for (int c = 0; c < HW / 16; ++c) tmem_ld16(s_tmem + hw0 + c * 16, sv[c]);
                tmem_wait_ld();
                // pass 1: does any valid score exceed the running max by more than tau?
                float excess = -INFINITY;
#pragma unroll
                for (int c = 0; c < HW / 16; ++c)
#pragma unroll
                    for (int e = 0; e < 16; ++e)
                        excess = fmaxf(excess, sv[c][e] * cl - sm_m[hw0 + c * 16 + e]);
                if (!valid) excess = -INFINITY;
                const bool rescale = named_barrier_or(bar, kSoftmaxThreads, excess > kTau);
                if (threadIdx.x == 64 && unsigned(ttr) < 3u) TRACE(29 + ttr * 4);
                if (rescale) {
                    // exact column max over the tile's valid tokens: warp reduce-scatter in
                    // chunks of up to 32 heads, then the 4 warps through shared memory
                    constexpr int RS = HW < 32 ? HW : 32;
#pragma unroll
                    for (int i0 = 0; i0 < HW; i0 += RS) {
                        float v[RS];
#pragma unroll
                        for (int i = 0; i < RS; ++i)
                            v[i] = valid ? sv[(i0 + i) / 16][(i0 + i) % 16] * cl : -INFINITY;
                        const float m = warp_reduce_scatter<RS, true>(v, lane);
                        const int h0 = hw0 + i0;
                        if (RS == 32) sm_red[quad * NPAD + h0 + lane] = m;
                        else if ((lane & 1) == 0) sm_red[quad * NPAD + h0 + (lane >> 1)] = m;
                    }
                    named_barrier_sync(bar, kSoftmaxThreads);
                    if (st < HW) {
                        const int h = hw0 + st;
                        const float mo = sm_m[h];
                        float mn = fmaxf(fmaxf(sm_red[h], sm_red[NPAD + h]),
                                         fmaxf(sm_red[2 * NPAD + h], sm_red[3 * NPAD + h]));
                        mn = fmaxf(mn, mo);
                        sm_mnew[h] = mn;
                        sm_alpha[h] = (mo == -INFINITY) ? 0.f : ex2_approx(mo - mn);
                    }
                    named_barrier_sync(bar, kSoftmaxThreads);
#pragma unroll
                    for (int h = 0; h < HW; ++h) lpart[h] *= sm_alpha[hw0 + h];
                    if (!first) {
                        // O^T columns are heads: scale column h of every dv block by alpha_h
#pragma unroll 1
                        for (int jj = 0; jj < 4; ++jj)
#pragma unroll 1
                            for (int c = 0; c < HW / 16; ++c) {
                                float o[16];
                                tmem_ld16(o_tmem + jj * NPAD + hw0 + c * 16, o);
                                tmem_wait_ld();
#pragma unroll
                                for (int e = 0; e < 16; ++e) o[e] *= sm_alpha[hw0 + c * 16 + e];
                                tmem_st16(o_tmem + jj * NPAD + hw0 + c * 16, o);
                            }
                        tmem_wait_st();
                    }
                    named_barrier_sync(bar, kSoftmaxThreads);
                    if (st < HW) sm_m[hw0 + st] = sm_mnew[hw0 + st];
                    named_barrier_sync(bar, kSoftmaxThreads);
                }
                if (threadIdx.x == 64 && unsigned(ttr) < 3u) TRACE(30 + ttr * 4);
                // pass 2: P^T row = exp2(s * c - m) as bf16 into the rope slot (MN-major,
                // 128-byte swizzle: 16-byte chunk ch of row r sits at chunk ch ^ (r & 7))
                uint8_t* prow = sRope + rs * kColBlockBytes + row * 128;
#pragma unroll
                for (int c = 0; c < HW / 16; ++c) {
                    uint32_t pk[8];
#pragma unroll
                    for (int e = 0; e < 16; e += 2) {
                        float p0 = valid ? ex2_approx(sv[c][e] * cl - sm_m[hw0 + c * 16 + e]) : 0.f;
                        float p1 = valid ? ex2_approx(sv[c][e + 1] * cl - sm_m[hw0 + c * 16 + e + 1]) : 0.f;
                        pk[e / 2] = pack_bf16x2(p0, p1);
                        lpart[c * 16 + e] += p0;       // l from the unrounded fp32 P
                        lpart[c * 16 + e + 1] += p1;
                    }
                    const int ch0 = (hw0 >> 3) + 2 * c, ch1 = ch0 + 1;
                    *reinterpret_cast<uint4*>(prow + ((ch0 ^ (row & 7)) << 4)) =
                        make_uint4(pk[0], pk[1], pk[2], pk[3]);
                    *reinterpret_cast<uint4*>(prow + ((ch1 ^ (row & 7)) << 4)) =
                        make_uint4(pk[4], pk[5], pk[6], pk[7]);
                }
                // rows outside the context (or of unreadable pages) hold arbitrary bits:
                // zero them in the V blocks so 0 * NaN never reaches the accumulator
                if (!in_ctx && wg == 0) {
                    const uint4 z = make_uint4(0u, 0u, 0u, 0u);
                    for (int jj = 0; jj < 4; ++jj) {
                        uint8_t* slot = sPair + ((ps_base + jj) % C::kPairs) * kPairBytes + row * 128;
#pragma unroll
                        for (int c2 = 0; c2 < 2; ++c2)
#pragma unroll
                            for (int ch = 0; ch < 8; ++ch)
                                *reinterpret_cast<uint4*>(slot + c2 * kColBlockBytes + ch * 16) = z;
                    }
                }
                ps_base = (ps_base + 4) % C::kPairs;
                if (++rs == C::kRopes) rs = 0;
                fence_proxy_async_smem();
                tc_fence_before();
                mbar_arrive(p_full);
                if (threadIdx.x == 64 && unsigned(ttr) < 3u) TRACE(31 + ttr * 4);
            }
            if (!ok) break;
            // ---------------------------------------------------------- epilogue
            bool w = mbar_wait(o_full, ofl, abort_flag, status);
            if (named_barrier_or(bar, kSoftmaxThreads, !w)) { ok = false; break; }
            ofl ^= 1;
            if (threadIdx.x == 64) TRACE(40);
            tc_fence_after();
            // l_h = sum over the 128 token lanes of the per-lane partial sums
            {
                constexpr int RS = HW < 32 ? HW : 32;
#pragma unroll
                for (int h0 = 0; h0 < HW; h0 += RS) {
                    float v[RS];
#pragma unroll
                    for (int i = 0; i < RS; ++i) v[i] = lpart[h0 + i];
                    const float sum = warp_reduce_scatter<RS, false>(v, lane);
                    if (RS == 32) sm_red[quad * NPAD + hw0 + h0 + lane] = sum;
                    else if ((lane & 1) == 0) sm_red[quad * NPAD + hw0 + h0 + (lane >> 1)] = sum;
                }
            }
            named_barrier_sync(bar, kSoftmaxThreads);
            if (st < HW) {
                const int h = hw0 + st;
                sm_alpha[h] = 1.0f / (sm_red[h] + sm_red[NPAD + h] + sm_red[2 * NPAD + h] +
                                      sm_red[3 * NPAD + h]);
            }
            named_barrier_sync(bar, kSoftmaxThreads);
            float* obase;
            float* lbase;
            int64_t hstride;
            if (p.nsplit == 1) {
                obase = a.out + (int64_t(pc.row) * a.H + a.head_lo + hbase) * kDv;
                lbase = a.lse + int64_t(pc.row) * a.H + a.head_lo + hbase;
            } else {
                const int64_t slot = p.slot_base + pc.split;
                obase = pout + (slot * a.Hs + hbase) * kDv;
                lbase = plse + slot * a.Hs + hbase;
            }
            hstride = kDv;
            // per 16 heads: the four dv blocks' loads are in flight together, then stored
#pragma unroll 1
            for (int c = 0; c < HW / 16; ++c) {
                const int hc = hw0 + c * 16;
                float o[4][16];
#pragma unroll
                for (int jj = 0; jj < 4; ++jj) tmem_ld16(o_tmem + jj * NPAD + hc, o[jj]);
                float inv[16];
#pragma unroll
                for (int e = 0; e < 16; ++e) inv[e] = sm_alpha[hc + e];
                float* ocol = obase + int64_t(hc) * hstride + row;
                tmem_wait_ld();
#pragma unroll
                for (int jj = 0; jj < 4; ++jj)
#pragma unroll
                    for (int e = 0; e < 16; ++e)
                        if (hc + e < nh) ocol[e * hstride + jj * 128] = o[jj][e] * inv[e];
            }
            if (st < HW && hw0 + st < nh) {
                const int h = hw0 + st;
                lbase[h] = (sm_m[h] - log2f(sm_alpha[h])) * 0.69314718055994531f;
            }
            tc_fence_before();
            mbar_arrive(o_free);
            if (threadIdx.x == 64) TRACE(41);
        }
    }

    // only now may the combine grid launch: launched at the start, its waiting CTAs would
    // hold the SMs that a decode call on another stream needs
    pdl_trigger();
    tc_fence_before();
    __syncthreads();
    if (threadIdx.x == 0)
        reinterpret_cast<uint32_t*>(ws + lay.sts_off)[blockIdx.x] = *cta_status_smem;
    if (threadIdx.x == 0) TRACE(42);
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, C::kTmemCols);
    }
}

template <int NPAD>
cudaError_t launch_tc(const CUtensorMap& mq, const CUtensorMap& mkv, const TcParams& prm,
                      int grid, cudaStream_t stream) {
    using C = TcConfig<NPAD>;
    cudaError_t e = ensure_smem_optin(reinterpret_cast<const void*>(mla_decode_tc_kernel<NPAD>),
                                      C::kSmemBytes);
    if (e != cudaSuccess) return e;
    return launch_pdl(mla_decode_tc_kernel<NPAD>, dim3(grid), dim3(C::kThreads), size_t(C::kSmemBytes),
                      stream, mq, mkv, prm);
}

}  // namespace

#ifdef SPLASH_TRACE
extern "C" __attribute__((visibility("default"))) int splash_trace_read(void* host_dst, size_t bytes) {
    if (bytes > sizeof(g_trace)) bytes = sizeof(g_trace);
    return cudaMemcpyFromSymbol(host_dst, g_trace, bytes) == cudaSuccess ? 0 : -1;
}
extern "C" __attribute__((visibility("default"))) int splash_trace_clear() {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_trace) != cudaSuccess) return -1;
    return cudaMemset(p, 0, sizeof(g_trace)) == cudaSuccess ? 0 : -1;
}
#endif

int tc_pad_heads(int group_heads) {
    return group_heads <= 16 ? 16 : (group_heads <= 32 ? 32 : 64);
}

cudaError_t launch_decode_tc(const DecodeArgs& a, const CUtensorMap& map_q,
                             const CUtensorMap& map_kv, int head_groups, int group_heads,
                             cudaStream_t stream) {
    TcParams prm;
    prm.a = a;
    prm.c_log2 = a.scale * 1.4426950408889634f;
    prm.group_heads = group_heads;
    prm.head_groups = head_groups;
    // every page the call could read (the capacity of its block tables) within 48 MB
    const double kv_bound = double(a.B) * a.max_pages * a.P * a.kv_heads * (kDqk * 2);
    prm.keep_kv = kv_bound <= 48.0 * 1024 * 1024;
    const int grid = a.num_groups * head_groups;
    switch (tc_pad_heads(group_heads)) {
        case 16: return launch_tc<16>(map_q, map_kv, prm, grid, stream);
        case 32: return launch_tc<32>(map_q, map_kv, prm, grid, stream);
        default: return launch_tc<64>(map_q, map_kv, prm, grid, stream);
    }
}

}  // namespace splash
