// common.cuh -- shared device helpers of the GB300 (sm_103a) decode library:
// workspace layout, bounded mbarrier waits, TMA and tcgen05 inline-PTX wrappers.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "splash.h"

namespace splash {

constexpr int kDqk = 576;        // 512 latent + 64 rope dims of the one shared KV head
constexpr int kDv = 512;         // values are the latent prefix of the key
constexpr int kTileTokens = 128; // token tile of every decode kernel (the MMA M)

// ---------------------------------------------------------------------------
// Decode workspace layout (all offsets 256-byte aligned):
//   [0, 256)                PlanHeader
//   [256, ...)              ReqPlan[B]
//   cta_status              uint32 [sts_cap]: SPLASH_DEVICE_* bits of each decode CTA
//                           (sts_cap: the device's SM count rounded up to 64, or the
//                           grid if larger, so the layout does not depend on the grid)
//   partial_out             fp32 [max_slots][Hs][512]
//   partial_lse             fp32 [max_slots][Hs]
// ---------------------------------------------------------------------------
struct PlanHeader {
    uint32_t status;       // SPLASH_DEVICE_* bits of the last call (OR of the CTAs' words)
    int32_t num_groups;    // CTA groups in use (<= G', <= T); the tile sequence is cut in that many ranges
    int64_t total_tiles;   // T: tiles over all requests
    int32_t num_reqs;
    int32_t heads;         // Hs = head_hi - head_lo
    int32_t max_slots;
    int32_t slots_used;
};

struct ReqPlan {
    int64_t tile_begin;    // first tile of the request in the concatenated sequence
    int32_t tile0;         // absolute index (token / 128) of the request's first tile
    int32_t ntiles;        // tiles covering [lo, hi)
    int32_t lo, hi;        // clipped token range, hi <= ctx_len; empty when hi <= lo
    int32_t ctx_len;
    int32_t first_grp;     // CTA group holding the request's first tile
    int32_t nsplit;        // number of CTA groups the request is cut across (0: empty)
    int32_t slot_base;     // first partial slot (only when nsplit > 1), else -1
    int32_t row;           // storage row of q / block_table / ctx_lens / out / lse (-1: none)
    int32_t pad;
};
static_assert(sizeof(ReqPlan) == 48, "ReqPlan layout");

__host__ __device__ inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// Capacity of the per-CTA status array for a device with `sms` SMs and a grid of `ctas`.
__host__ __device__ inline int status_capacity(int sms, int ctas) {
    const int n = sms > ctas ? sms : ctas;
    return (n + 63) / 64 * 64;
}

struct WorkspaceLayout {
    size_t req_off, sts_off, pout_off, plse_off, total;
    int max_slots;
    __host__ __device__ WorkspaceLayout(int B, int Hs, int num_groups, int sts_cap) {
        max_slots = B + num_groups;
        req_off = 256;
        sts_off = align256(req_off + sizeof(ReqPlan) * size_t(B));      // uint32 [sts_cap]
        pout_off = align256(sts_off + sizeof(uint32_t) * size_t(sts_cap));
        plse_off = align256(pout_off + size_t(max_slots) * Hs * kDv * sizeof(float));
        total = align256(plse_off + size_t(max_slots) * Hs * sizeof(float));
    }
};

// One piece of a CTA group's share of the tile sequence: a request, or the part of it
// that falls in the group's tile range.
struct Piece {
    int r;            // request of the call (plan order)
    int row;          // its storage row in q / block_table / out / lse
    int t_lo, t_hi;   // tiles of the request (relative to its first tile)
    int split;
    bool valid;
};

// CTA group j of G' owns tiles [a_j, a_{j+1}) of the T-tile sequence, a_j = floor(j T / G').
__host__ __device__ inline int64_t group_start(int64_t j, int64_t T, int64_t G) { return (j * T) / G; }
// The group holding tile x (0 <= x < T): the largest j with a_j <= x.
__host__ __device__ inline int64_t group_of_tile(int64_t x, int64_t T, int64_t G) {
    return ((x + 1) * G - 1) / T;
}

// ---------------------------------------------------------------------------
// Bounded waiting.  Every spin in these kernels gives up after kWaitLimitNs of
// wall time, records SPLASH_DEVICE_TIMEOUT in the workspace status word and
// lets the kernel unwind (no trap, no unbounded loop).
// ---------------------------------------------------------------------------
constexpr uint64_t kWaitLimitNs = 2000000000ull; // 2 s

__device__ __forceinline__ uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_barrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}

// One potentially blocking test of a phase, with the hardware's own short suspend
// limit (measured faster than a long suspend-time hint when the phase completes soon).
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(bar), "r"(parity)
        : "memory");
    return done != 0;
}

// Waits for phase `parity` of `bar` to complete.  Returns false (and raises the
// CTA abort flag and the workspace status bit) if the wait ran out of time or
// another role of the CTA already aborted.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                          uint32_t* status) {
    const uint32_t a = smem_u32(bar);
    if (mbar_try_wait(a, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t it = 0;; ++it) {
        if (mbar_try_wait(a, parity)) return true;
        if ((it & 63) == 63) {
            if (*abort_flag) return false;
            if (globaltimer_ns() - t0 > kWaitLimitNs) {
                *abort_flag = 1;
                if (status) atomicOr(status, (uint32_t)SPLASH_DEVICE_TIMEOUT);
                return false;
            }
        }
    }
}

// ---------------------------------------------------------------------------
// TMA (cp.async.bulk.tensor) -- 2D tiled loads into this CTA's shared memory.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void tma_load_2d(void* smem_dst, const CUtensorMap* map, uint64_t* bar,
                                            int32_t x, int32_t y, uint64_t cache_policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%3, %4}], [%2], %5;" ::"r"(smem_u32(smem_dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(x), "r"(y), "l"(cache_policy)
        : "memory");
}

__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap* map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

__device__ __forceinline__ uint64_t policy_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ __forceinline__ uint64_t policy_evict_last() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// Generic-proxy shared-memory writes -> visible to the async proxy (tensor core / TMA).
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ---------------------------------------------------------------------------
// tcgen05: tensor memory, MMA, commit, loads / stores
// ---------------------------------------------------------------------------
__device__ __forceinline__ void tmem_alloc(uint32_t* smem_dst, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(smem_dst)),
                 "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[smem desc] * B[smem desc]^T, kind::f16 (bf16 inputs, fp32 accumulate).
__device__ __forceinline__ void mma_bf16_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                            uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrive (once) on `bar` when every tcgen05 operation issued so far by this thread completes.
__device__ __forceinline__ void tc_commit(uint64_t* bar) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
            smem_u32(bar))
        : "memory");
}

// 32 lanes x 32 bit, 16 consecutive columns: thread i of the warp gets lane (base lane + i).
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%"
        "15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const float (&v)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%"
        "14,%15,%16};" ::"r"(taddr),
        "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
        "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
        "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])), "r"(__float_as_uint(v[8])),
        "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
        "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
        "r"(__float_as_uint(v[15]))
        : "memory");
}

__device__ __forceinline__ void tmem_wait_ld() {
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_wait_st() {
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// Shared-memory matrix descriptor (tcgen05 format): start address, leading and
// stride byte offsets (all >> 4), descriptor version 1 at bits 46-47, swizzle
// mode at bits 61-63 (2 = 128-byte swizzle).
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lbo_bytes, uint32_t sbo_bytes,
                                              uint32_t swizzle_mode) {
    uint64_t d = 0;
    d |= uint64_t((saddr >> 4) & 0x3FFF);
    d |= uint64_t((lbo_bytes >> 4) & 0x3FFF) << 16;
    d |= uint64_t((sbo_bytes >> 4) & 0x3FFF) << 32;
    d |= uint64_t(1) << 46;
    d |= uint64_t(swizzle_mode & 7) << 61;
    return d;
}

// Instruction descriptor for kind::f16: fp32 accumulator, bf16 A and B,
// a_mn / b_mn select MN-major (transposed) operands, M = 128 or 64, N % 16 == 0.
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int M, int N, bool a_mn, bool b_mn) {
    return (1u << 4)                       // D format: f32
           | (1u << 7)                     // A format: bf16
           | (1u << 10)                    // B format: bf16
           | (uint32_t(a_mn) << 15)        // A major: 0 K-major, 1 MN-major
           | (uint32_t(b_mn) << 16)        // B major
           | (uint32_t(N >> 3) << 17)      // N / 8
           | (uint32_t(M >> 4) << 24);     // M / 16
}

// Programmatic dependent launch.  A kernel launched with programmatic stream
// serialization may start while its predecessor on the stream is still running;
// pdl_wait() blocks until the predecessor grid has completed and its memory is
// visible (a no-op for an ordinary launch), so every kernel calls it before its
// first global-memory access.  pdl_trigger() lets the successor start launching.
// A successor that launches early holds SM slots while it waits, which a kernel on
// another stream may need: so the decode triggers only when its work is done, and the
// short kernels (combine, merge, migration) never trigger (their successors launch as
// they exit).
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// Named barrier over `count` threads with OR-reduction of a predicate.
__device__ __forceinline__ bool named_barrier_or(int id, int count, bool pred) {
    uint32_t out;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.or.pred q, %2, %3, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(out)
        : "r"(uint32_t(pred)), "r"(id), "r"(count)
        : "memory");
    return out != 0;
}

__device__ __forceinline__ void named_barrier_sync(int id, int count) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

}  // namespace splash
