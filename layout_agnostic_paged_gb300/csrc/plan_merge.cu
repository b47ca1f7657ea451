// plan_merge.cu -- intra-call combine of split partials (K3) and the public
// log-sum-exp merge (K4).  The split plan (K1) that decides which requests are cut
// across CTA groups is computed by the decode kernel itself (plan.cuh).
//
// Method context: "SPLASH: Switching Parallel Layouts of Attention with Seamless
// Handoff for LLM Serving", Appendix, Table 2 (CP reads an equal token share under
// ideal token partitioning; its partials merge by their log-sum-exp weights).
#include <math.h>

#include "common.cuh"
#include "kernels.h"

namespace splash {

namespace {

// Optional kernel-boundary trace (compiled in only with -DSPLASH_TRACE): globaltimer
// stamps of the combine kernel, read back with splash_ktrace_read().
#ifdef SPLASH_TRACE
__device__ unsigned long long g_ktrace[8];
#define KTRACE_MIN(slot) atomicMin(&g_ktrace[slot], globaltimer_ns())
#define KTRACE_MAX(slot) atomicMax(&g_ktrace[slot], globaltimer_ns())
#else
#define KTRACE_MIN(slot) ((void)0)
#define KTRACE_MAX(slot) ((void)0)
#endif

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
// empty-set result; single-piece requests were written by the decode kernel.  The
// first warp also ORs the decode CTAs' status words into the header.
__global__ void __launch_bounds__(256) combine_kernel(uint8_t* __restrict__ ws, int B, int H,
                                                      int head_lo, int Hs, int num_groups, int ctas,
                                                      int sts_cap, float* __restrict__ out,
                                                      float* __restrict__ lse) {
    if (threadIdx.x == 0) KTRACE_MIN(3);
    pdl_wait();
    if (threadIdx.x == 0) KTRACE_MIN(4);
    if (threadIdx.x == 0) KTRACE_MAX(5);
    const WorkspaceLayout lay(B, Hs, num_groups, sts_cap);
    if (blockIdx.x == 0 && threadIdx.x < 32) {
        const uint32_t* sts = reinterpret_cast<const uint32_t*>(ws + lay.sts_off);
        uint32_t bits = 0;
        for (int i = threadIdx.x; i < ctas; i += 32) bits |= sts[i];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) bits |= __shfl_xor_sync(0xffffffffu, bits, o);
        if (threadIdx.x == 0) reinterpret_cast<PlanHeader*>(ws)->status = bits;
    }
    const int64_t row = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    if (row >= int64_t(B) * Hs) return;
    const int r = int(row / Hs), hh = int(row % Hs);
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

cudaError_t launch_combine(const void* ws, int B, int H, int head_lo, int Hs, int num_groups,
                           int ctas, int sts_cap, float* out, float* lse, cudaStream_t stream) {
    const int64_t threads = int64_t(B) * Hs * 32;
    const int blocks = int((threads + 255) / 256);
    if (blocks == 0) return cudaSuccess;
    return launch_pdl(combine_kernel, dim3(blocks), dim3(256), 0, stream,
                      static_cast<uint8_t*>(const_cast<void*>(ws)), B, H, head_lo, Hs, num_groups,
                      ctas, sts_cap, out, lse);
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
