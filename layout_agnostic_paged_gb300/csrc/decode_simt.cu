// decode_simt.cu -- CUDA-core paged MLA decode kernel (fp32 FMA, exact softmax).
//
// A plain kernel over the same split plan as the tensor-core kernel: one CTA per
// (CTA group, group of 16 heads); each piece of a request is scanned in 32-token
// chunks gathered through the block table into shared memory, with an fp32
// online softmax.  It is the correctness baseline the tensor-core kernel is
// checked against on the GPU, and handles shapes the tensor-core kernel does
// not take.
//
// Method: "SPLASH: Switching Parallel Layouts of Attention with Seamless Handoff
// for LLM Serving", Abstract (all query heads read one shared latent KV stream)
// and Appendix, Table 2 (a call covers a head share, a token share or whole
// requests).
#include <math.h>

#include "common.cuh"
#include "kernels.h"

namespace splash {
namespace {

constexpr int kThreads = 256;
constexpr int kChunk = 32;
constexpr int kHG = kSimtHeads;

struct SimtSmem {
    float q[kHG][kDqk];
    __nv_bfloat16 k[kChunk][kDqk];
    float p[kHG][kChunk];
    float m[kHG], l[kHG], alpha[kHG];
};

__global__ void __launch_bounds__(kThreads) decode_simt_kernel(DecodeArgs a) {
    extern __shared__ __align__(16) uint8_t smem_raw[];
    SimtSmem& sm = *reinterpret_cast<SimtSmem*>(smem_raw);
    pdl_wait();
    const int NG = (a.Hs + kHG - 1) / kHG;
    const int j = blockIdx.x / NG, g = blockIdx.x % NG;
    uint8_t* ws = static_cast<uint8_t*>(a.ws);
    PlanHeader* hdr = reinterpret_cast<PlanHeader*>(ws);
    const WorkspaceLayout lay(a.B, a.Hs, a.num_groups);
    const ReqPlan* req = reinterpret_cast<const ReqPlan*>(ws + lay.req_off);
    float* pout = reinterpret_cast<float*>(ws + lay.pout_off);
    float* plse = reinterpret_cast<float*>(ws + lay.plse_off);

    const int64_t T = hdr->total_tiles;
    const int G = hdr->num_groups;  // groups in use (<= a.num_groups, <= T)
    if (T == 0 || j >= G) return;
    const int64_t aj = group_start(j, T, G), bj = group_start(j + 1, T, G);
    if (aj >= bj) return;
    const int hbase = g * kHG;                       // first head of the group within the slice
    const int nh = min(kHG, a.Hs - hbase);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const __nv_bfloat16* qg = static_cast<const __nv_bfloat16*>(a.q);
    const uint4* pool = static_cast<const uint4*>(a.kv_pool);
    constexpr int kVecPerRow = kDqk * 2 / 16;         // 72 x 16 B per token row

    const int32_t* first_req = reinterpret_cast<const int32_t*>(ws + lay.grp_off);
    for (int r = first_req[j]; r < a.B && req[r].tile_begin < bj; ++r) {
        const ReqPlan p = req[r];
        if (p.ntiles == 0) continue;
        const int row = p.row;  // storage row of q / block_table / out / lse
        const int64_t t_lo = max(aj, p.tile_begin) - p.tile_begin;
        const int64_t t_hi = min(bj, p.tile_begin + p.ntiles) - p.tile_begin;
        const int split = j - p.first_grp;
        const int tok_begin = int(max(int64_t(p.lo), (p.tile0 + t_lo) * kTileTokens));
        const int tok_end = int(min(int64_t(p.hi), (p.tile0 + t_hi) * kTileTokens));

        __syncthreads();
        for (int i = tid; i < kHG * kDqk; i += kThreads) {
            const int h = i / kDqk, d = i % kDqk;
            sm.q[h][d] = h < nh ? __bfloat162float(
                                      qg[(int64_t(row) * a.H + a.head_lo + hbase + h) * kDqk + d])
                                : 0.f;
        }
        if (tid < kHG) {
            sm.m[tid] = -INFINITY;
            sm.l[tid] = 0.f;
        }
        float acc[kHG][2];
#pragma unroll
        for (int h = 0; h < kHG; ++h) acc[h][0] = acc[h][1] = 0.f;

        for (int c0 = tok_begin; c0 < tok_end; c0 += kChunk) {
            __syncthreads();
            // Gather 32 token rows through the block table; rows past the range are zero.
            for (int i = tid; i < kChunk * kVecPerRow; i += kThreads) {
                const int t = i / kVecPerRow, v = i % kVecPerRow;
                const int tok = c0 + t;
                uint4 val = make_uint4(0u, 0u, 0u, 0u);
                if (tok < tok_end) {
                    const int pid = a.block_table[int64_t(row) * a.max_pages + tok / a.P];
                    if (pid >= 0 && pid < a.num_pages)
                        val = pool[(int64_t(pid) * a.P + tok % a.P) * kVecPerRow + v];
                    else if (v == 0)
                        atomicOr(&hdr->status, uint32_t(SPLASH_DEVICE_BAD_INPUT));
                }
                reinterpret_cast<uint4*>(&sm.k[t][0])[v] = val;
            }
            __syncthreads();
            // Scores: one warp per (head, token) pair, lanes over the 576 dims.
            for (int pair = warp; pair < kHG * kChunk; pair += kThreads / 32) {
                const int h = pair / kChunk, t = pair % kChunk;
                float s = 0.f;
                for (int d = lane; d < kDqk; d += 32) s += sm.q[h][d] * __bfloat162float(sm.k[t][d]);
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
                if (lane == 0) sm.p[h][t] = (c0 + t < tok_end) ? s * a.scale : -INFINITY;
            }
            __syncthreads();
            // Online softmax, one thread per head.
            if (tid < kHG) {
                const int h = tid;
                float cmax = -INFINITY;
                for (int t = 0; t < kChunk; ++t) cmax = fmaxf(cmax, sm.p[h][t]);
                const float m_new = fmaxf(sm.m[h], cmax);
                const float alpha = (sm.m[h] == -INFINITY) ? 0.f : expf(sm.m[h] - m_new);
                float lsum = 0.f;
                for (int t = 0; t < kChunk; ++t) {
                    const float s = sm.p[h][t];
                    const float e = (s == -INFINITY) ? 0.f : expf(s - m_new);
                    sm.p[h][t] = e;
                    lsum += e;
                }
                sm.l[h] = sm.l[h] * alpha + lsum;
                sm.m[h] = m_new;
                sm.alpha[h] = alpha;
            }
            __syncthreads();
            // O = alpha O + P V over the latent prefix; thread owns dv = tid, tid + 256.
#pragma unroll
            for (int h = 0; h < kHG; ++h) {
                acc[h][0] *= sm.alpha[h];
                acc[h][1] *= sm.alpha[h];
            }
            for (int t = 0; t < kChunk; ++t) {
                const float v0 = __bfloat162float(sm.k[t][tid]);
                const float v1 = __bfloat162float(sm.k[t][tid + 256]);
#pragma unroll
                for (int h = 0; h < kHG; ++h) {
                    const float w = sm.p[h][t];
                    acc[h][0] = fmaf(w, v0, acc[h][0]);
                    acc[h][1] = fmaf(w, v1, acc[h][1]);
                }
            }
        }
        __syncthreads();
        // Epilogue: final rows go to out / lse, split pieces to their partial slot.
        for (int h = 0; h < nh; ++h) {
            const float L = sm.l[h];
            const float inv = 1.0f / L;
            const int hh = hbase + h;
            float* dst;
            float* dlse;
            if (p.nsplit == 1) {
                dst = a.out + (int64_t(row) * a.H + a.head_lo + hh) * kDv;
                dlse = a.lse + int64_t(row) * a.H + a.head_lo + hh;
            } else {
                const int64_t slot = p.slot_base + split;
                dst = pout + (slot * a.Hs + hh) * kDv;
                dlse = plse + slot * a.Hs + hh;
            }
            dst[tid] = acc[h][0] * inv;
            dst[tid + 256] = acc[h][1] * inv;
            if (tid == 0) *dlse = sm.m[h] + logf(L);
        }
    }
}

}  // namespace

cudaError_t launch_decode_simt(const DecodeArgs& a, cudaStream_t stream) {
    const int NG = (a.Hs + kHG - 1) / kHG;
    const int smem = int(sizeof(SimtSmem));
    cudaError_t e = ensure_smem_optin(reinterpret_cast<const void*>(decode_simt_kernel), smem);
    if (e != cudaSuccess) return e;
    return launch_pdl(decode_simt_kernel, dim3(a.num_groups * NG), dim3(kThreads), smem, stream, a);
}

}  // namespace splash
