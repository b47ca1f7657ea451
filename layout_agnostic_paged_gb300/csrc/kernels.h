// kernels.h -- internal launchers shared by the C-ABI translation unit.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace splash {

// Launches `kernel` on `stream` with programmatic stream serialization (the kernel
// must call pdl_wait() before touching global memory).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t stream, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// Arguments of one decode-kernel launch (device pointers, already validated).
struct DecodeArgs {
    const void* q;              // bf16 [num_rows][H][576]
    const void* kv_pool;        // bf16 [num_pages][kv_heads][P][576]
    const int32_t* block_table; // [num_rows][max_pages]
    const int32_t* ctx_lens;    // [num_rows]
    const int32_t* lo_arr;      // [B] per-request token range starts, or null (tok_lo)
    const int32_t* hi_arr;      // [B] per-request token range ends, or null (tok_hi)
    const int32_t* rows;        // [B] storage row of request r, or null (row r)
    float* out;                 // [num_rows][H][512]
    float* lse;                 // [num_rows][H]
    void* ws;                   // workspace (plan + per-CTA status + partials)
    int64_t tok_lo, tok_hi;     // the call's scalar token range (tok_hi < 0: to the end)
    int B, H, P, num_pages, max_pages;
    int num_rows;               // rows of q / block_table / ctx_lens / out / lse
    int max_ctx;                // max_pages * P: longest valid context
    int head_lo, Hs;            // head slice
    int num_groups;             // CTA groups G'
    int ctas;                   // CTAs of the decode grid (num_groups x head groups)
    int sts_cap;                // capacity of the workspace's per-CTA status array
    int kv_heads;               // KV heads per token (1: the shared latent head)
    int q_per_kv;               // query heads per KV head (H / kv_heads)
    float scale;
};

// Raises a kernel's dynamic shared-memory limit once per (kernel, device).
cudaError_t ensure_smem_optin(const void* kernel, int bytes);

// K3: merges the partials of requests cut across CTA groups, writes the empty-set
// result of empty requests and ORs the decode CTAs' status words into the header.
cudaError_t launch_combine(const void* ws, int B, int H, int head_lo, int Hs, int num_groups,
                           int ctas, int sts_cap, float* out, float* lse, cudaStream_t stream);
cudaError_t launch_lse_merge(const float* part_out, const float* part_lse, int S, int64_t rows,
                             int d_v, float* out, float* lse, cudaStream_t stream);
cudaError_t launch_kv_migrate(const void* src, void* dst, size_t page_bytes, const int32_t* src_ids,
                              const int32_t* dst_ids, int n, int src_np, int dst_np, int sm_count,
                              cudaStream_t stream);

// Tensor-core decode kernel: head groups of at most 64 heads, one CTA per (CTA group,
// head group), persistent over the plan.  map_q covers q as [B*H rows][576] bf16 with
// a {64, pad(group_heads)} box; map_kv covers the pool as [num_pages*P rows][576] with
// a {64, P} box; both use the 128-byte swizzle.
constexpr int kTcMaxGroupHeads = 64;
int tc_pad_heads(int group_heads);
cudaError_t launch_decode_tc(const DecodeArgs& a, const CUtensorMap& map_q,
                             const CUtensorMap& map_kv, int head_groups, int group_heads,
                             cudaStream_t stream);

}  // namespace splash
