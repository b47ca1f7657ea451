// splash_api.cu -- the C ABI (include/splash.h): host-side validation, workspace
// sizing, per-device state and kernel launches.  No allocation, no stream
// synchronisation (except splash_workspace_status, which is documented to sync).
#include <stdlib.h>
#include <string.h>

#include <mutex>
#include <unordered_map>

#include "common.cuh"
#include "kernels.h"

namespace splash {
namespace {

std::mutex g_mu;
int g_sm_count[128];
std::unordered_map<uint64_t, int> g_smem_optin;  // (kernel ptr ^ device) -> bytes set

int current_device(int* dev) {
    return cudaGetDevice(dev) == cudaSuccess ? 0 : -1;
}

int sm_count(int dev) {
    if (dev < 0 || dev >= 128) return 0;
    std::lock_guard<std::mutex> lk(g_mu);
    if (g_sm_count[dev] == 0) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
        g_sm_count[dev] = n;
    }
    return g_sm_count[dev];
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

int validate_desc(const splash_attn_desc* d) {
    if (!d) return SPLASH_ERR_INVALID_ARG;
    if (d->num_reqs < 0 || d->num_heads <= 0 || d->num_pages < 0 || d->max_pages_per_req < 0)
        return SPLASH_ERR_INVALID_ARG;
    if (!(d->scale == d->scale)) return SPLASH_ERR_INVALID_ARG;  // NaN scale
    if (d->d_qk != kDqk || d->d_v != kDv) return SPLASH_ERR_UNSUPPORTED;
    const int P = d->page_size;
    if (P != 16 && P != 32 && P != 64 && P != 128) return SPLASH_ERR_UNSUPPORTED;
    if (int64_t(d->num_pages) * P >= (int64_t(1) << 31)) return SPLASH_ERR_UNSUPPORTED;
    if (int64_t(d->max_pages_per_req) * P >= (int64_t(1) << 31)) return SPLASH_ERR_UNSUPPORTED;
    if (int64_t(d->num_reqs) * d->num_heads >= (int64_t(1) << 31)) return SPLASH_ERR_UNSUPPORTED;
    return SPLASH_OK;
}

// Launch geometry of the decode kernel for a head slice of Hs heads.
struct Geometry {
    int head_groups;  // CTAs per CTA group (one per head group)
    int group_heads;  // heads per head group (the last group may have fewer)
    int num_groups;   // CTA groups G' (the tile sequence is cut into G' ranges)
};

// kv_group_heads > 0 forces head groups of that size (several KV heads: a group must
// stay within one KV head's query heads).
Geometry decode_geometry(int Hs, int sms, int kv_group_heads = 0) {
    Geometry g;
    if (kv_group_heads > 0) {
        g.group_heads = kv_group_heads;
        g.head_groups = (Hs + kv_group_heads - 1) / kv_group_heads;
        g.num_groups = sms / g.head_groups;
    } else {
        g.head_groups = (Hs + kTcMaxGroupHeads - 1) / kTcMaxGroupHeads;
        g.group_heads = (Hs + g.head_groups - 1) / g.head_groups;
        g.num_groups = sms / g.head_groups;  // one persistent CTA per SM
    }
    if (g.num_groups < 1) g.num_groups = 1;
    return g;
}

// cuTensorMapEncodeTiled through the runtime's driver entry point (no libcuda link).
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

// 2D bf16 map over [rows][576] with a {64, box_rows} box and the 128-byte swizzle.
bool encode_rows_576(CUtensorMap* m, const void* base, uint64_t rows, uint32_t box_rows) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {uint64_t(kDqk), rows};
    cuuint64_t strides[1] = {uint64_t(kDqk) * 2};
    cuuint32_t box[2] = {64u, box_rows};
    cuuint32_t es[2] = {1u, 1u};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
              es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

cudaError_t ensure_smem_optin(const void* kernel, int bytes) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const uint64_t key = reinterpret_cast<uint64_t>(kernel) * 131u + uint64_t(dev);
    std::lock_guard<std::mutex> lk(g_mu);
    auto it = g_smem_optin.find(key);
    if (it != g_smem_optin.end() && it->second >= bytes) return cudaSuccess;
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess) g_smem_optin[key] = bytes;
    return e;
}

}  // namespace splash

using namespace splash;

extern "C" {

const char* splash_status_string(int status) {
    switch (status) {
        case SPLASH_OK: return "SPLASH_OK";
        case SPLASH_ERR_INVALID_ARG: return "SPLASH_ERR_INVALID_ARG: invalid argument";
        case SPLASH_ERR_UNSUPPORTED: return "SPLASH_ERR_UNSUPPORTED: shape not supported";
        case SPLASH_ERR_WORKSPACE: return "SPLASH_ERR_WORKSPACE: workspace too small";
        case SPLASH_ERR_CUDA: return "SPLASH_ERR_CUDA: CUDA call failed";
        default: return "unknown splash status";
    }
}

size_t splash_decode_workspace_size(const splash_attn_desc* desc, int head_lo, int head_hi) {
    if (validate_desc(desc) != SPLASH_OK) return 0;
    if (head_lo < 0 || head_hi > desc->num_heads || head_lo >= head_hi) return 0;
    int dev = 0;
    if (current_device(&dev) != 0) return 0;
    const int sms = sm_count(dev);
    if (sms <= 0) return 0;
    const int Hs = head_hi - head_lo;
    const Geometry g = decode_geometry(Hs, sms);
    return WorkspaceLayout(desc->num_reqs, Hs, g.num_groups,
                           status_capacity(sms, g.num_groups * g.head_groups)).total;
}

int splash_decode_attn(const splash_attn_desc* desc, const void* q, const void* kv_pool,
                       const int32_t* block_table, const int32_t* ctx_lens, int head_lo,
                       int head_hi, int64_t tok_lo, int64_t tok_hi, float* out, float* lse,
                       void* workspace, size_t ws_bytes, splash_stream_t stream_) {
    return splash_decode_attn_ex(desc, nullptr, q, kv_pool, block_table, ctx_lens, head_lo, head_hi,
                                 tok_lo, tok_hi, out, lse, workspace, ws_bytes, stream_);
}

int splash_decode_attn_ex(const splash_attn_desc* desc, const splash_decode_ext* ext,
                          const void* q, const void* kv_pool, const int32_t* block_table,
                          const int32_t* ctx_lens, int head_lo, int head_hi, int64_t tok_lo,
                          int64_t tok_hi, float* out, float* lse, void* workspace,
                          size_t ws_bytes, splash_stream_t stream_) {
    int st = validate_desc(desc);
    if (st != SPLASH_OK) return st;
    if (head_lo < 0 || head_hi > desc->num_heads || head_lo >= head_hi) return SPLASH_ERR_INVALID_ARG;
    if (tok_lo < 0 || (tok_hi >= 0 && tok_hi < tok_lo)) return SPLASH_ERR_INVALID_ARG;
    if (tok_lo >= (int64_t(1) << 31)) tok_lo = (int64_t(1) << 31) - 1;   // beyond any context
    if (tok_hi >= (int64_t(1) << 31)) tok_hi = (int64_t(1) << 31) - 1;
    if (!workspace || !aligned(workspace, 256)) return SPLASH_ERR_INVALID_ARG;
    const int B = desc->num_reqs;
    const int32_t* lo_arr = ext ? ext->tok_lo : nullptr;
    const int32_t* hi_arr = ext ? ext->tok_hi : nullptr;
    const int32_t* rows = ext ? ext->rows : nullptr;
    const int num_rows = rows ? ext->num_rows : B;   // rows of q / block_table / ... / lse
    if (rows && num_rows < 1) return SPLASH_ERR_INVALID_ARG;
    const int max_sms = ext ? ext->max_sms : 0;
    if (max_sms < 0) return SPLASH_ERR_INVALID_ARG;
    const int kv_heads = ext && ext->num_kv_heads > 1 ? ext->num_kv_heads : 1;
    if (ext && ext->num_kv_heads < 0) return SPLASH_ERR_INVALID_ARG;
    int kv_group_heads = 0;   // head-group size forced by several KV heads
    if (kv_heads > 1) {
        if (desc->num_heads % kv_heads != 0) return SPLASH_ERR_INVALID_ARG;
        const int per_kv = desc->num_heads / kv_heads;
        if (per_kv > kTcMaxGroupHeads && per_kv % kTcMaxGroupHeads != 0) return SPLASH_ERR_UNSUPPORTED;
        kv_group_heads = per_kv < kTcMaxGroupHeads ? per_kv : kTcMaxGroupHeads;
        if (head_lo % kv_group_heads != 0) return SPLASH_ERR_UNSUPPORTED;
        if (int64_t(desc->num_pages) * kv_heads * desc->page_size >= (int64_t(1) << 31))
            return SPLASH_ERR_UNSUPPORTED;
    }
    if (!aligned(lo_arr, 4) || !aligned(hi_arr, 4) || !aligned(rows, 4)) return SPLASH_ERR_INVALID_ARG;
    if (B > 0) {
        if (!q || !block_table || !ctx_lens || !out || !lse) return SPLASH_ERR_INVALID_ARG;
        if (!aligned(q, 16) || !aligned(out, 16) || !aligned(lse, 4) || !aligned(block_table, 4) ||
            !aligned(ctx_lens, 4))
            return SPLASH_ERR_INVALID_ARG;
        if (desc->num_pages > 0 && (!kv_pool || !aligned(kv_pool, 16))) return SPLASH_ERR_INVALID_ARG;
    }
    int dev = 0;
    if (current_device(&dev) != 0) return SPLASH_ERR_CUDA;
    const int sms = sm_count(dev);
    if (sms <= 0) return SPLASH_ERR_CUDA;
    const int Hs = head_hi - head_lo;
    const Geometry g = decode_geometry(Hs, max_sms > 0 && max_sms < sms ? max_sms : sms,
                                       kv_group_heads);
    const int ctas = g.num_groups * g.head_groups;
    const int sts_cap = status_capacity(sms, ctas);
    const WorkspaceLayout lay(B, Hs, g.num_groups, sts_cap);
    if (ws_bytes < lay.total) return SPLASH_ERR_WORKSPACE;
    if (B == 0) return SPLASH_OK;

    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
    DecodeArgs a;
    a.q = q;
    a.kv_pool = kv_pool;
    a.block_table = block_table;
    a.ctx_lens = ctx_lens;
    a.lo_arr = lo_arr;
    a.hi_arr = hi_arr;
    a.rows = rows;
    a.out = out;
    a.lse = lse;
    a.ws = workspace;
    a.tok_lo = tok_lo;
    a.tok_hi = tok_hi;
    a.B = B;
    a.H = desc->num_heads;
    a.P = desc->page_size;
    a.num_pages = desc->num_pages;
    a.max_pages = desc->max_pages_per_req;
    a.num_rows = num_rows;
    a.max_ctx = desc->max_pages_per_req * desc->page_size;
    a.head_lo = head_lo;
    a.Hs = Hs;
    a.num_groups = g.num_groups;
    a.ctas = ctas;
    a.sts_cap = sts_cap;
    a.kv_heads = kv_heads;
    a.q_per_kv = desc->num_heads / kv_heads;
    a.scale = desc->scale;
    {
        CUtensorMap mq, mkv;
        const uint32_t qbox = uint32_t(tc_pad_heads(g.group_heads));
        if (!encode_rows_576(&mq, q, uint64_t(num_rows) * desc->num_heads, qbox)) return SPLASH_ERR_CUDA;
        // an empty pool still needs a valid map: point it at the workspace (never read,
        // every page id is then out of range)
        const void* kv = desc->num_pages > 0 ? kv_pool : workspace;
        const uint64_t kv_rows = desc->num_pages > 0
                                     ? uint64_t(desc->num_pages) * kv_heads * desc->page_size
                                     : uint64_t(1);
        if (!encode_rows_576(&mkv, kv, kv_rows, uint32_t(desc->page_size))) return SPLASH_ERR_CUDA;
        if (launch_decode_tc(a, mq, mkv, g.head_groups, g.group_heads, stream) != cudaSuccess)
            return SPLASH_ERR_CUDA;
    }
    if (launch_combine(workspace, B, desc->num_heads, head_lo, Hs, g.num_groups, ctas, sts_cap, out,
                       lse, stream) != cudaSuccess)
        return SPLASH_ERR_CUDA;
    return SPLASH_OK;
}

int splash_lse_merge(const float* part_out, const float* part_lse, int S, int B, int H, int d_v,
                     float* out, float* lse, splash_stream_t stream) {
    if (S < 1 || B < 0 || H < 0 || d_v <= 0 || (d_v % 4) != 0) return SPLASH_ERR_INVALID_ARG;
    const int64_t rows = int64_t(B) * H;
    if (rows == 0) return SPLASH_OK;
    if (!part_out || !part_lse || !out || !lse) return SPLASH_ERR_INVALID_ARG;
    if (!aligned(part_out, 16) || !aligned(out, 16) || !aligned(part_lse, 4) || !aligned(lse, 4))
        return SPLASH_ERR_INVALID_ARG;
    // out must not overlap part_out
    const uintptr_t po0 = reinterpret_cast<uintptr_t>(part_out);
    const uintptr_t po1 = po0 + uintptr_t(S) * rows * d_v * sizeof(float);
    const uintptr_t o0 = reinterpret_cast<uintptr_t>(out);
    const uintptr_t o1 = o0 + uintptr_t(rows) * d_v * sizeof(float);
    if (o0 < po1 && po0 < o1) return SPLASH_ERR_INVALID_ARG;
    if (launch_lse_merge(part_out, part_lse, S, rows, d_v, out, lse,
                         reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
        return SPLASH_ERR_CUDA;
    return SPLASH_OK;
}

int splash_kv_migrate(const void* src_pool, void* dst_pool, size_t page_bytes,
                      const int32_t* src_ids, const int32_t* dst_ids, int n_pages,
                      int32_t src_num_pages, int32_t dst_num_pages, splash_stream_t stream) {
    if (n_pages < 0 || page_bytes == 0 || (page_bytes % 16) != 0 || src_num_pages < 0 ||
        dst_num_pages < 0)
        return SPLASH_ERR_INVALID_ARG;
    if (n_pages == 0) return SPLASH_OK;
    if (!src_pool || !dst_pool || !src_ids || !dst_ids) return SPLASH_ERR_INVALID_ARG;
    if (!aligned(src_pool, 16) || !aligned(dst_pool, 16) || !aligned(src_ids, 4) ||
        !aligned(dst_ids, 4))
        return SPLASH_ERR_INVALID_ARG;
    int dev = 0;
    if (current_device(&dev) != 0) return SPLASH_ERR_CUDA;
    const int sms = sm_count(dev);
    if (sms <= 0) return SPLASH_ERR_CUDA;
    if (launch_kv_migrate(src_pool, dst_pool, page_bytes, src_ids, dst_ids, n_pages, src_num_pages,
                          dst_num_pages, sms, reinterpret_cast<cudaStream_t>(stream)) !=
        cudaSuccess)
        return SPLASH_ERR_CUDA;
    return SPLASH_OK;
}

int splash_workspace_status(const void* workspace, uint32_t* flags, splash_stream_t stream) {
    if (!workspace || !flags) return SPLASH_ERR_INVALID_ARG;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (cudaStreamSynchronize(s) != cudaSuccess) return SPLASH_ERR_CUDA;
    if (cudaMemcpy(flags, workspace, sizeof(uint32_t), cudaMemcpyDeviceToHost) != cudaSuccess)
        return SPLASH_ERR_CUDA;
    return SPLASH_OK;
}

}  // extern "C"
