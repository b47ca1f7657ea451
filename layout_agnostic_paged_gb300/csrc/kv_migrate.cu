// kv_migrate.cu -- bit-exact KV-page migration between block pools (K5).
//
// "SPLASH: Switching Parallel Layouts of Attention with Seamless Handoff for LLM
// Serving", Abstract: a layout switch reuses the state already in place and
// moves the rest in the background; for the paged cache that is whole pages
// copied from one pool to another at new ids, after which the owner's block
// table is rewritten.  HBM-bound: every page is read once and written once, in
// 16-byte vectors with several loads in flight per thread, pages cut into 24 KB
// chunks so that small handoffs still use every SM; loads and stores use
// the streaming cache hints so a background copy does not evict decode data.
#include "common.cuh"
#include "kernels.h"

namespace splash {
namespace {

constexpr int kMigThreads = 256;
constexpr int kMigUnroll = 6;
constexpr int kMigChunkVec = kMigThreads * kMigUnroll;  // 16-byte vectors per work item (24 KB)

// Work item i copies chunk i % chunks_per_page of page i / chunks_per_page, so a
// handoff of a few pages still spreads over many CTAs; one pass of kMigUnroll
// loads in flight per thread covers a chunk.
__global__ void __launch_bounds__(kMigThreads) kv_migrate_kernel(
    const uint4* __restrict__ src, uint4* __restrict__ dst, int64_t vec_per_page,
    int chunks_per_page, const int32_t* __restrict__ src_ids,
    const int32_t* __restrict__ dst_ids, int n, int src_np, int dst_np) {
    pdl_wait();
    const int64_t items = int64_t(n) * chunks_per_page;
    for (int64_t i = blockIdx.x; i < items; i += gridDim.x) {
        const int pg = int(i / chunks_per_page);
        const int64_t v0 = (i % chunks_per_page) * int64_t(kMigChunkVec);
        const int s = src_ids[pg];
        const int d = dst_ids[pg];
        if (s < 0 || s >= src_np || d < 0 || d >= dst_np) continue;
        const uint4* sp = src + int64_t(s) * vec_per_page;
        uint4* dp = dst + int64_t(d) * vec_per_page;
        const int64_t v = v0 + threadIdx.x;
        if (v0 + kMigChunkVec <= vec_per_page) {
            uint4 buf[kMigUnroll];
#pragma unroll
            for (int u = 0; u < kMigUnroll; ++u) buf[u] = __ldcs(sp + v + u * kMigThreads);
#pragma unroll
            for (int u = 0; u < kMigUnroll; ++u) __stcs(dp + v + u * kMigThreads, buf[u]);
        } else {
            for (int64_t w = v; w < vec_per_page; w += kMigThreads) __stcs(dp + w, __ldcs(sp + w));
        }
    }
}

}  // namespace

cudaError_t launch_kv_migrate(const void* src, void* dst, size_t page_bytes, const int32_t* src_ids,
                              const int32_t* dst_ids, int n, int src_np, int dst_np, int sm_count,
                              cudaStream_t stream) {
    if (n == 0) return cudaSuccess;
    const int64_t vec_per_page = int64_t(page_bytes / 16);
    const int cpp = int((vec_per_page + kMigChunkVec - 1) / kMigChunkVec);
    const int64_t items = int64_t(n) * cpp;
    const int blocks = int(items < int64_t(sm_count) * 8 ? items : int64_t(sm_count) * 8);
    return launch_pdl(kv_migrate_kernel, dim3(blocks), dim3(kMigThreads), 0, stream,
                      static_cast<const uint4*>(src), static_cast<uint4*>(dst), vec_per_page, cpp,
                      src_ids, dst_ids, n, src_np, dst_np);
}

}  // namespace splash
