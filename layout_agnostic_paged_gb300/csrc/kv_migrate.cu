// kv_migrate.cu -- bit-exact KV-page migration between block pools (K5).
//
// "SPLASH: Switching Parallel Layouts of Attention with Seamless Handoff for LLM
// Serving", Abstract: a layout switch reuses the state already in place and
// moves the rest in the background; for the paged cache that is whole pages
// copied from one pool to another at new ids, after which the owner's block
// table is rewritten.  HBM-bound: every page is read once and written once, in
// 16-byte vectors with several loads in flight per thread; loads and stores use
// the streaming cache hints so a background copy does not evict decode data.
#include "common.cuh"
#include "kernels.h"

namespace splash {
namespace {

constexpr int kMigThreads = 256;
constexpr int kMigUnroll = 6;

__global__ void __launch_bounds__(kMigThreads) kv_migrate_kernel(
    const uint4* __restrict__ src, uint4* __restrict__ dst, int64_t vec_per_page,
    const int32_t* __restrict__ src_ids, const int32_t* __restrict__ dst_ids, int n, int src_np,
    int dst_np) {
    pdl_wait();
    pdl_trigger();
    for (int i = blockIdx.x; i < n; i += gridDim.x) {
        const int s = src_ids[i];
        const int d = dst_ids[i];
        if (s < 0 || s >= src_np || d < 0 || d >= dst_np) continue;
        const uint4* sp = src + int64_t(s) * vec_per_page;
        uint4* dp = dst + int64_t(d) * vec_per_page;
        int64_t v = threadIdx.x;
        for (; v + (kMigUnroll - 1) * kMigThreads < vec_per_page; v += kMigUnroll * kMigThreads) {
            uint4 buf[kMigUnroll];
#pragma unroll
            for (int u = 0; u < kMigUnroll; ++u) buf[u] = __ldcs(sp + v + u * kMigThreads);
#pragma unroll
            for (int u = 0; u < kMigUnroll; ++u) __stcs(dp + v + u * kMigThreads, buf[u]);
        }
        for (; v < vec_per_page; v += kMigThreads) __stcs(dp + v, __ldcs(sp + v));
    }
}

}  // namespace

cudaError_t launch_kv_migrate(const void* src, void* dst, size_t page_bytes, const int32_t* src_ids,
                              const int32_t* dst_ids, int n, int src_np, int dst_np, int sm_count,
                              cudaStream_t stream) {
    if (n == 0) return cudaSuccess;
    const int blocks = n < sm_count * 8 ? n : sm_count * 8;
    return launch_pdl(kv_migrate_kernel, dim3(blocks), dim3(kMigThreads), 0, stream,
                      static_cast<const uint4*>(src), static_cast<uint4*>(dst),
                      int64_t(page_bytes / 16), src_ids, dst_ids, n, src_np, dst_np);
}

}  // namespace splash
