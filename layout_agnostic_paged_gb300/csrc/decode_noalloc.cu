// decode_noalloc.cu -- splash_decode_attn_noalloc: paged decode attention whose
// scratch memory is a fixed array inside the library, so the caller passes only
// inputs and outputs and nothing is allocated at call time.
//
// The attention itself is splash_decode_attn's: this entry point forwards to it
// with the library-owned scratch in place of a caller workspace.
#include <mutex>

#include "common.cuh"

namespace splash {
namespace {

// Library-owned scratch of the no-allocation entry point.  Every GPU that loads
// the library holds these bytes until the process exits.
constexpr size_t kNoAllocScratchBytes = size_t(32) << 20;  // 32 MiB
static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 128;
std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices];  // device address of g_noalloc_scratch, per device

// Resolves the device address of the scratch array on the current device (once per
// device).  In host code `g_noalloc_scratch` names only a host-side stand-in, so
// the address must come from cudaGetSymbolAddress with that device current.
int scratch_address(int dev, void** out) {
    if (dev < 0 || dev >= kMaxDevices) return SPLASH_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_scratch_ptr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return SPLASH_ERR_CUDA;
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return SPLASH_OK;
}

}  // namespace
}  // namespace splash

extern "C" {

int splash_decode_attn_noalloc(const splash_attn_desc* desc, const void* q, const void* kv_pool,
                               const int32_t* block_table, const int32_t* ctx_lens, int head_lo,
                               int head_hi, int64_t tok_lo, int64_t tok_hi, float* out,
                               float* lse, splash_stream_t stream) {
    const size_t need = splash_decode_workspace_size(desc, head_lo, head_hi);
    if (need == 0) {
        // invalid or unsupported shape (or no device): let the regular entry point report
        // which, with the same argument checks in the same order
        return splash_decode_attn(desc, q, kv_pool, block_table, ctx_lens, head_lo, head_hi,
                                  tok_lo, tok_hi, out, lse, nullptr, 0, stream);
    }
    if (need > splash::kNoAllocScratchBytes) return SPLASH_ERR_WORKSPACE;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return SPLASH_ERR_CUDA;
    void* scratch = nullptr;
    const int st = splash::scratch_address(dev, &scratch);
    if (st != SPLASH_OK) return st;
    return splash_decode_attn(desc, q, kv_pool, block_table, ctx_lens, head_lo, head_hi, tok_lo,
                              tok_hi, out, lse, scratch, splash::kNoAllocScratchBytes, stream);
}

// The status word lives at the start of the scratch array (the plan header), where the
// decode kernels of the last splash_decode_attn_noalloc call on this device left it.
int splash_noalloc_status(uint32_t* flags, splash_stream_t stream) {
    if (!flags) return SPLASH_ERR_INVALID_ARG;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return SPLASH_ERR_CUDA;
    void* scratch = nullptr;
    const int st = splash::scratch_address(dev, &scratch);
    if (st != SPLASH_OK) return st;
    if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
        return SPLASH_ERR_CUDA;
    if (cudaMemcpy(flags, scratch, sizeof(uint32_t), cudaMemcpyDeviceToHost) != cudaSuccess)
        return SPLASH_ERR_CUDA;
    return SPLASH_OK;
}

}  // extern "C"
