/*
 * splash.h -- C ABI of the GB300 (sm_103a) paged MLA decode-attention hot path.
 *
 * Method: "SPLASH: Switching Parallel Layouts of Attention with Seamless Handoff
 * for LLM Serving".
 *   Abstract -- with few or no KV heads (MLA: one shared latent KV head), where a
 *     request's KV cache lives is decoupled from how attention weights are
 *     sharded, so the four attention layouts (TP, CP, DP-attention and DOP)
 *     differ only in who owns weights and cache; a layout switch moves the state
 *     that is not yet in place and hands off at a batch boundary.
 *   Appendix, Table 2 -- per-layout ownership: TP reads every request's history
 *     for a share of the heads; CP reads a B/T share of every request's tokens
 *     ("ideal token partitioning"); DP-attention and DOP own whole requests.
 *
 * One call of splash_decode_attn computes any of those ownership slices on one
 * GPU: a head range [head_lo, head_hi) (TP / DOP shard), a token range
 * [tok_lo, tok_hi) returning partial output plus log-sum-exp (CP), or whole
 * requests (DP-attention / DOP: pass only the owned requests' rows).
 * splash_lse_merge combines CP partials; splash_kv_migrate moves KV pages
 * between block pools for a handoff.
 *
 * Conventions shared by every entry point
 *   - Every pointer argument is DEVICE memory owned by the caller, unless stated
 *     otherwise.  The library allocates no device memory, keeps no reference to
 *     any buffer after the call returns, and never synchronises the stream.
 *   - Work is enqueued on `stream` (a cudaStream_t; NULL is the legacy default
 *     stream).  Buffers must stay alive until that work completes.
 *   - Arguments are validated on the host before anything is enqueued; a call
 *     that returns an error has enqueued nothing.  Launch failures are reported
 *     as SPLASH_ERR_CUDA (the CUDA error is not cleared from the device).
 *   - Calls are thread-safe; the only library state is a per-device cache of
 *     the SM count and of the dynamic shared memory opt-in.
 *   - The calling thread's current CUDA device must be the device that owns
 *     the pointers and the stream.
 */
#ifndef SPLASH_H_
#define SPLASH_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define SPLASH_API __attribute__((visibility("default")))
#else
#define SPLASH_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* ABI-identical to cudaStream_t / CUstream. */
typedef struct CUstream_st* splash_stream_t;

typedef enum {
    SPLASH_OK = 0,
    SPLASH_ERR_INVALID_ARG = -1, /* null pointer, bad range, misaligned pointer   */
    SPLASH_ERR_UNSUPPORTED = -2, /* shape outside what the kernels implement      */
    SPLASH_ERR_WORKSPACE = -3,   /* workspace smaller than the size query returns */
    SPLASH_ERR_CUDA = -4         /* a CUDA runtime / driver call failed           */
} splash_status;

/* Bits of the device-side status word (see splash_workspace_status). */
enum {
    SPLASH_DEVICE_TIMEOUT = 1u << 0,   /* a bounded wait gave up; outputs are invalid  */
    SPLASH_DEVICE_BAD_INPUT = 1u << 1  /* a needed page id or a context length was out of range */
};

/*
 * Shape of one paged decode batch.
 *   num_reqs          B, requests in this call (rows of q, block_table, ctx_lens, out, lse)
 *   num_heads         H, query heads per request (rows per request in q / out / lse)
 *   d_qk              key / query width: must be 576 (512 latent + 64 rope dims)
 *   d_v               value width: must be 512 (values are the latent prefix of the key)
 *   page_size         P, tokens per KV page: 16, 32, 64 or 128
 *   num_pages         pages in kv_pool
 *   max_pages_per_req row stride of block_table (entries per request)
 *   scale             softmax temperature applied to q.k (e.g. 1/sqrt(192)), fp32
 */
typedef struct {
    int32_t num_reqs;
    int32_t num_heads;
    int32_t d_qk;
    int32_t d_v;
    int32_t page_size;
    int32_t num_pages;
    int32_t max_pages_per_req;
    float scale;
} splash_attn_desc;

/*
 * Bytes of device workspace splash_decode_attn needs for this shape and head
 * range on the current device (it depends on B, head_hi - head_lo and the
 * device's SM count, not on the context lengths).  Returns 0 when the shape is
 * invalid or unsupported.
 */
SPLASH_API size_t splash_decode_workspace_size(const splash_attn_desc* desc, int head_lo, int head_hi);

/*
 * Paged decode attention for one ownership slice (Abstract; Appendix, Table 2).
 *
 * For every request r < B and head h in [head_lo, head_hi), over the token set
 *   T_r = [tok_lo, min(tok_hi < 0 ? ctx_lens[r] : tok_hi, ctx_lens[r]))
 * with key k_t = kv_pool[block_table[r][t / P]][t % P][0:576] and value
 * v_t = k_t[0:512]:
 *   s_t = scale * q[r][h] . k_t
 *   out[r][h][j] = sum_t exp(s_t - m) v_t[j] / sum_t exp(s_t - m)
 *   lse[r][h]    = m + ln sum_t exp(s_t - m)          (natural log, m = max_t s_t)
 * An empty T_r gives out = 0 and lse = -inf.  A token range [tok_lo, tok_hi)
 * that is a share of the context yields the CP partial (out normalised over the
 * share, lse of the share) that splash_lse_merge combines.
 *
 *   q           bf16 [B][H][576], 16-byte aligned rows (contiguous)
 *   kv_pool     bf16 [num_pages][P][576], 16-byte aligned, contiguous
 *   block_table int32 [B][max_pages_per_req]; entries for pages at or beyond
 *               ceil(ctx_len / P) are never read
 *   ctx_lens    int32 [B], 0 <= ctx_lens[r] <= max_pages_per_req * P
 *   head_lo/hi  0 <= head_lo < head_hi <= H
 *   tok_lo      >= 0;  tok_hi < 0 means "to the end of each context", else tok_hi >= tok_lo
 *   out         fp32 [B][H][512]: only rows [head_lo, head_hi) are written
 *   lse         fp32 [B][H]:      only rows [head_lo, head_hi) are written
 *   workspace   >= splash_decode_workspace_size(...) bytes, 256-byte aligned; reused
 *               across calls on one stream; must not be shared by calls that may
 *               overlap on the device
 * Slot contents of KV pages beyond ctx_len (tail slots, unused pages) may hold
 * any bits, NaN included: they never reach an output.  A block-table id outside
 * [0, num_pages) for a needed page is not read: that page's tokens are left out of
 * T_r.  A context length outside [0, max_pages_per_req * P] is clamped into it.
 * Both set SPLASH_DEVICE_BAD_INPUT.
 * Returns SPLASH_OK or a splash_status error (nothing enqueued on error).
 */
SPLASH_API int splash_decode_attn(const splash_attn_desc* desc, const void* q, const void* kv_pool,
                       const int32_t* block_table, const int32_t* ctx_lens, int head_lo,
                       int head_hi, int64_t tok_lo, int64_t tok_hi, float* out, float* lse,
                       void* workspace, size_t ws_bytes, splash_stream_t stream);

/*
 * Per-request token ranges and storage rows for splash_decode_attn_ex.  Every
 * pointer may be NULL, and NULL restores the splash_decode_attn behaviour for
 * that field.
 *   tok_lo, tok_hi  int32 [B] device: request r's token set is
 *                   [tok_lo[r], min(tok_hi[r] < 0 ? ctx_len : tok_hi[r], ctx_len)),
 *                   for CP with an uneven share per request (the "ideal token
 *                   partitioning" of Appendix, Table 2, for ragged contexts).  A NULL
 *                   array uses the call's scalar for every request.  A negative
 *                   tok_lo[r] is bad input: it is taken as 0 and sets
 *                   SPLASH_DEVICE_BAD_INPUT.
 *   rows            int32 [B] device: request r of the call reads row rows[r] of q,
 *                   block_table and ctx_lens and writes row rows[r] of out and lse.
 *                   Those arrays then have num_rows rows.  This lets a DP-attention /
 *                   DOP owner decode its subset of a batch in place.  The rows must be
 *                   distinct.  A row outside [0, num_rows) is bad input: nothing is
 *                   read or written for that request, and SPLASH_DEVICE_BAD_INPUT is set.
 *   num_rows        rows of q / block_table / ctx_lens / out / lse when rows != NULL
 *                   (>= 1); ignored otherwise (the arrays then have B rows).
 *   max_sms         at most this many SMs run the call's persistent decode grid (0: all
 *                   of them), leaving the rest to work on other streams, e.g. a
 *                   background splash_kv_migrate of a layout handoff.  Must be >= 0.
 *   num_kv_heads    KV heads per token, Hkv (0 or 1: the one shared latent head).  With
 *                   Hkv > 1 (grouped-query attention, the Abstract's "few KV heads") the
 *                   pool is bf16 [num_pages][Hkv][P][576] and query head h reads KV head
 *                   h / (H / Hkv).  H must be a multiple of Hkv.  H / Hkv must be at most 64
 *                   or a multiple of 64, and head_lo a multiple of min(H / Hkv, 64); other
 *                   shapes return SPLASH_ERR_UNSUPPORTED.
 */
typedef struct {
    const int32_t* tok_lo;
    const int32_t* tok_hi;
    const int32_t* rows;
    int32_t num_rows;
    int32_t max_sms;
    int32_t num_kv_heads;
} splash_decode_ext;

/*
 * splash_decode_attn with per-request token ranges and storage rows.
 * `ext` may be NULL.  desc->num_reqs is B, the number of requests in the call
 * and the length of the ext arrays.  The scalars tok_lo / tok_hi apply to every
 * request whose array is NULL, and are validated as in splash_decode_attn.  The
 * workspace size is splash_decode_workspace_size(desc, head_lo, head_hi), as
 * for splash_decode_attn.  Alignment: the ext arrays 4 bytes.  Otherwise the
 * same arguments, results and errors as splash_decode_attn.
 */
SPLASH_API int splash_decode_attn_ex(const splash_attn_desc* desc, const splash_decode_ext* ext,
                          const void* q, const void* kv_pool, const int32_t* block_table,
                          const int32_t* ctx_lens, int head_lo, int head_hi, int64_t tok_lo,
                          int64_t tok_hi, float* out, float* lse, void* workspace,
                          size_t ws_bytes, splash_stream_t stream);

/*
 * splash_decode_attn without a caller workspace.  This entry point has no
 * counterpart in the paper; it exists for callers that cannot allocate device
 * memory at the point where they decode: code inside CUDA stream capture (a
 * cudaMalloc there is not captured and can invalidate the capture), serving loops
 * whose memory is owned by another allocator or capped by a fixed budget, and
 * plugins that are handed only input and output buffers.
 *
 * Same arguments, results and errors as splash_decode_attn, minus the workspace:
 * the scratch is a 32 MiB array inside the library, resident on every GPU that
 * loads the library until the process exits.  No cudaMalloc, cudaFree or other
 * allocating routine is called.
 *   - A shape whose splash_decode_workspace_size exceeds 32 MiB is rejected with
 *     SPLASH_ERR_WORKSPACE.  With 128 heads on a 152-SM GB300 that is more than
 *     51 requests per call; a 16-head shard takes up to 868.
 *   - The first call on a device resolves the array's device address
 *     (cudaGetSymbolAddress with that device current); make that first call
 *     before any stream capture.
 *   - Every call on a device shares the one array and it keeps the last call's
 *     contents (each call rewrites all of it that it reads).  Calls that may
 *     overlap on the GPU (different streams, or graphs replayed concurrently)
 *     race on it: serialise them.
 *   - The device status word (SPLASH_DEVICE_* bits) of the last call on the
 *     device is read with splash_noalloc_status.
 */
SPLASH_API int splash_decode_attn_noalloc(const splash_attn_desc* desc, const void* q,
                                          const void* kv_pool, const int32_t* block_table,
                                          const int32_t* ctx_lens, int head_lo, int head_hi,
                                          int64_t tok_lo, int64_t tok_hi, float* out, float* lse,
                                          splash_stream_t stream);

/*
 * Device status word of the most recent splash_decode_attn_noalloc call on the
 * current device (the SPLASH_DEVICE_* bits that splash_workspace_status reports
 * for a caller workspace).  Like splash_decode_attn_noalloc it has no counterpart
 * in the paper.  Synchronises `stream` (the stream of that call), then copies 4
 * bytes from the library's scratch to *flags (host pointer).  The word belongs to
 * the last call on the device, whichever stream issued it.  Allocates nothing.
 * Returns SPLASH_OK or an error.
 */
SPLASH_API int splash_noalloc_status(uint32_t* flags, splash_stream_t stream);

/*
 * Log-sum-exp merge of S partial results over disjoint token sets (the CP
 * combine; Appendix, Table 2, ideal token partitioning):
 *   m = max_s part_lse[s][b][h], w_s = exp(part_lse[s][b][h] - m),
 *   out[b][h] = sum_s w_s part_out[s][b][h] / sum_s w_s,  lse[b][h] = m + ln sum_s w_s;
 *   rows whose parts are all empty (-inf) give out = 0, lse = -inf.
 *   part_out fp32 [S][B][H][d_v], part_lse fp32 [S][B][H]; out fp32 [B][H][d_v],
 *   lse fp32 [B][H].  S >= 1, d_v a positive multiple of 4, 16-byte aligned
 *   part_out / out.  out may not alias part_out.
 */
SPLASH_API int splash_lse_merge(const float* part_out, const float* part_lse, int S, int B, int H, int d_v,
                     float* out, float* lse, splash_stream_t stream);

/*
 * KV-page migration between block pools (Abstract: a switch moves the state
 * that is not yet where the next layout needs it):
 *   dst_pool page dst_ids[i]  <-  byte copy of src_pool page src_ids[i],  i < n_pages.
 *   page_bytes  size of one page (P * 576 * 2 for this cache), multiple of 16
 *   src_ids, dst_ids int32 [n_pages] (device); dst_ids must be distinct; when
 *               src_pool == dst_pool the two id sets must be disjoint
 *   src_num_pages, dst_num_pages  pool sizes: a pair with an id outside its pool
 *               is skipped (no byte of either pool is touched for it)
 * Pools must be 16-byte aligned.  The caller rewrites its block tables.
 */
SPLASH_API int splash_kv_migrate(const void* src_pool, void* dst_pool, size_t page_bytes,
                      const int32_t* src_ids, const int32_t* dst_ids, int n_pages,
                      int32_t src_num_pages, int32_t dst_num_pages, splash_stream_t stream);

/*
 * Reads the device status word of a decode workspace (SPLASH_DEVICE_* bits set
 * by the most recent splash_decode_attn that used it): synchronises `stream`,
 * then copies 4 bytes to *flags (host pointer).  Returns SPLASH_OK or an error.
 */
SPLASH_API int splash_workspace_status(const void* workspace, uint32_t* flags, splash_stream_t stream);

/* Static string for a splash_status value. */
SPLASH_API const char* splash_status_string(int status);

#ifdef __cplusplus
}
#endif

#endif /* SPLASH_H_ */
