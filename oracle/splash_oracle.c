/*
 * splash_oracle.c -- plain fp64 CPU oracle for the paged decode-attention hot path.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may call, link or load
 * this file: only the tests, the package smoke check and the benchmark's CPU
 * baseline leg use it.  It shares no code, header, table or helper with the CUDA
 * library; the two meet only in the seeded inputs they are both given.
 *
 * Source: "SPLASH: Switching Parallel Layouts of Attention with Seamless Handoff
 * for LLM Serving".
 *   - Abstract: with few or no KV heads, where a request's KV cache lives is
 *     independent of how attention weights are sharded, so the four layouts
 *     (TP, CP, DP-attention, DOP) differ only in who owns weights and cache;
 *     a layout switch moves the state that is not yet in place (KV pages) and
 *     hands off at a batch boundary.
 *   - Appendix, Table 2: per-layout ownership -- TP reads every request's
 *     history for its head share, CP reads a B/T token share of every request
 *     ("ideal token partitioning"), DP-attention and DOP own whole requests.
 *
 * The pages print no formula for attention, for the merge of partial results or
 * for page migration.  What is computed here is the textbook definition each of
 * those operations reaches exactly (up to rounding order):
 *
 *   token set   T_r = [max(tok_lo,0), min(tok_hi < 0 ? L_r : tok_hi, L_r))
 *   key/value   k_t = pool[block_table[r][t / P]][t % P][0 : d_qk],
 *               v_t = k_t[0 : d_v]                      (one shared latent head)
 *   score       s_t = scale * sum_d q[r][h][d] * k_t[d]
 *   output      M = max_t s_t,  Z = sum_t exp(s_t - M),
 *               out[r][h][j] = sum_t exp(s_t - M) * v_t[j] / Z,
 *               lse[r][h]    = M + ln Z                 (natural log)
 *   empty T_r   out = 0, lse = -inf
 *
 * Partial results over disjoint token sets merge by their log-sum-exp weights:
 *   M = max_s lse_s, w_s = exp(lse_s - M),
 *   out = sum_s w_s out_s / sum_s w_s,  lse = M + ln sum_s w_s,
 *   and if every lse_s is -inf then out = 0, lse = -inf.
 *
 * Migration copies whole pages byte for byte: dst[dst_ids[i]] = src[src_ids[i]].
 *
 * All arithmetic is IEEE double; bf16 inputs are widened exactly (bf16 bits are
 * the top half of an IEEE single).  No blocking, fusion or reordering beyond the
 * definition: scores are computed first, then the max, then the sums.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

/* Exact bf16 -> double: the 16 bf16 bits are the high half of an IEEE binary32. */
static double bf16_to_double(uint16_t bits) {
    uint32_t u = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* Number of OpenMP threads the oracle would use (1 without OpenMP). */
int oracle_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

void oracle_set_num_threads(int n) {
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

/*
 * Paged decode attention for one ownership slice (Abstract; Appendix, Table 2):
 * heads [head_lo, head_hi) of all B requests given, over the token range
 * [tok_lo, tok_hi) clipped to each request's context (tok_hi < 0 means "to the
 * end of the context").  A request subset (DP-attention / DOP ownership) is the
 * caller passing only that subset's rows.
 *
 *   q           bf16 bits [B][H][d_qk]
 *   pool        bf16 bits [num_pages][P][d_qk] (one shared KV head; see
 *               oracle_decode_attn_kv for several)
 *   block_table int32 [B][max_pages]
 *   ctx_lens    int32 [B]
 *   out         double [B][H][d_v]; only rows [head_lo, head_hi) are written
 *   lse         double [B][H];      only rows [head_lo, head_hi) are written
 *
 * Returns 0 on success, -1 on an invalid argument (nothing is written then), -2
 * if a block-table entry needed by the slice is outside [0, num_pages).
 */
/* The same with Hkv key/value heads (grouped-query attention; the Abstract's "few
 * or no KV heads"): the pool is [num_pages][Hkv][P][d_qk] and query head h reads KV
 * head h / (H / Hkv).  Hkv = 1 is the shared latent head of MLA. */
int oracle_decode_attn_kv(int B, int H, int Hkv, int d_qk, int d_v, int P, int num_pages,
                          int max_pages, double scale, const uint16_t* q, const uint16_t* pool,
                          const int32_t* block_table, const int32_t* ctx_lens, int head_lo,
                          int head_hi, int64_t tok_lo, int64_t tok_hi, double* out, double* lse) {
    if (B < 0 || H <= 0 || Hkv <= 0 || H % Hkv != 0 || d_qk <= 0 || d_v <= 0 || d_v > d_qk ||
        P <= 0 || num_pages < 0 || max_pages < 0 || head_lo < 0 || head_hi > H ||
        head_lo >= head_hi || tok_lo < 0 || (tok_hi >= 0 && tok_hi < tok_lo))
        return -1;
    const int group = H / Hkv;   /* query heads per KV head */
    /* Every page id the slice needs must name a pool page. */
    for (int r = 0; r < B; ++r) {
        int64_t L = ctx_lens[r];
        if (L < 0 || L > (int64_t)max_pages * P) return -1;
        int64_t hi = (tok_hi < 0) ? L : (tok_hi < L ? tok_hi : L);
        if (hi <= tok_lo) continue;
        for (int64_t pg = tok_lo / P; pg <= (hi - 1) / P; ++pg) {
            int32_t id = block_table[(int64_t)r * max_pages + pg];
            if (id < 0 || id >= num_pages) return -2;
        }
    }
    const int nh = head_hi - head_lo;
    int status = 0;
#pragma omp parallel for collapse(2) schedule(dynamic, 1)
    for (int r = 0; r < B; ++r) {
        for (int hh = 0; hh < nh; ++hh) {
            const int h = head_lo + hh;
            const int64_t L = ctx_lens[r];
            const int64_t lo = tok_lo;
            const int64_t hi = (tok_hi < 0) ? L : (tok_hi < L ? tok_hi : L);
            double* o = out + ((int64_t)r * H + h) * d_v;
            if (hi <= lo) { /* empty token set */
                for (int j = 0; j < d_v; ++j) o[j] = 0.0;
                lse[(int64_t)r * H + h] = -INFINITY;
                continue;
            }
            const int64_t n = hi - lo;
            double* s = (double*)malloc((size_t)n * sizeof(double));
            if (!s) {
#pragma omp atomic write
                status = -3;
                continue;
            }
            const uint16_t* qrow = q + ((int64_t)r * H + h) * d_qk;
            const int kvh = h / group;
            /* 1. scores s_t = scale * <q, k_t> */
            for (int64_t t = lo; t < hi; ++t) {
                int32_t page = block_table[(int64_t)r * max_pages + t / P];
                const uint16_t* k = pool + (((int64_t)page * Hkv + kvh) * P + t % P) * d_qk;
                double acc = 0.0;
                for (int d = 0; d < d_qk; ++d) acc += bf16_to_double(qrow[d]) * bf16_to_double(k[d]);
                s[t - lo] = scale * acc;
            }
            /* 2. M = max_t s_t */
            double M = -INFINITY;
            for (int64_t i = 0; i < n; ++i) if (s[i] > M) M = s[i];
            /* 3. Z = sum_t exp(s_t - M); out = sum_t exp(s_t - M) v_t / Z */
            double Z = 0.0;
            for (int j = 0; j < d_v; ++j) o[j] = 0.0;
            for (int64_t t = lo; t < hi; ++t) {
                double w = exp(s[t - lo] - M);
                Z += w;
                int32_t page = block_table[(int64_t)r * max_pages + t / P];
                const uint16_t* v = pool + (((int64_t)page * Hkv + kvh) * P + t % P) * d_qk;
                for (int j = 0; j < d_v; ++j) o[j] += w * bf16_to_double(v[j]);
            }
            for (int j = 0; j < d_v; ++j) o[j] /= Z;
            lse[(int64_t)r * H + h] = M + log(Z);
            free(s);
        }
    }
    return status;
}

int oracle_decode_attn(int B, int H, int d_qk, int d_v, int P, int num_pages, int max_pages,
                       double scale, const uint16_t* q, const uint16_t* pool,
                       const int32_t* block_table, const int32_t* ctx_lens, int head_lo,
                       int head_hi, int64_t tok_lo, int64_t tok_hi, double* out, double* lse) {
    return oracle_decode_attn_kv(B, H, 1, d_qk, d_v, P, num_pages, max_pages, scale, q, pool,
                                 block_table, ctx_lens, head_lo, head_hi, tok_lo, tok_hi, out, lse);
}

/*
 * Log-sum-exp merge of S partial results over disjoint token sets of the same
 * (request, head) rows -- the step that turns CP's per-rank token shares
 * (Appendix, Table 2: "ideal token partitioning") back into one result.
 *
 *   part_out double [S][R][d_v], part_lse double [S][R]  (R = rows, e.g. B*H)
 *   out      double [R][d_v],    lse      double [R]
 */
int oracle_lse_merge(int S, int64_t R, int d_v, const double* part_out, const double* part_lse,
                     double* out, double* lse) {
    if (S <= 0 || R < 0 || d_v <= 0) return -1;
#pragma omp parallel for schedule(static)
    for (int64_t row = 0; row < R; ++row) {
        double M = -INFINITY;
        for (int s = 0; s < S; ++s) {
            double l = part_lse[(int64_t)s * R + row];
            if (l > M) M = l;
        }
        double* o = out + row * d_v;
        if (M == -INFINITY) { /* every part empty */
            for (int j = 0; j < d_v; ++j) o[j] = 0.0;
            lse[row] = -INFINITY;
            continue;
        }
        double W = 0.0;
        for (int j = 0; j < d_v; ++j) o[j] = 0.0;
        for (int s = 0; s < S; ++s) {
            double w = exp(part_lse[(int64_t)s * R + row] - M);
            W += w;
            const double* po = part_out + ((int64_t)s * R + row) * d_v;
            for (int j = 0; j < d_v; ++j) o[j] += w * po[j];
        }
        for (int j = 0; j < d_v; ++j) o[j] /= W;
        lse[row] = M + log(W);
    }
    return 0;
}

/*
 * KV-page migration between block pools (Abstract: a switch moves the state
 * that is not yet where the next layout needs it): page dst_ids[i] of dst
 * becomes a byte copy of page src_ids[i] of src, for i < n.  Returns -1 if an
 * id is out of range (nothing is copied then).
 */
int oracle_kv_migrate(const uint8_t* src, uint8_t* dst, int64_t page_bytes, const int32_t* src_ids,
                      const int32_t* dst_ids, int n, int32_t src_num_pages, int32_t dst_num_pages) {
    if (page_bytes <= 0 || n < 0) return -1;
    for (int i = 0; i < n; ++i)
        if (src_ids[i] < 0 || src_ids[i] >= src_num_pages || dst_ids[i] < 0 ||
            dst_ids[i] >= dst_num_pages)
            return -1;
    for (int i = 0; i < n; ++i)
        memcpy(dst + (int64_t)dst_ids[i] * page_bytes, src + (int64_t)src_ids[i] * page_bytes,
               (size_t)page_bytes);
    return 0;
}
