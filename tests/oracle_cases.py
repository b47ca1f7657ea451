"""Small hand-built inputs for pinning the oracle (CPU only, no method arithmetic).

Values are chosen exactly representable in bf16 so that the bits both sides read
are the values written here.
"""
from __future__ import annotations

import numpy as np

D_QK = 576
D_V = 512


def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float values to bf16 (nearest even) and return the uint16 bits."""
    f = np.ascontiguousarray(x, dtype=np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    rounding = 0x7FFF + ((u >> 16) & 1)
    bits = ((u + rounding) >> 16).astype(np.uint16)
    nan = np.isnan(f)
    bits[nan] = 0x7FC0
    return bits


def from_bf16_bits(b: np.ndarray) -> np.ndarray:
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def paged(tokens_per_req, page_size, page_ids=None, poison=True, spare=1, num_heads=1):
    """Lay out per-request token rows [L_r][576] (float) into a paged pool.

    page_ids: optional list (per request) of physical page ids; default packs pages
    in order.  Returns (pool_bits, block_table, ctx_lens).
    """
    P = page_size
    ppr = [(len(t) + P - 1) // P for t in tokens_per_req]
    used = sum(ppr)
    num_pages = used + spare
    if page_ids is None:
        ids, k = [], 0
        for n in ppr:
            ids.append(list(range(k, k + n)))
            k += n
        page_ids = ids
    pool = np.full((num_pages, P, D_QK), np.nan if poison else 0.0, dtype=np.float32)
    mp = max(max(ppr), 1)
    bt = np.full((len(tokens_per_req), mp), -1, dtype=np.int32)
    for r, toks in enumerate(tokens_per_req):
        toks = np.asarray(toks, dtype=np.float32).reshape(-1, D_QK)
        for i, pid in enumerate(page_ids[r]):
            bt[r, i] = pid
            rows = toks[i * P:(i + 1) * P]
            pool[pid, :rows.shape[0]] = rows
    ctx = np.array([len(np.asarray(t).reshape(-1, D_QK)) for t in tokens_per_req], dtype=np.int32)
    return to_bf16_bits(pool), bt, ctx


def random_case(rng, ctx_lens, num_heads, page_size, scale_kv=1.0, shuffle=True):
    """Random bf16 q / tokens with shuffled physical page ids; returns a dict."""
    toks = [rng.standard_normal((L, D_QK)).astype(np.float32) * scale_kv for L in ctx_lens]
    q = rng.standard_normal((len(ctx_lens), num_heads, D_QK)).astype(np.float32)
    P = page_size
    ppr = [(L + P - 1) // P for L in ctx_lens]
    used = sum(ppr)
    perm = rng.permutation(used + 2) if shuffle else np.arange(used + 2)
    ids, k = [], 0
    for n in ppr:
        ids.append([int(x) for x in perm[k:k + n]])
        k += n
    pool, bt, ctx = paged(toks, P, ids, spare=2)
    qb = to_bf16_bits(q)
    toks_exact = [from_bf16_bits(to_bf16_bits(t)) for t in toks]
    return dict(q=qb, pool=pool, bt=bt, ctx=ctx, tokens=toks_exact, page_ids=ids)


def random_gqa_case(rng, ctx_lens, num_heads, num_kv_heads, page_size):
    """Random bf16 q and per-KV-head tokens in a shuffled pool [pages][Hkv][P][576]
    (NaN in unused slots); tokens[r][j] are request r's KV-head-j rows."""
    Hkv, P = num_kv_heads, page_size
    toks = [[rng.standard_normal((L, D_QK)).astype(np.float32) for _ in range(Hkv)]
            for L in ctx_lens]
    q = rng.standard_normal((len(ctx_lens), num_heads, D_QK)).astype(np.float32)
    ppr = [(L + P - 1) // P for L in ctx_lens]
    used = sum(ppr)
    perm = rng.permutation(used + 2)
    pool = np.full((used + 2, Hkv, P, D_QK), np.nan, dtype=np.float32)
    bt = np.full((len(ctx_lens), max(max(ppr), 1)), -1, dtype=np.int32)
    k = 0
    for r, L in enumerate(ctx_lens):
        for i in range(ppr[r]):
            pid = int(perm[k])
            k += 1
            bt[r, i] = pid
            for j in range(Hkv):
                rows = toks[r][j][i * P:(i + 1) * P]
                pool[pid, j, :rows.shape[0]] = rows
    exact = [[from_bf16_bits(to_bf16_bits(t)) for t in per_head] for per_head in toks]
    return dict(q=to_bf16_bits(q), pool=to_bf16_bits(pool), bt=bt,
                ctx=np.array(ctx_lens, dtype=np.int32), tokens=exact)
