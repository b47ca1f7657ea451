"""Seeded synthetic inputs for paged MLA decode: the one module that both the CUDA
path's tests/benchmark and the fp64 oracle draw their inputs from.

It holds shapes, distributions and page layouts only -- none of the method's
arithmetic.  The workloads are the five synthetic configurations the hot path is
specified on, plus a ragged CP batch with per-request shares (the pages themselves
serve GLM-5.3 / DeepSeek-V3.2 with trained
weights and real prompts, which are not available; see "SPLASH: Switching
Parallel Layouts of Attention with Seamless Handoff for LLM Serving", Appendix,
Tables 4-6 for the B=16, 1,024..65,536-token sweeps these shapes stand in for).

Recipe (every tensor is a pure function of its seed):
  * q and the KV latent are N(0,1) float32 draws rounded to bf16 (round to
    nearest even), generated on the requested device with a seeded
    torch.Generator, in logical page order;
  * the pool holds the used pages plus 10% spare pages; logical page k of the
    concatenated requests is stored at physical id perm[k] for a seeded random
    permutation (so block tables are shuffled);
  * tail slots of every request's last page and every spare page are NaN
    ("poison"): a correct kernel never lets them reach an output;
  * unused block-table entries are -1;
  * ragged context lengths are floor(exp(U(ln lo, ln hi))) from
    numpy.random.default_rng(seed), clamped to [lo, hi].
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np
import torch

D_QK = 576          # 512 latent + 64 rope dims: the one shared KV head
D_V = 512           # values are the latent prefix of the key
MLA_SCALE = 1.0 / math.sqrt(192.0)
TILE_TOKENS = 128   # not used by the inputs; exported for tests that pick ragged sizes


@dataclass(frozen=True)
class Workload:
    """One synthetic decode batch description (ownership slices are per call)."""
    name: str
    ctx_lens: tuple
    num_heads: int
    page_size: int
    seed: int
    scale: float = MLA_SCALE
    spare_frac: float = 0.10
    # ownership slices exercised by the configuration
    head_shards: int = 1          # TP / DOP: number of equal head shards
    token_splits: int = 1         # CP: number of equal contiguous token ranges
    per_request_splits: bool = False  # CP shares of each request's own length (not one span)
    num_kv_heads: int = 1         # KV heads per token (1: the shared latent head)
    migrate_frac: float = 0.0     # handoff: fraction of requests whose pages move
    notes: str = ""

    @property
    def batch(self) -> int:
        return len(self.ctx_lens)

    @property
    def kv_tokens(self) -> int:
        return int(sum(self.ctx_lens))


def ragged_ctx_lens(n: int, lo: int, hi: int, seed: int) -> tuple:
    """Log-uniform context lengths in [lo, hi] (seeded numpy Generator)."""
    rng = np.random.default_rng(seed)
    x = np.floor(np.exp(rng.uniform(math.log(lo), math.log(hi), size=n))).astype(np.int64)
    return tuple(int(v) for v in np.clip(x, lo, hi))


def tiny() -> Workload:
    return Workload("tiny decode: B=2, ctx 64/100, page 16, 8 heads", (64, 100), 8, 16, seed=1000)


def full_heads() -> Workload:
    return Workload("MLA decode full heads: B=16, ctx 1024, 128 heads, page 64",
                    (1024,) * 16, 128, 64, seed=1001)


def cp_long() -> Workload:
    return Workload("CP long context: B=16, ctx 65536, 128 heads, page 64, 8 token ranges",
                    (65536,) * 16, 128, 64, seed=1002, token_splits=8)


def head_shard() -> Workload:
    return Workload("TP/DOP head shard: B=128, ctx 4096, 16 of 128 heads per call, page 64",
                    (4096,) * 128, 128, 64, seed=1003, head_shards=8)


def ragged_handoff() -> Workload:
    return Workload("ragged mixed batch + handoff: 256 requests, ctx log-uniform 512..131072, "
                    "128 heads, page 64, migrate 25%",
                    ragged_ctx_lens(256, 512, 131072, seed=1004), 128, 64, seed=1004,
                    migrate_frac=0.25)


def ragged_small() -> Workload:
    """The ragged + handoff batch scaled to 64 requests (same length distribution): a
    pool of a few GB, small enough for multi-pass profiler captures of one decode call."""
    return Workload("ragged mixed batch + handoff, scaled: 64 requests, ctx log-uniform "
                    "512..131072, 128 heads, page 64, migrate 25%",
                    ragged_ctx_lens(64, 512, 131072, seed=1007), 128, 64, seed=1007,
                    migrate_frac=0.25)


def ragged_cp() -> Workload:
    return Workload("ragged CP: 128 requests, ctx log-uniform 512..131072, 128 heads, page 64, "
                    "8 token shares of each request's own length",
                    ragged_ctx_lens(128, 512, 131072, seed=1005), 128, 64, seed=1005,
                    token_splits=8, per_request_splits=True)


def gqa() -> Workload:
    return Workload("grouped-query decode: B=16, ctx 8192, 128 query heads over 8 KV heads, "
                    "page 64", (8192,) * 16, 128, 64, seed=1006, token_splits=2, num_kv_heads=8)


def per_request_ranges(w: Workload) -> torch.Tensor:
    """int32 [splits][2][B]: share i of request r is [L_r i / n, L_r (i + 1) / n)
    (the ideal token partitioning of each request's own context)."""
    n = max(2, w.token_splits)
    L = torch.tensor(w.ctx_lens, dtype=torch.int64)
    return torch.stack([torch.stack([L * i // n, L * (i + 1) // n]) for i in range(n)]).to(torch.int32)


ALL = {"tiny": tiny, "full_heads": full_heads, "cp_long": cp_long, "head_shard": head_shard,
       "ragged_handoff": ragged_handoff, "ragged_small": ragged_small, "ragged_cp": ragged_cp,
       "gqa": gqa}


@dataclass
class DecodeInputs:
    q: torch.Tensor            # bf16 [B][H][576]
    pool: torch.Tensor         # bf16 [num_pages][P][576]
    block_table: torch.Tensor  # int32 [B][max_pages]
    ctx_lens: torch.Tensor     # int32 [B]
    perm: torch.Tensor         # int64 [num_pages]: logical page k -> physical id perm[k]
    pages_per_req: list = field(default_factory=list)

    @property
    def num_pages(self) -> int:
        return int(self.pool.shape[0])

    @property
    def page_size(self) -> int:
        return int(self.pool.shape[1])


def _gen(device, seed: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def make_decode_inputs(ctx_lens, num_heads: int, page_size: int, seed: int, device="cpu",
                       spare_frac: float = 0.10, perm_seed: int | None = None,
                       poison: bool = True, max_pages: int | None = None,
                       chunk_pages: int = 4096, num_kv_heads: int = 1) -> DecodeInputs:
    """Build q, a shuffled paged KV pool and block tables for the given lengths.

    The logical KV content depends only on ``seed`` (and the lengths), the
    physical placement only on ``perm_seed`` (default: seed + 1), so two calls
    differing in ``perm_seed`` hold the same cache under different page ids.
    """
    device = torch.device(device)
    ctx = [int(x) for x in ctx_lens]
    B = len(ctx)
    P = int(page_size)
    ppr = [(L + P - 1) // P for L in ctx]
    used = sum(ppr)
    spare = max(1, int(math.ceil(spare_frac * used))) if spare_frac > 0 else 0
    num_pages = used + spare
    mp = max(ppr) if ppr else 0
    if max_pages is not None:
        assert max_pages >= mp
        mp = max_pages
    mp = max(mp, 1)

    g_perm = _gen("cpu", seed + 1 if perm_seed is None else perm_seed)
    perm = torch.randperm(num_pages, generator=g_perm)

    g_q = _gen(device, seed)
    q = torch.randn((B, num_heads, D_QK), generator=g_q, device=device,
                    dtype=torch.float32).to(torch.bfloat16)

    # one KV head: [num_pages][P][576]; several: [num_pages][Hkv][P][576]
    page_shape = (P, D_QK) if num_kv_heads == 1 else (num_kv_heads, P, D_QK)
    pool = torch.empty((num_pages,) + page_shape, dtype=torch.bfloat16, device=device)
    g_kv = _gen(device, seed + 7)
    perm_dev = perm.to(device)
    step = max(1, chunk_pages // num_kv_heads)
    for k0 in range(0, used, step):
        k1 = min(used, k0 + step)
        chunk = torch.randn((k1 - k0,) + page_shape, generator=g_kv, device=device,
                            dtype=torch.float32).to(torch.bfloat16)
        pool[perm_dev[k0:k1]] = chunk
    if spare:
        pool[perm_dev[used:]] = float("nan") if poison else 0.0

    bt = torch.full((B, mp), -1, dtype=torch.int32)
    k = 0
    tails = []
    for r, n in enumerate(ppr):
        if n:
            bt[r, :n] = perm[k:k + n].to(torch.int32)
            rem = ctx[r] - (n - 1) * P
            if rem < P:
                tails.append((int(perm[k + n - 1]), rem))
        k += n
    if poison:
        for pid, rem in tails:
            if num_kv_heads == 1:
                pool[pid, rem:] = float("nan")
            else:
                pool[pid, :, rem:] = float("nan")
    return DecodeInputs(q=q, pool=pool, block_table=bt.to(device),
                        ctx_lens=torch.tensor(ctx, dtype=torch.int32, device=device), perm=perm,
                        pages_per_req=ppr)


def make_workload_inputs(w: Workload, device="cpu", **kw) -> DecodeInputs:
    return make_decode_inputs(w.ctx_lens, w.num_heads, w.page_size, w.seed, device=device,
                              spare_frac=w.spare_frac, num_kv_heads=w.num_kv_heads, **kw)


@dataclass
class MigrationPlan:
    requests: list             # request indices whose pages move
    src_ids: torch.Tensor      # int32 [n]: page ids in the source pool
    dst_ids: torch.Tensor      # int32 [n]: fresh distinct ids in the destination pool
    dst_num_pages: int
    new_block_table: torch.Tensor  # int32 [len(requests)][max_pages]: rows for the dst pool


def make_migration(inp: DecodeInputs, frac: float, seed: int, dst_spare_frac: float = 0.10
                   ) -> MigrationPlan:
    """Seeded handoff plan: move all pages of a random ``frac`` of the requests to a
    second pool at fresh, distinct, random page ids."""
    B = inp.block_table.shape[0]
    rng = np.random.default_rng(seed + 11)
    n_move = int(round(frac * B))
    reqs = sorted(int(x) for x in rng.choice(B, size=n_move, replace=False)) if n_move else []
    bt = inp.block_table.cpu()
    src = []
    rows = []
    for r in reqs:
        n = inp.pages_per_req[r]
        src.append(bt[r, :n].clone())
        rows.append(n)
    n_pages = int(sum(rows))
    dst_num_pages = n_pages + max(1, int(math.ceil(dst_spare_frac * n_pages)))
    g = _gen("cpu", seed + 13)
    dst_perm = torch.randperm(dst_num_pages, generator=g)[:n_pages].to(torch.int32)
    new_bt = torch.full((len(reqs), bt.shape[1]), -1, dtype=torch.int32)
    k = 0
    for i, n in enumerate(rows):
        new_bt[i, :n] = dst_perm[k:k + n]
        k += n
    src_ids = torch.cat(src).to(torch.int32) if src else torch.empty(0, dtype=torch.int32)
    return MigrationPlan(requests=reqs, src_ids=src_ids, dst_ids=dst_perm,
                         dst_num_pages=dst_num_pages, new_block_table=new_bt)
