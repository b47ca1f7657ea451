"""Busiest-rank load of SPLASH's attention layouts, and the one-GPU call pattern
that emulates each layout.

"SPLASH: Switching Parallel Layouts of Attention with Seamless Handoff for LLM
Serving", Appendix, Table 2 gives, for B equal-length requests on T ranks, the
busiest rank's share of the attention weights, of the KV histories it stores,
of the histories it reads per decode step, and of the attention work (counted
in one request's attention):

    layout         weights   KV stored   KV read    attention work
    TP             WA / T    B           B          B / T
    CP             WA        B / T       B / T      B / T
    DP-attention   WA        ceil(B/T)   ceil(B/T)  ceil(B/T)
    DOP            WA / T    ceil(B/T)   ceil(B/T)  ceil(B/T)

with count-balanced request ownership and ideal token partitioning for CP.  The
table's caption converts loads into time with an equation the pages do not
print, so the time estimate here is only the plain reading: the busiest rank's
KV bytes read divided by a measured decode bandwidth (the caller supplies it).

On one GPU a layout becomes a list of decode calls, one per rank, each naming
the slice that rank owns (Abstract: where a request's KV cache lives is decoupled
from how attention is sharded, so every layout reads the same paged cache):
TP a head range, CP a per-request token share (merged afterwards by log-sum-exp),
DP-attention and DOP a count-balanced subset of the requests.
"""
from __future__ import annotations

import math
from dataclasses import dataclass

LAYOUTS = ("TP", "CP", "DP-attention", "DOP")
BYTES_PER_KV_TOKEN = 576 * 2   # one shared latent KV head: 512 latent + 64 rope, bf16


@dataclass(frozen=True)
class RankLoad:
    """Busiest-rank load in Table 2's units: weights as a fraction of the attention
    weights WA, KV in histories (one request's cache), work in request-attentions."""
    weights: float
    kv_stored: float
    kv_read: float
    attn_work: float


def busiest_rank_load(layout: str, B: int, T: int) -> RankLoad:
    """Appendix, Table 2, for B equal-length requests on T ranks."""
    if B < 0 or T < 1:
        raise ValueError("need B >= 0 requests and T >= 1 ranks")
    owned = math.ceil(B / T)   # count-balanced request ownership
    if layout == "TP":
        return RankLoad(1.0 / T, B, B, B / T)
    if layout == "CP":
        return RankLoad(1.0, B / T, B / T, B / T)
    if layout == "DP-attention":
        return RankLoad(1.0, owned, owned, owned)
    if layout == "DOP":
        return RankLoad(1.0 / T, owned, owned, owned)
    raise ValueError(f"unknown layout {layout!r}; expected one of {LAYOUTS}")


@dataclass(frozen=True)
class RankCall:
    """One rank's decode call on one GPU (arguments of splash_decode_attn_ex)."""
    rank: int
    head_lo: int
    head_hi: int
    rows: tuple | None        # storage rows of the owned requests (None: all, in order)
    tok_lo: tuple | None      # per-request token range start (None: 0)
    tok_hi: tuple | None      # per-request token range end (None: to the end)


def owned_requests(B: int, T: int, rank: int) -> tuple:
    """Count-balanced ownership: request r belongs to rank r mod T."""
    return tuple(range(rank, B, T))


def emulated_calls(layout: str, ctx_lens, H: int, T: int) -> list:
    """The T calls that emulate `layout` on one GPU; together they compute every
    (request, head, token) once.  CP's calls return partials that splash_lse_merge
    combines; the other layouts write disjoint rows of one output."""
    B = len(ctx_lens)
    if T < 1:
        raise ValueError("need T >= 1 ranks")
    calls = []
    for i in range(T):
        if layout == "TP":
            if H % T:
                raise ValueError("TP needs the heads to divide evenly over the ranks")
            calls.append(RankCall(i, i * H // T, (i + 1) * H // T, None, None, None))
        elif layout == "CP":
            # ideal token partitioning of each request's own context
            lo = tuple(int(L) * i // T for L in ctx_lens)
            hi = tuple(int(L) * (i + 1) // T for L in ctx_lens)
            calls.append(RankCall(i, 0, H, None, lo, hi))
        elif layout in ("DP-attention", "DOP"):
            calls.append(RankCall(i, 0, H, owned_requests(B, T, i), None, None))
        else:
            raise ValueError(f"unknown layout {layout!r}; expected one of {LAYOUTS}")
    return calls


def busiest_rank_kv_bytes(layout: str, ctx_lens, T: int) -> int:
    """KV bytes the busiest rank reads in one step for these (possibly ragged) lengths:
    the ranks' call slices, not Table 2's equal-length idealisation.  (The head range
    does not change what a call reads, so any head count dividing T will do.)"""
    per_rank = []
    for c in emulated_calls(layout, ctx_lens, T, T):
        if c.rows is not None:
            toks = sum(int(ctx_lens[r]) for r in c.rows)
        elif c.tok_lo is not None:
            toks = sum(h - l for l, h in zip(c.tok_lo, c.tok_hi))
        else:
            toks = sum(int(L) for L in ctx_lens)
        per_rank.append(toks * BYTES_PER_KV_TOKEN)
    return max(per_rank) if per_rank else 0


def predicted_step_seconds(layout: str, ctx_lens, T: int, decode_bytes_per_s: float) -> float:
    """Busiest-rank KV read time at a measured decode bandwidth (the plain reading
    of the time conversion the pages cite but do not print)."""
    if decode_bytes_per_s <= 0:
        raise ValueError("need a positive measured bandwidth")
    return busiest_rank_kv_bytes(layout, ctx_lens, T) / decode_bytes_per_s
