"""The layout load calculator against Appendix, Table 2 of "SPLASH: Switching
Parallel Layouts of Attention with Seamless Handoff for LLM Serving" (the table
as printed, from tests/golden/), and its one-GPU call patterns: every layout's
calls cover each (request, head, token) exactly once."""
import json
import math
import os

import numpy as np
import pytest

from layout_agnostic_paged_gb300 import layouts as L

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "table2_busiest_rank_load.json")


def _eval(expr, B, T):
    return eval(expr, {"__builtins__": {}}, {"B": B, "T": T, "ceil": math.ceil})


def test_busiest_rank_load_is_table_2():
    g = json.load(open(GOLDEN))
    assert set(g["table"]) == set(L.LAYOUTS)
    for B, T in g["cases"]:
        for layout, row in g["table"].items():
            got = L.busiest_rank_load(layout, B, T)
            want = [_eval(e, B, T) for e in row]
            assert [got.weights, got.kv_stored, got.kv_read, got.attn_work] == pytest.approx(want), \
                (layout, B, T)


def test_owner_entries_equal_b_over_t_when_t_divides_b():
    for B, T in [(16, 8), (64, 16), (9, 3)]:
        for layout in ("DP-attention", "DOP"):
            ld = L.busiest_rank_load(layout, B, T)
            assert ld.kv_stored == ld.kv_read == ld.attn_work == B // T


def test_unknown_layout_and_bad_sizes_are_rejected():
    with pytest.raises(ValueError):
        L.busiest_rank_load("PP", 4, 2)
    with pytest.raises(ValueError):
        L.busiest_rank_load("TP", 4, 0)
    with pytest.raises(ValueError):
        L.emulated_calls("TP", [5, 6], 6, 4)   # 6 heads over 4 ranks


@pytest.mark.parametrize("layout", L.LAYOUTS)
@pytest.mark.parametrize("ctx,H,T", [([5, 0, 13, 7, 1], 8, 4), ([3], 4, 4), ([9, 9, 9], 6, 3)])
def test_calls_cover_every_request_head_token_once(layout, ctx, H, T):
    B = len(ctx)
    cover = np.zeros((B, H, max(ctx) if ctx and max(ctx) else 1), dtype=np.int64)
    for c in L.emulated_calls(layout, ctx, H, T):
        rows = c.rows if c.rows is not None else range(B)
        for k, r in enumerate(rows):   # per-request arrays are indexed by call position k
            lo = c.tok_lo[k] if c.tok_lo is not None else 0
            hi = c.tok_hi[k] if c.tok_hi is not None else ctx[r]
            cover[r, c.head_lo:c.head_hi, lo:min(hi, ctx[r])] += 1
    for r in range(B):
        assert (cover[r, :, :ctx[r]] == 1).all(), (layout, r)
        assert (cover[r, :, ctx[r]:] == 0).all()


def test_busiest_rank_bytes_match_table_2_for_equal_lengths():
    Lr, B, T = 1000, 16, 8
    for layout in L.LAYOUTS:
        want = L.busiest_rank_load(layout, B, T).kv_read * Lr * L.BYTES_PER_KV_TOKEN
        assert L.busiest_rank_kv_bytes(layout, [Lr] * B, T) == want


def test_ragged_lengths_make_the_busiest_rank_the_longest_owner():
    ctx = [100, 5000, 10, 10]
    # DP-attention with T = 2: rank 0 owns requests 0, 2; rank 1 owns 1, 3
    assert L.busiest_rank_kv_bytes("DP-attention", ctx, 2) == 5010 * L.BYTES_PER_KV_TOKEN
    # CP splits every request: the busiest share is at most one token per request over B/T
    cp = L.busiest_rank_kv_bytes("CP", ctx, 2) // L.BYTES_PER_KV_TOKEN
    assert sum(ctx) // 2 <= cp <= sum(ctx) // 2 + len(ctx)
    assert L.predicted_step_seconds("TP", ctx, 2, 1e12) == pytest.approx(
        sum(ctx) * L.BYTES_PER_KV_TOKEN / 1e12)
