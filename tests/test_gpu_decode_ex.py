"""GPU parity of splash_decode_attn_ex: per-request token ranges and storage rows
(marked gpu).

Per-request ranges are CP's "ideal token partitioning" of "SPLASH: Switching
Parallel Layouts of Attention with Seamless Handoff for LLM Serving", Appendix,
Table 2, for ragged contexts: every request contributes its own equal share, so
the shares' bounds differ per request.  Storage rows let a DP-attention / DOP
owner decode its subset of a batch in place (same table: whole requests).  Each
request is checked against the fp64 oracle called for that request alone with
its own scalar range.
"""
import pytest
import torch

from layout_agnostic_paged_gb300 import splash as S
from layout_agnostic_paged_gb300 import workloads as W
from tests.gpu_helpers import assert_attn_close, oracle_rows

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    S.load_library()


def _i32(xs):
    return torch.tensor(xs, dtype=torch.int32, device=DEV)


def _decode_ex(inp, lo=None, hi=None, rows=None, out=None, lse=None, tok_lo=0, tok_hi=-1,
               head_lo=0, head_hi=None, max_sms=0):
    R, H, _ = inp.q.shape
    head_hi = H if head_hi is None else head_hi
    if out is None:
        out = torch.full((R, H, 512), float("nan"), device=DEV)
    if lse is None:
        lse = torch.full((R, H), float("nan"), device=DEV)
    B = len(rows) if rows is not None else R
    ws = S.decode_workspace(inp.q, inp.pool, inp.block_table, W.MLA_SCALE, head_lo, head_hi,
                            num_reqs=B)
    S.splash_decode_attn_ex(inp.q, inp.pool, inp.block_table, inp.ctx_lens, head_lo, head_hi,
                            tok_lo, tok_hi, out, lse, ws, W.MLA_SCALE,
                            tok_lo_r=None if lo is None else _i32(lo),
                            tok_hi_r=None if hi is None else _i32(hi),
                            rows=None if rows is None else _i32(rows), max_sms=max_sms)
    return out, lse, ws


def _check_request(inp, out, lse, row, lo, hi, what, head_lo=0, head_hi=None):
    H = inp.q.shape[1]
    head_hi = H if head_hi is None else head_hi
    if 0 <= hi < lo:   # a per-request range that ends before it starts is the empty set
        hi = lo
    ro, rl = oracle_rows(inp, W.MLA_SCALE, row, head_lo, head_hi, tok_lo=lo, tok_hi=hi)
    assert_attn_close(out[row, head_lo:head_hi].cpu(), ro, lse[row, head_lo:head_hi].cpu(), rl, what)


@pytest.mark.parametrize("H,P", [(128, 64), (8, 16), (40, 64)])
def test_per_request_ranges_match_oracle(H, P):
    ctx = [300, 1024, 77, 2000, 513, 0, 129]
    inp = W.make_decode_inputs(ctx, H, P, seed=41 + H, device=DEV)
    lo = [0, 128, 50, 1000, 600, 0, 1]
    hi = [-1, 900, 40, 1999, -1, 10, 129]   # to the end, inside, empty, unaligned, beyond, empty ctx
    out, lse, ws = _decode_ex(inp, lo, hi)
    for r in range(len(ctx)):
        _check_request(inp, out, lse, r, lo[r], hi[r], f"request {r} [{lo[r]}, {hi[r]})")
    assert S.splash_workspace_status(ws) == 0


def test_only_one_bound_per_request():
    ctx = [700, 1500, 90]
    inp = W.make_decode_inputs(ctx, 128, 64, seed=45, device=DEV)
    out, lse, _ = _decode_ex(inp, lo=[10, 700, 0], tok_hi=1200)
    for r, lo in enumerate([10, 700, 0]):
        _check_request(inp, out, lse, r, lo, 1200, f"array lo, scalar hi, request {r}")
    out, lse, _ = _decode_ex(inp, hi=[100, 1499, -1], tok_lo=64)
    for r, hi in enumerate([100, 1499, -1]):
        _check_request(inp, out, lse, r, 64, hi, f"scalar lo, array hi, request {r}")


def test_per_request_cp_shares_merge_to_unsplit():
    """Each request split into 4 equal shares of its own length, merged by splash_lse_merge."""
    ctx = [4096, 1500, 333, 2050, 64, 1]
    n = 4
    inp = W.make_decode_inputs(ctx, 128, 64, seed=46, device=DEV)
    B = len(ctx)
    po = torch.empty(n, B, 128, 512, device=DEV)
    pl = torch.empty(n, B, 128, device=DEV)
    for i in range(n):
        lo = [L * i // n for L in ctx]
        hi = [L * (i + 1) // n for L in ctx]
        _decode_ex(inp, lo, hi, out=po[i], lse=pl[i])
    mo = torch.empty(B, 128, 512, device=DEV)
    ml = torch.empty(B, 128, device=DEV)
    S.splash_lse_merge(po, pl, mo, ml)
    for r in range(B):
        _check_request(inp, mo, ml, r, 0, -1, f"merged shares, request {r}")


def test_rows_decode_a_subset_in_place():
    ctx = [300, 900, 50, 2000, 129, 700]
    inp = W.make_decode_inputs(ctx, 64, 64, seed=47, device=DEV)
    rows = [4, 0, 5]
    out, lse, ws = _decode_ex(inp, rows=rows)
    for r in rows:
        _check_request(inp, out, lse, r, 0, -1, f"row {r}")
    others = [r for r in range(len(ctx)) if r not in rows]
    assert torch.isnan(out[others]).all() and torch.isnan(lse[others]).all(), "rows outside the call written"
    assert S.splash_workspace_status(ws) == 0


def test_rows_with_ranges_and_a_head_slice():
    ctx = [1000, 64, 2500, 480]
    inp = W.make_decode_inputs(ctx, 128, 64, seed=48, device=DEV)
    rows, lo, hi = [2, 3, 0], [256, 0, 1], [2304, 200, 999]
    out, lse, _ = _decode_ex(inp, lo, hi, rows, head_lo=32, head_hi=64)
    for r, a, b in zip(rows, lo, hi):
        _check_request(inp, out, lse, r, a, b, f"row {r} [{a}, {b}) heads 32..63", 32, 64)
    assert torch.isnan(out[:, :32]).all() and torch.isnan(out[:, 64:]).all()
    assert torch.isnan(out[1]).all()


def test_rows_in_any_order_match_the_oracle():
    """Whole requests decoded through a permutation of the rows match the oracle of
    each row."""
    ctx = [513, 77, 1024]
    inp = W.make_decode_inputs(ctx, 128, 64, seed=49, device=DEV)
    out, lse, _ = _decode_ex(inp, rows=[2, 1, 0])
    for r in range(3):
        _check_request(inp, out, lse, r, 0, -1, f"reversed rows, row {r}")


def test_bad_row_and_negative_start_are_flagged_and_skipped():
    ctx = [200, 300, 400]
    inp = W.make_decode_inputs(ctx, 16, 64, seed=50, device=DEV)
    out, lse, ws = _decode_ex(inp, rows=[1, 99])
    assert S.splash_workspace_status(ws) & S.SPLASH_DEVICE_BAD_INPUT
    _check_request(inp, out, lse, 1, 0, -1, "valid row next to a bad one")
    assert torch.isnan(out[[0, 2]]).all() and torch.isnan(lse[[0, 2]]).all()
    out, lse, ws = _decode_ex(inp, lo=[-5, 0, 100])
    assert S.splash_workspace_status(ws) & S.SPLASH_DEVICE_BAD_INPUT
    _check_request(inp, out, lse, 0, 0, -1, "negative start taken as 0")
    _check_request(inp, out, lse, 2, 100, -1, "request 2")


@pytest.mark.parametrize("max_sms", [1, 7, 16, 34, 80, 100000])
def test_sm_budget_changes_the_split_not_the_result(max_sms):
    """A decode grid held to max_sms SMs (the rest left to background work) cuts the
    tiles differently but computes the same attention."""
    ctx = [5000, 300, 2048, 129, 64]
    inp = W.make_decode_inputs(ctx, 128, 64, seed=51, device=DEV)
    out, lse, ws = _decode_ex(inp, max_sms=max_sms)
    for r in range(len(ctx)):
        _check_request(inp, out, lse, r, 0, -1, f"max_sms={max_sms} request {r}")
    assert S.splash_workspace_status(ws) == 0
    # the plan's cut: at most ceil(T / groups) tiles on a group; with at most 4 tiles per
    # group it uses the fewest groups that keep that count, else every group (<= T)
    hdr = ws[:16].cpu()
    G = int(hdr[4:8].view(torch.int32)[0])
    T = int(hdr[8:16].view(torch.int64)[0])
    assert T == sum(-(-L // 128) for L in ctx)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    groups = max(1, min(sms, max_sms) // 2)      # 128 heads: two head-group CTAs per group
    k = -(-T // groups)
    assert G == (-(-T // k) if k <= 4 else min(groups, T)), (G, T, groups)


def test_concurrent_share_calls_on_two_streams_with_half_the_sms():
    """Two CP share calls issued on two streams at once, each held to half the SMs and
    with its own workspace (the benchmark's pattern for small steps), then merged:
    the same result as the unsplit oracle."""
    ctx = [1024] * 6 + [700, 129]
    inp = W.make_decode_inputs(ctx, 128, 64, seed=52, device=DEV)
    B = len(ctx)
    half = torch.cuda.get_device_properties(0).multi_processor_count // 2
    po = torch.full((2, B, 128, 512), float("nan"), device=DEV)
    pl = torch.full((2, B, 128), float("nan"), device=DEV)
    wss = [S.decode_workspace(inp.q, inp.pool, inp.block_table, W.MLA_SCALE) for _ in range(2)]
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    torch.cuda.synchronize()
    for i, (lo, hi) in enumerate([(0, 512), (512, -1)]):
        with torch.cuda.stream(streams[i]):
            S.splash_decode_attn_ex(inp.q, inp.pool, inp.block_table, inp.ctx_lens, 0, 128, lo, hi,
                                    po[i], pl[i], wss[i], W.MLA_SCALE, max_sms=half)
    torch.cuda.synchronize()
    mo = torch.empty(B, 128, 512, device=DEV)
    ml = torch.empty(B, 128, device=DEV)
    S.splash_lse_merge(po, pl, mo, ml)
    torch.cuda.synchronize()
    for ws in wss:
        assert S.splash_workspace_status(ws) == 0
    for r in range(B):
        _check_request(inp, mo, ml, r, 0, -1, f"two-stream shares, request {r}")
