"""Every layout's one-GPU call pattern from the load calculator (TP head ranges,
CP per-request token shares merged by log-sum-exp, DP-attention / DOP request
subsets decoded in place) gives the unsplit result of the fp64 oracle (marked gpu).

"SPLASH: Switching Parallel Layouts of Attention with Seamless Handoff for LLM
Serving", Abstract (layouts differ only in ownership) and Appendix, Table 2.
"""
import pytest
import torch

from layout_agnostic_paged_gb300 import layouts as LY
from layout_agnostic_paged_gb300 import splash as S
from layout_agnostic_paged_gb300 import workloads as W
from tests.gpu_helpers import assert_attn_close, oracle_full

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _i32(xs):
    return None if xs is None else torch.tensor(xs, dtype=torch.int32, device=DEV)


def run_layout(inp, layout, T):
    B, H, _ = inp.q.shape
    ctx = inp.ctx_lens.cpu().tolist()
    calls = LY.emulated_calls(layout, ctx, H, T)
    out = torch.full((B, H, 512), float("nan"), device=DEV)
    lse = torch.full((B, H), float("nan"), device=DEV)
    if layout == "CP":
        po = torch.empty(T, B, H, 512, device=DEV)
        pl = torch.empty(T, B, H, device=DEV)
    for c in calls:
        n = len(c.rows) if c.rows is not None else B
        if n == 0:
            continue
        ws = S.decode_workspace(inp.q, inp.pool, inp.block_table, W.MLA_SCALE, c.head_lo, c.head_hi,
                                num_reqs=n)
        o, l = (po[c.rank], pl[c.rank]) if layout == "CP" else (out, lse)
        S.splash_decode_attn_ex(inp.q, inp.pool, inp.block_table, inp.ctx_lens, c.head_lo,
                                c.head_hi, 0, -1, o, l, ws, W.MLA_SCALE, tok_lo_r=_i32(c.tok_lo),
                                tok_hi_r=_i32(c.tok_hi), rows=_i32(c.rows))
        assert S.splash_workspace_status(ws) == 0
    if layout == "CP":
        S.splash_lse_merge(po, pl, out, lse)
    return out, lse


@pytest.mark.parametrize("layout", LY.LAYOUTS)
@pytest.mark.parametrize("ctx,H,T", [([700, 33, 2048, 129, 1000, 0, 512], 128, 4),
                                     ([300, 4100, 77], 64, 8)])
def test_layout_call_patterns_give_the_unsplit_result(layout, ctx, H, T):
    inp = W.make_decode_inputs(ctx, H, 64, seed=60 + T, device=DEV)
    out, lse = run_layout(inp, layout, T)
    ro, rl = oracle_full(inp, W.MLA_SCALE)
    assert_attn_close(out.cpu(), ro, lse.cpu(), rl, f"{layout} on {T} ranks")
