"""splash_decode_attn_noalloc: the decode entry point for callers that cannot
allocate device memory where they decode (for instance inside stream capture, or
under an allocator they do not own).  It must give the same results as the
regular entry point with a caller workspace, call after call, match the fp64
oracle, leave a clear device status word, and reject shapes whose scratch need
exceeds its fixed 32 MiB.  This file is collected last."""
import pytest
import torch

from layout_agnostic_paged_gb300 import splash as S
from layout_agnostic_paged_gb300 import workloads as W
from tests.gpu_helpers import assert_attn_close, oracle_full

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _run_noalloc(inp, scale, head_lo, head_hi, tok_lo=0, tok_hi=-1):
    B, H, _ = inp.q.shape
    out = torch.full((B, H, 512), float("nan"), device=DEV)
    lse = torch.full((B, H), float("nan"), device=DEV)
    S.splash_decode_attn_noalloc(inp.q, inp.pool, inp.block_table, inp.ctx_lens, head_lo, head_hi,
                                 tok_lo, tok_hi, out, lse, scale)
    return out, lse


@pytest.mark.parametrize("ctx,H,P,hl,hh,tok", [
    ([1024] * 16, 128, 64, 0, 128, (0, -1)),          # full heads
    ([4096] * 8, 128, 64, 32, 48, (0, -1)),           # one 16-head shard
    ([1, 127, 300, 5000], 8, 16, 0, 8, (100, 2000)),  # ragged, a CP-style token range
])
def test_noalloc_matches_workspace_entry_point_twice(ctx, H, P, hl, hh, tok):
    inp = W.make_decode_inputs(ctx, H, P, seed=len(ctx) + H, device=DEV)
    B = len(ctx)
    ref_o = torch.full((B, H, 512), float("nan"), device=DEV)
    ref_l = torch.full((B, H), float("nan"), device=DEV)
    ws = S.decode_workspace(inp.q, inp.pool, inp.block_table, W.MLA_SCALE, hl, hh)
    S.splash_decode_attn(inp.q, inp.pool, inp.block_table, inp.ctx_lens, hl, hh, tok[0], tok[1],
                         ref_o, ref_l, ws, W.MLA_SCALE)
    ro = ref_o[:, hl:hh].cpu().double().numpy()
    rl = ref_l[:, hl:hh].cpu().double().numpy()
    oo, ol = oracle_full(inp, W.MLA_SCALE, head_lo=hl, head_hi=hh, tok_lo=tok[0], tok_hi=tok[1])
    for call in range(2):                       # two calls in a row share the scratch
        o, l = _run_noalloc(inp, W.MLA_SCALE, hl, hh, tok[0], tok[1])
        assert S.splash_noalloc_status() == 0   # synchronises the stream
        assert_attn_close(o[:, hl:hh].cpu(), ro, l[:, hl:hh].cpu(), rl, f"noalloc call {call}")
        assert_attn_close(o[:, hl:hh].cpu(), oo[:, hl:hh], l[:, hl:hh].cpu(), ol[:, hl:hh],
                          f"noalloc call {call} vs oracle")
        # rows outside the head slice are never written
        assert torch.isnan(o[:, :hl]).all() and torch.isnan(o[:, hh:]).all()


def test_noalloc_status_word_reports_bad_input():
    """A bad page id in a no-allocation call is flagged in the scratch's status word, and
    the next clean call clears it."""
    inp = W.make_decode_inputs([200, 64], 16, 64, seed=7, device=DEV)
    good = inp.block_table.clone()
    inp.block_table[0, 1] = 10_000_000
    _run_noalloc(inp, W.MLA_SCALE, 0, 16)
    assert S.splash_noalloc_status() & S.SPLASH_DEVICE_BAD_INPUT
    inp.block_table.copy_(good)
    _run_noalloc(inp, W.MLA_SCALE, 0, 16)
    assert S.splash_noalloc_status() == 0


def test_noalloc_rejects_shapes_beyond_its_scratch():
    inp = W.make_decode_inputs([64] * 512, 128, 64, seed=3, device=DEV)
    with pytest.raises(S.SplashError) as e:
        _run_noalloc(inp, W.MLA_SCALE, 0, 128)
    assert e.value.code == S.SPLASH_ERR_WORKSPACE
