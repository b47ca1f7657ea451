"""Seeded random decode calls against the fp64 oracle (marked gpu).

Each case draws a call shape the fixed tests do not pin one by one: head counts from 8
to 192 (head groups of 8..64 heads, several groups per CTA group), page sizes 16..128,
ragged contexts with empty requests, a head slice, a scalar or per-request token range,
a request subset given as storage rows in any order, and an SM budget.  Every written
output row is compared with the oracle run for that request alone, rows outside the
slice and requests outside the subset must stay untouched, and the device status word
must be clear ("SPLASH: Switching Parallel Layouts of Attention with Seamless Handoff
for LLM Serving", Abstract and Appendix, Table 2: every ownership slice computes the
same attention).
"""
import numpy as np
import pytest
import torch

from layout_agnostic_paged_gb300 import splash as S
from layout_agnostic_paged_gb300 import workloads as W
from tests.gpu_helpers import assert_attn_close, oracle_rows

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
CASES = 24


@pytest.fixture(scope="module", autouse=True)
def _lib():
    S.load_library()


def draw(case):
    rng = np.random.default_rng(700 + case)
    H = int(rng.choice([8, 16, 24, 40, 64, 96, 100, 128, 192]))
    P = int(rng.choice([16, 32, 64, 128]))
    R = int(rng.integers(1, 9))                       # rows of the batch
    ctx = [int(x) for x in rng.integers(0, 3000, size=R)]
    if R > 2:
        ctx[int(rng.integers(0, R))] = 0              # an empty request
    if rng.random() < 0.5:
        head_lo, head_hi = 0, H
    else:
        head_lo = int(rng.integers(0, H))
        head_hi = int(rng.integers(head_lo + 1, H + 1))
    rows = None
    if rng.random() < 0.4:                            # a subset of the rows, in any order
        n = int(rng.integers(1, R + 1))
        rows = [int(x) for x in rng.permutation(R)[:n]]
    B = len(rows) if rows is not None else R
    mode = rng.choice(["all", "scalar", "per_request"])
    tok_lo, tok_hi, lo_r, hi_r = 0, -1, None, None
    if mode == "scalar":
        tok_lo = int(rng.integers(0, 1500))
        tok_hi = -1 if rng.random() < 0.3 else int(rng.integers(tok_lo, 3200))
    elif mode == "per_request":
        lo_r = [int(x) for x in rng.integers(0, 1500, size=B)]
        hi_r = [-1 if rng.random() < 0.3 else int(lo + rng.integers(0, 2000)) for lo in lo_r]
    max_sms = int(rng.choice([0, 0, 2, 7, 34]))
    return dict(H=H, P=P, ctx=ctx, head_lo=head_lo, head_hi=head_hi, rows=rows, tok_lo=tok_lo,
                tok_hi=tok_hi, lo_r=lo_r, hi_r=hi_r, max_sms=max_sms, seed=700 + case)


def _i32(xs):
    return None if xs is None else torch.tensor(xs, dtype=torch.int32, device=DEV)


@pytest.mark.parametrize("case", range(CASES))
def test_random_call_matches_oracle(case):
    c = draw(case)
    inp = W.make_decode_inputs(c["ctx"], c["H"], c["P"], seed=c["seed"], device=DEV)
    R, H = len(c["ctx"]), c["H"]
    out = torch.full((R, H, 512), float("nan"), device=DEV)
    lse = torch.full((R, H), float("nan"), device=DEV)
    B = len(c["rows"]) if c["rows"] is not None else R
    ws = S.decode_workspace(inp.q, inp.pool, inp.block_table, W.MLA_SCALE, c["head_lo"],
                            c["head_hi"], num_reqs=B)
    S.splash_decode_attn_ex(inp.q, inp.pool, inp.block_table, inp.ctx_lens, c["head_lo"],
                            c["head_hi"], c["tok_lo"], c["tok_hi"], out, lse, ws, W.MLA_SCALE,
                            tok_lo_r=_i32(c["lo_r"]), tok_hi_r=_i32(c["hi_r"]),
                            rows=_i32(c["rows"]), max_sms=c["max_sms"])
    assert S.splash_workspace_status(ws) == 0, c
    hl, hh = c["head_lo"], c["head_hi"]
    owned = c["rows"] if c["rows"] is not None else list(range(R))
    for i, row in enumerate(owned):
        lo = c["lo_r"][i] if c["lo_r"] is not None else c["tok_lo"]
        hi = c["hi_r"][i] if c["hi_r"] is not None else c["tok_hi"]
        if 0 <= hi < lo:   # a per-request range that ends before it starts is empty
            hi = lo
        ro, rl = oracle_rows(inp, W.MLA_SCALE, row, hl, hh, tok_lo=lo, tok_hi=hi)
        assert_attn_close(out[row, hl:hh].cpu(), ro, lse[row, hl:hh].cpu(), rl,
                          f"case {case} {c} row {row}")
    # nothing outside the slice or the owned rows is written
    assert torch.isnan(out[:, :hl]).all() and torch.isnan(out[:, hh:]).all()
    others = [r for r in range(R) if r not in set(owned)]
    if others:
        assert torch.isnan(out[others]).all() and torch.isnan(lse[others]).all()
