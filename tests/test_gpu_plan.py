"""The split plan written into the decode workspace (marked gpu): every request's
tiles are cut into consecutive non-empty CTA-group ranges, partial slots are
distinct, and the cut is independent of physical page ids."""
import numpy as np
import pytest
import torch

from layout_agnostic_paged_gb300 import workloads as W
from tests.gpu_helpers import gpu_decode

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
REQ = np.dtype([("tile_begin", "<i8"), ("tile0", "<i4"), ("ntiles", "<i4"), ("lo", "<i4"),
                ("hi", "<i4"), ("ctx_len", "<i4"), ("first_grp", "<i4"), ("nsplit", "<i4"),
                ("slot_base", "<i4"), ("pad", "<i4", 2)])


def read_plan(ws, B):
    raw = ws.cpu().numpy()
    hdr = raw[:32]
    status = int(np.frombuffer(hdr[0:4], "<u4")[0])
    groups = int(np.frombuffer(hdr[4:8], "<i4")[0])
    T = int(np.frombuffer(hdr[8:16], "<i8")[0])
    req = np.frombuffer(raw[256:256 + 48 * B].tobytes(), REQ)
    return status, groups, T, req


@pytest.mark.parametrize("ctx,tok", [([1, 127, 128, 129, 300], (0, -1)),
                                     ([5000, 0, 70000, 3, 129], (0, -1)),
                                     ([4096] * 40, (1000, 3000)),
                                     ([64], (0, -1))])
def test_plan_cuts_are_consistent(ctx, tok):
    inp = W.make_decode_inputs(ctx, 16, 64, seed=len(ctx), device=DEV)
    _, _, ws = gpu_decode(inp, W.MLA_SCALE, tok_lo=tok[0], tok_hi=tok[1])
    torch.cuda.synchronize()
    status, G, T, req = read_plan(ws, len(ctx))
    assert status == 0
    assert T == int(req["ntiles"].sum()) and 0 <= G <= T
    starts = [(j * T) // G for j in range(G + 1)] if G else [0]
    assert all(starts[j] < starts[j + 1] for j in range(G))   # every group non-empty
    slots = []
    t = 0
    for r, p in enumerate(req):
        L = ctx[r]
        lo, hi = tok[0], (L if tok[1] < 0 else min(tok[1], L))
        if hi <= lo:
            assert p["ntiles"] == 0 and p["nsplit"] == 0
            continue
        assert (p["lo"], p["hi"]) == (lo, hi)
        assert p["ntiles"] == (hi + 127) // 128 - lo // 128
        assert p["tile_begin"] == t
        groups = {j for j in range(G) for x in range(t, t + p["ntiles"])
                  if starts[j] <= x < starts[j + 1]}
        assert p["first_grp"] == min(groups) and p["nsplit"] == len(groups)
        assert sorted(groups) == list(range(min(groups), max(groups) + 1))
        if p["nsplit"] > 1:
            slots += list(range(p["slot_base"], p["slot_base"] + p["nsplit"]))
        else:
            assert p["slot_base"] == -1
        t += int(p["ntiles"])
    assert len(slots) == len(set(slots))
