"""Every workload at its full size, in the launch configuration the benchmark times,
against the fp64 oracle over every output element (marked gpu).

The benchmark's step (bench.step_pattern) is run as the benchmark runs it: its calls
alternate between two streams with one workspace each, small calls share the SMs,
and the ragged workload's step decodes the batch, migrates a quarter of the
requests' pages to a second pool and decodes again as two calls owning request
subsets.  Each output the step writes is compared with the oracle on that call's
own inputs ("SPLASH: Switching Parallel Layouts of Attention with Seamless Handoff
for LLM Serving", Abstract: layouts differ only in who owns weights and cache, and a
handoff moves KV state; Appendix, Table 2: head shares, ideal token partitioning,
whole-request ownership), and migrated pages are compared bit for bit.
"""
import os
import sys

import numpy as np
import pytest
import torch

import oracle
from layout_agnostic_paged_gb300 import splash as S
from layout_agnostic_paged_gb300 import workloads as W
from tests.gpu_helpers import assert_attn_close, oracle_full

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
import bench  # noqa: E402

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    S.load_library()


def _run_step(name):
    w = W.ALL[name]()
    inp = W.make_workload_inputs(w, device=DEV)
    step = bench.Step(w, inp, DEV)
    step.run()
    torch.cuda.synchronize()
    for ws in step.wss:
        assert S.splash_workspace_status(ws) == 0
    return w, inp, step


def _host(t):
    return t.cpu().double().numpy()


@pytest.mark.parametrize("name", ["tiny", "full_heads", "gqa"])
def test_single_and_two_share_steps(name):
    w, inp, step = _run_step(name)
    ro, rl = oracle_full(inp, w.scale)
    assert_attn_close(step.out.cpu(), ro, step.lse.cpu(), rl, f"{name} step")
    if step.phases[-1][0] == "merge":
        for i, c in enumerate(step.phases[0][1]):
            po, pl = oracle_full(inp, w.scale, tok_lo=c.tok_lo, tok_hi=c.tok_hi)
            assert_attn_close(step.po[i].cpu(), po, step.pl[i].cpu(), pl, f"{name} share {i}")


def test_cp_long_context_every_share_and_the_merge():
    """B=16, ctx 65,536, 128 heads: each of the 8 token shares against the oracle's
    share, the merged result and one unsplit call against the unsplit oracle."""
    w, inp, step = _run_step("cp_long")
    calls = step.phases[0][1]
    assert len(calls) == 8
    for i, c in enumerate(calls):
        po, pl = oracle_full(inp, w.scale, tok_lo=c.tok_lo, tok_hi=c.tok_hi)
        assert_attn_close(step.po[i].cpu(), po, step.pl[i].cpu(), pl, f"CP share {i}")
    ro, rl = oracle_full(inp, w.scale)
    assert_attn_close(step.out.cpu(), ro, step.lse.cpu(), rl, "CP merged")
    out = torch.full_like(step.out, float("nan"))
    lse = torch.full_like(step.lse, float("nan"))
    ws = S.decode_workspace(inp.q, inp.pool, inp.block_table, w.scale)
    S.splash_decode_attn(inp.q, inp.pool, inp.block_table, inp.ctx_lens, 0, w.num_heads, 0, -1,
                         out, lse, ws, w.scale)
    assert S.splash_workspace_status(ws) == 0
    assert_attn_close(out.cpu(), ro, lse.cpu(), rl, "CP unsplit call")


def test_head_shard_every_shard():
    """B=128, ctx 4,096: 8 calls of 16 heads each, concatenated, against the oracle."""
    w, inp, step = _run_step("head_shard")
    ro, rl = oracle_full(inp, w.scale)
    assert_attn_close(step.out.cpu(), ro, step.lse.cpu(), rl, "concatenated head shards")


def test_ragged_cp_per_request_shares():
    """128 ragged requests, 8 shares of each request's own length, merged."""
    w, inp, step = _run_step("ragged_cp")
    ro, rl = oracle_full(inp, w.scale)
    assert_attn_close(step.out.cpu(), ro, step.lse.cpu(), rl, "ragged CP merged")


def test_ragged_handoff_before_and_after_the_migration():
    """256 requests, log-uniform 512..131,072, 128 heads: the whole-batch decode, the
    migration of 25% of the requests' pages (bit-exact), and the rerun as two calls
    (remaining requests on pool 1, moved ones on pool 2 at their new page ids), each
    against the oracle run on that call's own pool and block table."""
    w, inp, step = _run_step("ragged_handoff")
    mig = step.mig
    # pages: bit-exact copies
    a = inp.pool.index_select(0, step.src_ids.long()).view(torch.int16)
    b = step.pool2.index_select(0, step.dst_ids.long()).view(torch.int16)
    assert torch.equal(a, b)
    del a, b
    q = oracle.bf16_bits(inp.q)
    ctx = inp.ctx_lens.cpu().numpy()
    bt1 = inp.block_table.cpu().numpy()
    bt2 = step.dev["bt2"].cpu().numpy()
    pool1 = oracle.bf16_bits(inp.pool)
    # before the handoff: the whole batch on pool 1
    ro, rl = oracle.decode_attn(q, pool1, bt1, ctx, w.scale)
    pre_o, pre_l = step.outs["pre"]
    assert_attn_close(pre_o.cpu(), ro, pre_l.cpu(), rl, "before the handoff")
    # after: remaining requests on pool 1, moved ones on pool 2
    moved = np.array(mig.requests)
    keep = np.array([r for r in range(w.batch) if r not in set(mig.requests)])
    ko, kl = oracle.decode_attn(q[keep], pool1, bt1[keep], ctx[keep], w.scale)
    del pool1
    assert_attn_close(step.out[keep].cpu(), ko, step.lse[keep].cpu(), kl, "rerun, pool 1")
    pool2 = oracle.bf16_bits(step.pool2)
    mo, ml = oracle.decode_attn(q[moved], pool2, bt2[moved], ctx[moved], w.scale)
    assert_attn_close(step.out[moved].cpu(), mo, step.lse[moved].cpu(), ml, "rerun, pool 2")
