"""GPU parity of paged decode attention against the fp64 oracle (marked gpu).

Every call goes through the C ABI (ctypes binding) into the CUDA kernels; the
oracle sees the same bf16 bits.  Ownership slices follow "SPLASH: Switching
Parallel Layouts of Attention with Seamless Handoff for LLM Serving", Appendix,
Table 2: head shares (TP / DOP), token shares merged by log-sum-exp (CP) and
whole-request subsets (DP-attention / DOP).
"""
import numpy as np
import pytest
import torch

from layout_agnostic_paged_gb300 import splash as S
from layout_agnostic_paged_gb300 import workloads as W
from tests.gpu_helpers import assert_attn_close, gpu_decode, oracle_full, oracle_rows

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    S.load_library()


def _inputs(ctx, H, P, seed, **kw):
    return W.make_decode_inputs(ctx, H, P, seed, device=DEV, **kw)


def test_tiny_workload_full_parity():
    w = W.tiny()
    inp = W.make_workload_inputs(w, device=DEV)
    out, lse, _ = gpu_decode(inp, w.scale)
    ro, rl = oracle_full(inp, w.scale)
    assert_attn_close(out.cpu(), ro, lse.cpu(), rl, "tiny")


@pytest.mark.parametrize("ctx,H,P", [
    ([1, 127, 128, 129, 300], 8, 16),
    ([5, 64, 65, 1000, 2], 16, 64),
    ([129, 255, 256, 257], 128, 64),
    ([700, 33], 100, 32),
    ([1, 1, 1], 8, 128),
])
def test_ragged_lengths_and_page_sizes(ctx, H, P):
    inp = _inputs(ctx, H, P, seed=sum(ctx) + H)
    out, lse, _ = gpu_decode(inp, W.MLA_SCALE)
    ro, rl = oracle_full(inp, W.MLA_SCALE)
    assert_attn_close(out.cpu(), ro, lse.cpu(), rl, f"ctx={ctx} H={H} P={P}")


def test_full_heads_workload_full_parity():
    w = W.full_heads()
    inp = W.make_workload_inputs(w, device=DEV)
    out, lse, _ = gpu_decode(inp, w.scale)
    ro, rl = oracle_full(inp, w.scale)
    assert_attn_close(out.cpu(), ro, lse.cpu(), rl, "full heads")


def test_head_shards_write_only_their_rows_and_concatenate():
    inp = _inputs([300, 64, 1000, 7], 128, 64, seed=21)
    full_o, full_l, _ = gpu_decode(inp, W.MLA_SCALE)
    o = torch.full_like(full_o, float("nan"))
    l = torch.full_like(full_l, float("nan"))
    for s in range(8):
        gpu_decode(inp, W.MLA_SCALE, 16 * s, 16 * s + 16, out=o, lse=l)
        # rows of later shards are still untouched
        if s < 7:
            assert torch.isnan(o[:, 16 * (s + 1):]).all() and torch.isnan(l[:, 16 * (s + 1):]).all()
    ro, rl = oracle_full(inp, W.MLA_SCALE)
    assert_attn_close(o.cpu(), ro, l.cpu(), rl, "concatenated shards")
    assert_attn_close(o.cpu(), full_o.cpu().double().numpy(), l.cpu(),
                      full_l.cpu().double().numpy(), "shards vs unsplit")


def test_cp_token_ranges_merge_to_unsplit():
    ctx = [2048, 1500, 4096, 100]
    inp = _inputs(ctx, 128, 64, seed=22)
    splits = 4
    span = 1024
    po = torch.empty(splits, 4, 128, 512, device=DEV)
    pl = torch.empty(splits, 4, 128, device=DEV)
    for i in range(splits):
        gpu_decode(inp, W.MLA_SCALE, tok_lo=i * span, tok_hi=(i + 1) * span, out=po[i], lse=pl[i])
    # an empty share: request 3 has 100 tokens, shares 1..3 are empty
    assert torch.isneginf(pl[1:, 3]).all() and (po[1:, 3] == 0).all()
    mo = torch.empty(4, 128, 512, device=DEV)
    ml = torch.empty(4, 128, device=DEV)
    S.splash_lse_merge(po, pl, mo, ml)
    ro, rl = oracle_full(inp, W.MLA_SCALE)
    assert_attn_close(mo.cpu(), ro, ml.cpu(), rl, "CP merged")
    # each partial against the oracle's partial
    for i in (0, 2):
        pro, prl = oracle_full(inp, W.MLA_SCALE, tok_lo=i * span, tok_hi=(i + 1) * span)
        assert_attn_close(po[i].cpu(), pro, pl[i].cpu(), prl, f"CP share {i}")


def test_request_subset_matches_rows_of_full_batch():
    inp = _inputs([300, 900, 50, 2000, 129], 16, 64, seed=23)
    full_o, full_l, _ = gpu_decode(inp, W.MLA_SCALE)
    sub = torch.tensor([1, 3], device=DEV)
    sub_inp = W.DecodeInputs(q=inp.q[sub].contiguous(), pool=inp.pool,
                             block_table=inp.block_table[sub].contiguous(),
                             ctx_lens=inp.ctx_lens[sub].contiguous(), perm=inp.perm,
                             pages_per_req=[inp.pages_per_req[1], inp.pages_per_req[3]])
    o, l, _ = gpu_decode(sub_inp, W.MLA_SCALE)
    assert_attn_close(o.cpu(), full_o[sub].cpu().double().numpy(), l.cpu(),
                      full_l[sub].cpu().double().numpy(), "subset vs full")
    ro, rl = oracle_full(sub_inp, W.MLA_SCALE)
    assert_attn_close(o.cpu(), ro, l.cpu(), rl, "subset vs oracle")


def test_physical_page_permutation_gives_identical_bits():
    a = _inputs([1000, 77, 513], 128, 64, seed=24, perm_seed=1)
    b = _inputs([1000, 77, 513], 128, 64, seed=24, perm_seed=2)
    assert not torch.equal(a.block_table, b.block_table)
    oa, la, _ = gpu_decode(a, W.MLA_SCALE)
    ob, lb, _ = gpu_decode(b, W.MLA_SCALE)
    assert torch.equal(oa, ob) and torch.equal(la, lb)


def test_repeat_calls_are_bit_identical():
    inp = _inputs([5000, 3, 700], 64, 64, seed=25)
    o1, l1, ws = gpu_decode(inp, W.MLA_SCALE)
    o2, l2, _ = gpu_decode(inp, W.MLA_SCALE, ws=ws)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_empty_contexts_and_ranges():
    inp = _inputs([0, 10, 0, 300], 16, 16, seed=26)
    out, lse, ws = gpu_decode(inp, W.MLA_SCALE)
    ro, rl = oracle_full(inp, W.MLA_SCALE)
    assert_attn_close(out.cpu(), ro, lse.cpu(), rl, "zero-length contexts")
    out, lse, _ = gpu_decode(inp, W.MLA_SCALE, tok_lo=400, tok_hi=-1)
    assert (out == 0).all() and torch.isneginf(lse).all()
    out, lse, _ = gpu_decode(inp, W.MLA_SCALE, tok_lo=7, tok_hi=7)
    assert (out == 0).all() and torch.isneginf(lse).all()
    assert S.splash_workspace_status(ws) == 0


def test_unaligned_token_ranges():
    inp = _inputs([1000, 333], 16, 16, seed=27)
    for lo, hi in [(5, 17), (100, 999), (127, 129), (0, 1)]:
        out, lse, _ = gpu_decode(inp, W.MLA_SCALE, tok_lo=lo, tok_hi=hi)
        ro, rl = oracle_full(inp, W.MLA_SCALE, tok_lo=lo, tok_hi=hi)
        assert_attn_close(out.cpu(), ro, lse.cpu(), rl, f"range [{lo},{hi})")


def test_bad_page_id_is_flagged_not_faulted():
    inp = _inputs([200, 64], 16, 64, seed=28)
    inp.block_table[0, 1] = 10_000_000
    out, lse, ws = gpu_decode(inp, W.MLA_SCALE)
    flags = S.splash_workspace_status(ws)
    assert flags & S.SPLASH_DEVICE_BAD_INPUT


def test_workspace_too_small_is_rejected():
    inp = _inputs([64], 8, 16, seed=29)
    ws = S.decode_workspace(inp.q, inp.pool, inp.block_table, W.MLA_SCALE)
    with pytest.raises(S.SplashError):
        gpu_decode(inp, W.MLA_SCALE, ws=ws[:ws.numel() - 256])


# ---------------------------------------------------------------- full-size configs

def test_cp_long_context_workload_sampled():
    """B=16, ctx 65,536, 128 heads: 8 token shares merged vs the unsplit call, and
    sampled rows against the oracle."""
    w = W.cp_long()
    inp = W.make_workload_inputs(w, device=DEV)
    B, H = w.batch, w.num_heads
    span = 65536 // w.token_splits
    po = torch.empty(w.token_splits, B, H, 512, device=DEV)
    pl = torch.empty(w.token_splits, B, H, device=DEV)
    for i in range(w.token_splits):
        gpu_decode(inp, w.scale, tok_lo=i * span, tok_hi=(i + 1) * span, out=po[i], lse=pl[i])
    mo = torch.empty(B, H, 512, device=DEV)
    ml = torch.empty(B, H, device=DEV)
    S.splash_lse_merge(po, pl, mo, ml)
    uo, ul, _ = gpu_decode(inp, w.scale)
    assert_attn_close(mo.cpu(), uo.cpu().double().numpy(), ml.cpu(), ul.cpu().double().numpy(),
                      "CP merged vs unsplit")
    for r, h0 in [(0, 0), (7, 61), (15, 125)]:
        ro, rl = oracle_rows(inp, w.scale, r, h0, h0 + 3)
        assert_attn_close(uo[r, h0:h0 + 3].cpu(), ro, ul[r, h0:h0 + 3].cpu(), rl, f"cp r{r}")
        ro, rl = oracle_rows(inp, w.scale, r, h0, h0 + 3, tok_lo=3 * span, tok_hi=4 * span)
        assert_attn_close(po[3, r, h0:h0 + 3].cpu(), ro, pl[3, r, h0:h0 + 3].cpu(), rl,
                          f"cp share r{r}")


def test_head_shard_workload_sampled():
    """B=128, ctx 4,096: 8 calls of 16 heads each; concatenation vs sampled oracle rows."""
    w = W.head_shard()
    inp = W.make_workload_inputs(w, device=DEV)
    B, H = w.batch, w.num_heads
    o = torch.full((B, H, 512), float("nan"), device=DEV)
    l = torch.full((B, H), float("nan"), device=DEV)
    ws = None
    for s in range(w.head_shards):
        _, _, ws = gpu_decode(inp, w.scale, 16 * s, 16 * s + 16, out=o, lse=l, ws=ws)
    assert torch.isfinite(o).all() and torch.isfinite(l).all()
    for r, h0 in [(0, 0), (64, 40), (127, 112)]:
        ro, rl = oracle_rows(inp, w.scale, r, h0, h0 + 16)
        assert_attn_close(o[r, h0:h0 + 16].cpu(), ro, l[r, h0:h0 + 16].cpu(), rl, f"shard r{r}")


def test_ragged_handoff_workload_sampled():
    """256 requests, log-uniform 512..131,072: decode, migrate 25% of requests' pages
    to a second pool (bit-exact), rerun as two calls, compare."""
    w = W.ragged_handoff()
    inp = W.make_workload_inputs(w, device=DEV)
    out, lse, _ = gpu_decode(inp, w.scale)
    assert torch.isfinite(out).all()
    B = w.batch
    lens = list(w.ctx_lens)
    longest = int(np.argmax(lens))
    shortest = int(np.argmin(lens))
    for r in (longest, shortest, 100):
        ro, rl = oracle_rows(inp, w.scale, r, 0, 4)
        assert_attn_close(out[r, :4].cpu(), ro, lse[r, :4].cpu(), rl, f"ragged r{r}")
    m = W.make_migration(inp, w.migrate_frac, seed=w.seed)
    pool2 = torch.full((m.dst_num_pages, 64, 576), float("nan"), dtype=torch.bfloat16, device=DEV)
    S.splash_kv_migrate(inp.pool, pool2, m.src_ids.to(DEV), m.dst_ids.to(DEV))
    torch.cuda.synchronize()
    src = inp.pool.index_select(0, m.src_ids.to(DEV).long())
    dst = pool2.index_select(0, m.dst_ids.to(DEV).long())
    assert torch.equal(src.view(torch.int16), dst.view(torch.int16))
    moved = torch.tensor(m.requests, device=DEV)
    keep = torch.tensor([r for r in range(B) if r not in set(m.requests)], device=DEV)
    inp2 = W.DecodeInputs(q=inp.q[moved].contiguous(), pool=pool2,
                          block_table=m.new_block_table.to(DEV),
                          ctx_lens=inp.ctx_lens[moved].contiguous(), perm=inp.perm,
                          pages_per_req=[inp.pages_per_req[r] for r in m.requests])
    inp1 = W.DecodeInputs(q=inp.q[keep].contiguous(), pool=inp.pool,
                          block_table=inp.block_table[keep].contiguous(),
                          ctx_lens=inp.ctx_lens[keep].contiguous(), perm=inp.perm,
                          pages_per_req=[inp.pages_per_req[int(r)] for r in keep])
    o2, l2, _ = gpu_decode(inp2, w.scale)
    o1, l1, _ = gpu_decode(inp1, w.scale)
    assert_attn_close(o2.cpu(), out[moved].cpu().double().numpy(), l2.cpu(),
                      lse[moved].cpu().double().numpy(), "migrated requests")
    assert_attn_close(o1.cpu(), out[keep].cpu().double().numpy(), l1.cpu(),
                      lse[keep].cpu().double().numpy(), "remaining requests")
    r0 = 0
    ro, rl = oracle_rows(inp2, w.scale, r0, 120, 128)
    assert_attn_close(o2[r0, 120:].cpu(), ro, l2[r0, 120:].cpu(), rl, "migrated vs oracle")


def test_batch_beyond_the_plans_shared_memory_search():
    """More requests (9,000) than the plan keeps tile ends for in shared memory (8,192):
    the group search then reads the plan from global memory.  Short ragged contexts,
    some empty; sampled requests against the oracle, and every output finite."""
    rng = np.random.default_rng(60)
    ctx = [int(x) for x in rng.integers(0, 400, size=9000)]
    inp = W.make_decode_inputs(ctx, 16, 64, seed=60, device=DEV)
    out, lse, ws = gpu_decode(inp, W.MLA_SCALE)
    torch.cuda.synchronize()
    assert S.splash_workspace_status(ws) == 0
    nonempty = [r for r, L in enumerate(ctx) if L > 0]
    assert torch.isfinite(out[nonempty]).all() and torch.isfinite(lse[nonempty]).all()
    empty = [r for r, L in enumerate(ctx) if L == 0]
    assert empty and (out[empty] == 0).all() and torch.isneginf(lse[empty]).all()
    for r in [nonempty[0], 4095, 8191, 8192, 8193, nonempty[-1]] + list(rng.choice(nonempty, 6)):
        r = int(r)
        ro, rl = oracle_rows(inp, W.MLA_SCALE, r, 0, 16)
        assert_attn_close(out[r].cpu(), ro, lse[r].cpu(), rl, f"request {r} of 9000")


@pytest.mark.parametrize("name", ["full_heads", "tiny"])
def test_benchmark_step_matches_oracle(name):
    """The step the benchmark times, in its own launch configuration (two share calls
    on two streams, each on half the SMs, then the merge and the handoff's page
    migration), against the unsplit fp64 oracle and bit-exact pages."""
    import os
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import bench
    w = W.ALL[name]()
    inp = W.make_workload_inputs(w, device=DEV)
    step = bench.Step(w, inp, DEV)
    assert step.call_sms == torch.cuda.get_device_properties(0).multi_processor_count // 2
    step.run()
    torch.cuda.synchronize()
    assert S.splash_workspace_status(step.ws) == 0 and S.splash_workspace_status(step.ws_b) == 0
    ro, rl = oracle_full(inp, w.scale)
    assert_attn_close(step.out.cpu(), ro, step.lse.cpu(), rl, f"{name} benchmark step")
    src = inp.pool.index_select(0, step.src_ids.long())
    dst = step.pool2.index_select(0, step.dst_ids.long())
    assert torch.equal(src.view(torch.int16), dst.view(torch.int16))
