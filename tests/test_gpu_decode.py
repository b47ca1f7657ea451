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


@pytest.mark.parametrize("H", [128, 16])
def test_bad_page_ids_are_flagged_and_their_tokens_left_out(H):
    """A block-table id outside the pool for a needed page is not read: the kernel flags
    it and leaves that page's tokens out of the attention.  The expectation is the
    oracle over each request's readable tokens (two token ranges merged by their
    log-sum-exp weights)."""
    import oracle
    inp = _inputs([200, 64, 1000], H, 64, seed=28)
    good = W.DecodeInputs(q=inp.q, pool=inp.pool, block_table=inp.block_table.clone(),
                          ctx_lens=inp.ctx_lens, perm=inp.perm, pages_per_req=inp.pages_per_req)
    inp.block_table[0, 1] = 10_000_000        # tokens [64, 128) of request 0
    inp.block_table[2, 7] = -5                # tokens [448, 512) of request 2
    out, lse, ws = gpu_decode(inp, W.MLA_SCALE)
    flags = S.splash_workspace_status(ws)
    assert flags & S.SPLASH_DEVICE_BAD_INPUT
    assert not flags & S.SPLASH_DEVICE_TIMEOUT
    for r, (b0, b1) in {0: (64, 128), 2: (448, 512)}.items():
        o0, l0 = oracle_rows(good, W.MLA_SCALE, r, 0, H, tok_lo=0, tok_hi=b0)
        o1, l1 = oracle_rows(good, W.MLA_SCALE, r, 0, H, tok_lo=b1, tok_hi=-1)
        mo, ml = oracle.lse_merge(np.stack([o0, o1]), np.stack([l0, l1]))
        assert_attn_close(out[r].cpu(), mo, lse[r].cpu(), ml, f"request {r} without its bad page")
    ro, rl = oracle_rows(good, W.MLA_SCALE, 1, 0, H)
    assert_attn_close(out[1].cpu(), ro, lse[1].cpu(), rl, "request 1 (all pages readable)")


def test_workspace_too_small_is_rejected():
    inp = _inputs([64], 8, 16, seed=29)
    ws = S.decode_workspace(inp.q, inp.pool, inp.block_table, W.MLA_SCALE)
    with pytest.raises(S.SplashError):
        gpu_decode(inp, W.MLA_SCALE, ws=ws[:ws.numel() - 256])


# ---------------------------------------------------------------- large batches

def test_batch_beyond_the_plans_shared_memory_search():
    """More requests (9,000) than the plan keeps tile ends for in shared memory (8,192):
    the group search then reads the plan from global memory.  Short ragged contexts,
    some empty; every request against the oracle."""
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
    ro, rl = oracle_full(inp, W.MLA_SCALE)
    assert_attn_close(out.cpu(), ro, lse.cpu(), rl, "9000 requests")
