"""GPU parity of grouped-query decode over several KV heads (the Abstract of
"SPLASH: Switching Parallel Layouts of Attention with Seamless Handoff for LLM
Serving": layouts for models with few or no KV heads) against the fp64 oracle
(marked gpu).  The pool is [num_pages][Hkv][P][576]; query head h reads KV head
h / (H / Hkv).  Head shards are aligned to KV-head groups (Appendix, Table 2's TP
and DOP shares)."""
import pytest
import torch

from layout_agnostic_paged_gb300 import splash as S
from layout_agnostic_paged_gb300 import workloads as W
from tests.gpu_helpers import assert_attn_close, oracle_full

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _decode(inp, head_lo=0, head_hi=None, tok_lo=0, tok_hi=-1, out=None, lse=None):
    B, H, _ = inp.q.shape
    head_hi = H if head_hi is None else head_hi
    out = torch.full((B, H, 512), float("nan"), device=DEV) if out is None else out
    lse = torch.full((B, H), float("nan"), device=DEV) if lse is None else lse
    ws = S.decode_workspace(inp.q, inp.pool, inp.block_table, W.MLA_SCALE, head_lo, head_hi)
    S.splash_decode_attn_ex(inp.q, inp.pool, inp.block_table, inp.ctx_lens, head_lo, head_hi,
                            tok_lo, tok_hi, out, lse, ws, W.MLA_SCALE)
    assert S.splash_workspace_status(ws) == 0
    return out, lse


@pytest.mark.parametrize("ctx,H,Hkv,P", [
    ([300, 1024, 77, 2000], 128, 8, 64),     # 16 query heads per KV head
    ([129, 513], 64, 2, 64),                 # 32 per KV head
    ([1, 100, 257], 16, 4, 16),              # 4 per KV head
    ([700, 64], 256, 2, 64),                 # 128 per KV head: two head groups each
    ([333], 24, 2, 16),                      # 12 per KV head (padded to 16)
])
def test_gqa_matches_oracle(ctx, H, Hkv, P):
    inp = W.make_decode_inputs(ctx, H, P, seed=70 + H + Hkv, device=DEV, num_kv_heads=Hkv)
    assert inp.pool.shape[1:] == (Hkv, P, 576)
    out, lse = _decode(inp)
    ro, rl = oracle_full(inp, W.MLA_SCALE)
    assert_attn_close(out.cpu(), ro, lse.cpu(), rl, f"H={H} Hkv={Hkv} P={P}")


def test_gqa_head_shards_aligned_to_kv_groups_concatenate():
    inp = W.make_decode_inputs([900, 2048, 15], 128, 64, seed=80, device=DEV, num_kv_heads=8)
    out = torch.full((3, 128, 512), float("nan"), device=DEV)
    lse = torch.full((3, 128), float("nan"), device=DEV)
    for i in range(4):   # 4 shards of 32 heads = 2 KV heads each
        _decode(inp, 32 * i, 32 * (i + 1), out=out, lse=lse)
    ro, rl = oracle_full(inp, W.MLA_SCALE)
    assert_attn_close(out.cpu(), ro, lse.cpu(), rl, "KV-aligned head shards")


def test_gqa_cp_shares_merge_to_unsplit():
    inp = W.make_decode_inputs([4096, 1500, 100], 64, 64, seed=81, device=DEV, num_kv_heads=4)
    po = torch.empty(3, 3, 64, 512, device=DEV)
    pl = torch.empty(3, 3, 64, device=DEV)
    for i in range(3):
        _decode(inp, tok_lo=1400 * i, tok_hi=1400 * (i + 1) if i < 2 else -1, out=po[i], lse=pl[i])
    mo = torch.empty(3, 64, 512, device=DEV)
    ml = torch.empty(3, 64, device=DEV)
    S.splash_lse_merge(po, pl, mo, ml)
    ro, rl = oracle_full(inp, W.MLA_SCALE)
    assert_attn_close(mo.cpu(), ro, ml.cpu(), rl, "GQA CP merged")


def test_gqa_rejects_misaligned_head_slices_and_the_plain_entry_point():
    inp = W.make_decode_inputs([64], 16, 16, seed=82, device=DEV, num_kv_heads=4)
    with pytest.raises(S.SplashError):
        _decode(inp, head_lo=2, head_hi=8)      # groups of 4 heads: 2 is inside one
    ws = S.decode_workspace(inp.q, inp.pool, inp.block_table, W.MLA_SCALE)
    out = torch.empty(1, 16, 512, device=DEV)
    lse = torch.empty(1, 16, device=DEV)
    with pytest.raises(ValueError):
        S.splash_decode_attn(inp.q, inp.pool, inp.block_table, inp.ctx_lens, 0, 16, 0, -1, out,
                             lse, ws, W.MLA_SCALE)


def test_gqa_pages_migrate_bit_exactly():
    inp = W.make_decode_inputs([300, 70], 32, 64, seed=83, device=DEV, num_kv_heads=2)
    dst = torch.zeros_like(inp.pool)
    src_ids = inp.block_table[0, :5].contiguous()
    dst_ids = torch.tensor([4, 0, 3, 1, 2], dtype=torch.int32, device=DEV)
    S.splash_kv_migrate(inp.pool, dst, src_ids, dst_ids)
    torch.cuda.synchronize()
    for s_, d_ in zip(src_ids.tolist(), dst_ids.tolist()):
        a = inp.pool[s_].view(torch.int16)
        b = dst[d_].view(torch.int16)
        assert torch.equal(a, b)
