"""Pins of the fp64 oracle against things other than itself (CPU only).

Each test checks the oracle against a closed form, a library routine
(torch scaled_dot_product_attention / logsumexp in float64), brute force, or an
invariant the pages fix: "SPLASH: Switching Parallel Layouts of Attention with
Seamless Handoff for LLM Serving", Abstract (layouts differ only in who owns the
weights and the cache) and Appendix, Table 2 (TP head shares, CP token shares
with ideal token partitioning, DP-attention / DOP whole-request ownership).
"""
import math

import numpy as np
import pytest
import torch

import oracle
from tests.oracle_cases import (D_QK, D_V, from_bf16_bits, paged, random_case, random_gqa_case,
                                to_bf16_bits)

SCALE = 1.0 / math.sqrt(192.0)


def _run(case, H=None, **kw):
    return oracle.decode_attn(case["q"], case["pool"], case["bt"], case["ctx"], kw.pop("scale", SCALE),
                              **kw)


# ---------------------------------------------------------------- closed forms

def test_single_token_returns_its_value():
    rng = np.random.default_rng(1)
    case = random_case(rng, [1], num_heads=3, page_size=16)
    out, lse = _run(case)
    v0 = case["tokens"][0][0]
    q = from_bf16_bits(case["q"])
    for h in range(3):
        assert np.array_equal(out[0, h], v0[:D_V])          # weight exp(0)/1 = 1 exactly
        s0 = SCALE * float(np.dot(q[0, h], v0))
        assert abs(lse[0, h] - s0) <= 1e-12 * max(1.0, abs(s0))


def test_zero_query_gives_mean_of_values_and_log_count():
    rng = np.random.default_rng(2)
    case = random_case(rng, [100, 37], num_heads=2, page_size=16)
    case["q"][:] = 0
    out, lse = _run(case)
    for r, L in enumerate([100, 37]):
        mean = case["tokens"][r][:, :D_V].mean(axis=0)
        for h in range(2):
            np.testing.assert_allclose(out[r, h], mean, rtol=0, atol=1e-13)
            assert abs(lse[r, h] - math.log(L)) <= 1e-13


def test_equal_scores_through_rope_dims_only():
    """q lives only in the 64 rope dims and every token shares its rope part: the
    scores are all equal, so the output is the plain mean of the 512 latent
    dims -- which also pins that values are the latent prefix of the key."""
    rng = np.random.default_rng(3)
    L = 50
    toks = rng.standard_normal((L, D_QK)).astype(np.float32)
    toks[:, D_V:] = rng.standard_normal(D_QK - D_V).astype(np.float32)  # shared rope part
    q = np.zeros((1, 1, D_QK), np.float32)
    q[0, 0, D_V:] = rng.standard_normal(D_QK - D_V)
    pool, bt, ctx = paged([toks], 16)
    qb = to_bf16_bits(q)
    out, lse = oracle.decode_attn(qb, pool, bt, ctx, SCALE)
    t = from_bf16_bits(to_bf16_bits(toks))
    s = SCALE * float(np.dot(from_bf16_bits(qb)[0, 0], t[0]))
    np.testing.assert_allclose(out[0, 0], t[:, :D_V].mean(axis=0), rtol=0, atol=1e-13)
    assert abs(lse[0, 0] - (s + math.log(L))) <= 1e-12


def test_two_tokens_sigmoid_weights():
    rng = np.random.default_rng(4)
    case = random_case(rng, [2], num_heads=4, page_size=16)
    out, lse = _run(case)
    q = from_bf16_bits(case["q"])
    k = case["tokens"][0]
    for h in range(4):
        s0 = SCALE * float(np.dot(q[0, h], k[0]))
        s1 = SCALE * float(np.dot(q[0, h], k[1]))
        w0 = 1.0 / (1.0 + math.exp(s1 - s0))
        w1 = 1.0 / (1.0 + math.exp(s0 - s1))
        np.testing.assert_allclose(out[0, h], w0 * k[0, :D_V] + w1 * k[1, :D_V], rtol=0, atol=1e-12)
        assert abs(lse[0, h] - np.logaddexp(s0, s1)) <= 1e-12


def test_dominant_token_wins():
    rng = np.random.default_rng(5)
    L = 40
    toks = rng.standard_normal((L, D_QK)).astype(np.float32) * 0.01
    q = np.zeros((1, 1, D_QK), np.float32)
    q[0, 0, :] = 1.0
    toks[17, :] = 4.0                     # s_17 = 576*4*scale ~ 166 vs |s_other| < 3
    pool, bt, ctx = paged([toks], 16)
    out, lse = oracle.decode_attn(to_bf16_bits(q), pool, bt, ctx, SCALE)
    np.testing.assert_allclose(out[0, 0], np.full(D_V, 4.0), rtol=0, atol=1e-40)
    assert abs(lse[0, 0] - SCALE * 576 * 4.0) <= 1e-10


def test_empty_token_sets():
    rng = np.random.default_rng(6)
    case = random_case(rng, [10, 30], num_heads=2, page_size=16)
    out, lse = _run(case, tok_lo=30)
    assert np.all(out[:, :, :] == 0.0)
    assert np.all(np.isneginf(lse))
    out, lse = _run(case, tok_lo=5, tok_hi=5)
    assert np.all(out == 0.0) and np.all(np.isneginf(lse))


# ------------------------------------------------------- library routine (SDPA)

@pytest.mark.parametrize("ctx,H,P", [([1, 17, 40], 5, 16), ([64, 100], 8, 16), ([130, 3], 3, 64)])
def test_matches_torch_sdpa_float64(ctx, H, P):
    rng = np.random.default_rng(sum(ctx) + H)
    case = random_case(rng, ctx, num_heads=H, page_size=P)
    out, lse = _run(case)
    q = torch.from_numpy(from_bf16_bits(case["q"]))
    for r, L in enumerate(ctx):
        K = torch.from_numpy(case["tokens"][r])               # [L][576], bf16-exact
        V = K[:, :D_V]
        qr = q[r].unsqueeze(1)                                 # [H][1][576]
        ref = torch.nn.functional.scaled_dot_product_attention(
            qr.unsqueeze(0), K.expand(H, L, D_QK).unsqueeze(0), V.expand(H, L, D_V).unsqueeze(0),
            scale=SCALE)[0, :, 0, :]
        ref_lse = torch.logsumexp(SCALE * (q[r] @ K.T), dim=-1)
        np.testing.assert_allclose(out[r], ref.numpy(), rtol=0, atol=1e-12)
        np.testing.assert_allclose(lse[r], ref_lse.numpy(), rtol=0, atol=1e-12)


# --------------------------------------- several KV heads (grouped-query attention)

@pytest.mark.parametrize("ctx,H,Hkv,P", [([1, 17, 40], 8, 2, 16), ([70, 3], 6, 3, 16),
                                        ([130], 4, 4, 64)])
def test_gqa_matches_torch_sdpa_float64(ctx, H, Hkv, P):
    """Query head h attends to KV head h / (H / Hkv): per KV head, SDPA over its
    group of query heads (the Abstract's "few or no KV heads")."""
    rng = np.random.default_rng(sum(ctx) + 10 * H + Hkv)
    case = random_gqa_case(rng, ctx, H, Hkv, P)
    out, lse = _run(case)
    q = torch.from_numpy(from_bf16_bits(case["q"]))
    g = H // Hkv
    for r, L in enumerate(ctx):
        for j in range(Hkv):
            K = torch.from_numpy(case["tokens"][r][j])
            V = K[:, :D_V]
            qg = q[r, j * g:(j + 1) * g]                            # [g][576]
            ref = torch.nn.functional.scaled_dot_product_attention(
                qg.unsqueeze(1).unsqueeze(0), K.expand(g, L, D_QK).unsqueeze(0),
                V.expand(g, L, D_V).unsqueeze(0), scale=SCALE)[0, :, 0, :]
            ref_lse = torch.logsumexp(SCALE * (qg @ K.T), dim=-1)
            np.testing.assert_allclose(out[r, j * g:(j + 1) * g], ref.numpy(), rtol=0, atol=1e-12)
            np.testing.assert_allclose(lse[r, j * g:(j + 1) * g], ref_lse.numpy(), rtol=0, atol=1e-12)


def test_gqa_with_one_kv_head_is_the_shared_head():
    rng = np.random.default_rng(11)
    case = random_case(rng, [33, 70, 5], num_heads=8, page_size=16)
    o3, l3 = _run(case)
    four = dict(case, pool=case["pool"][:, None])          # [pages][1][P][576]
    o4, l4 = _run(four)
    assert np.array_equal(o3, o4) and np.array_equal(l3, l4)


def test_gqa_rejects_heads_not_divisible_by_kv_heads():
    rng = np.random.default_rng(12)
    case = random_gqa_case(rng, [10], 6, 4, 16)
    with pytest.raises(ValueError):
        _run(case)


# ------------------------------------------ invariants of the layouts (Table 2)

def test_head_shards_concatenate_to_unsplit():
    rng = np.random.default_rng(7)
    case = random_case(rng, [33, 70, 5], num_heads=16, page_size=16)
    full_o, full_l = _run(case)
    o = np.full_like(full_o, np.nan)
    l = np.full_like(full_l, np.nan)
    for s in range(4):
        _run(case, head_lo=4 * s, head_hi=4 * s + 4, out=o, lse=l)
    assert np.array_equal(o, full_o) and np.array_equal(l, full_l)


def test_head_shard_writes_only_its_rows():
    rng = np.random.default_rng(8)
    case = random_case(rng, [20], num_heads=8, page_size=16)
    o, l = _run(case, head_lo=2, head_hi=5)
    assert np.all(np.isnan(o[0, :2])) and np.all(np.isnan(o[0, 5:]))
    assert np.all(np.isfinite(o[0, 2:5]))


@pytest.mark.parametrize("splits", [2, 8])
def test_cp_token_ranges_merge_to_unsplit(splits):
    rng = np.random.default_rng(9 + splits)
    ctx = [256, 200, 64]
    case = random_case(rng, ctx, num_heads=4, page_size=16)
    full_o, full_l = _run(case)
    span = 256 // splits
    parts_o, parts_l = [], []
    for i in range(splits):
        o, l = _run(case, tok_lo=i * span, tok_hi=(i + 1) * span)
        parts_o.append(o)
        parts_l.append(l)
    mo, ml = oracle.lse_merge(np.stack(parts_o), np.stack(parts_l))
    np.testing.assert_allclose(mo, full_o, rtol=0, atol=1e-12)
    np.testing.assert_allclose(ml, full_l, rtol=0, atol=1e-12)


def test_request_subset_equals_rows_of_full_batch():
    rng = np.random.default_rng(10)
    case = random_case(rng, [30, 90, 1, 47], num_heads=3, page_size=16)
    full_o, full_l = _run(case)
    sub = [1, 3]
    o, l = oracle.decode_attn(case["q"][sub], case["pool"], case["bt"][sub], case["ctx"][sub], SCALE)
    assert np.array_equal(o, full_o[sub]) and np.array_equal(l, full_l[sub])


def test_physical_page_permutation_is_invisible():
    rng = np.random.default_rng(11)
    ctx = [100, 64, 7]
    toks = [rng.standard_normal((L, D_QK)).astype(np.float32) for L in ctx]
    q = to_bf16_bits(rng.standard_normal((3, 4, D_QK)).astype(np.float32))
    pa, bta, c = paged(toks, 16)                                  # identity layout
    ppr = [7, 4, 1]
    perm = rng.permutation(sum(ppr) + 1)
    ids, k = [], 0
    for n in ppr:
        ids.append([int(x) for x in perm[k:k + n]])
        k += n
    pb, btb, _ = paged(toks, 16, ids)
    oa, la = oracle.decode_attn(q, pa, bta, c, SCALE)
    ob, lb = oracle.decode_attn(q, pb, btb, c, SCALE)
    assert np.array_equal(oa, ob) and np.array_equal(la, lb)


def test_identity_layout_is_a_contiguous_cache():
    """With pages packed in order the pool rows are the tokens themselves."""
    rng = np.random.default_rng(12)
    L = 45
    toks = rng.standard_normal((L, D_QK)).astype(np.float32)
    q = to_bf16_bits(rng.standard_normal((1, 2, D_QK)).astype(np.float32))
    pool, bt, ctx = paged([toks], 16, poison=True)
    out, lse = oracle.decode_attn(q, pool, bt, ctx, SCALE)
    K = torch.from_numpy(from_bf16_bits(pool).reshape(-1, D_QK)[:L])
    qq = torch.from_numpy(from_bf16_bits(q))[0]
    w = torch.softmax(SCALE * qq @ K.T, dim=-1)
    np.testing.assert_allclose(out[0], (w @ K[:, :D_V]).numpy(), rtol=0, atol=1e-12)


def test_poisoned_tails_never_reach_outputs():
    rng = np.random.default_rng(13)
    case = random_case(rng, [17, 33], num_heads=2, page_size=16)
    assert np.isnan(from_bf16_bits(case["pool"])).any()
    out, lse = _run(case)
    assert np.all(np.isfinite(out)) and np.all(np.isfinite(lse))


def test_rejects_bad_arguments_and_bad_page_ids():
    rng = np.random.default_rng(14)
    case = random_case(rng, [20], num_heads=2, page_size=16)
    with pytest.raises(ValueError):
        _run(case, head_lo=1, head_hi=1)
    with pytest.raises(ValueError):
        _run(case, tok_lo=5, tok_hi=3)
    bt = case["bt"].copy()
    bt[0, 1] = 10_000
    with pytest.raises(ValueError):
        oracle.decode_attn(case["q"], case["pool"], bt, case["ctx"], SCALE)


# --------------------------------------------------------------- LSE merge

def test_merge_single_part_is_identity():
    rng = np.random.default_rng(20)
    o = rng.standard_normal((1, 3, 5, D_V))
    l = rng.standard_normal((1, 3, 5))
    mo, ml = oracle.lse_merge(o, l)
    assert np.array_equal(mo, o[0]) and np.array_equal(ml, l[0])


def test_merge_weights_closed_form():
    o0 = np.full((1, D_V), 1.0)
    o1 = np.full((1, D_V), 5.0)
    mo, ml = oracle.lse_merge(np.stack([o0, o1]), np.array([[0.0], [math.log(3.0)]]))
    np.testing.assert_allclose(mo, np.full((1, D_V), (1.0 + 3 * 5.0) / 4.0), rtol=0, atol=1e-15)
    assert abs(ml[0] - math.log(4.0)) <= 1e-15


def test_merge_equal_parts_adds_ln2():
    rng = np.random.default_rng(21)
    o = rng.standard_normal((4, D_V))
    l = rng.standard_normal(4)
    mo, ml = oracle.lse_merge(np.stack([o, o]), np.stack([l, l]))
    np.testing.assert_allclose(mo, o, rtol=0, atol=1e-15)
    np.testing.assert_allclose(ml, l + math.log(2.0), rtol=0, atol=1e-15)


def test_merge_empty_parts():
    rng = np.random.default_rng(22)
    o = rng.standard_normal((2, D_V))
    l = np.array([0.3, -1.2])
    empty_o = np.zeros((2, D_V))
    empty_l = np.full(2, -np.inf)
    mo, ml = oracle.lse_merge(np.stack([empty_o, o, empty_o]), np.stack([empty_l, l, empty_l]))
    np.testing.assert_allclose(mo, o, rtol=0, atol=1e-15)
    np.testing.assert_allclose(ml, l, rtol=0, atol=1e-15)
    mo, ml = oracle.lse_merge(np.stack([empty_o, empty_o]), np.stack([empty_l, empty_l]))
    assert np.all(mo == 0) and np.all(np.isneginf(ml))


def test_merge_order_does_not_matter():
    rng = np.random.default_rng(23)
    o = rng.standard_normal((5, 3, D_V))
    l = rng.standard_normal((5, 3)) * 3
    a = oracle.lse_merge(o, l)
    p = rng.permutation(5)
    b = oracle.lse_merge(o[p], l[p])
    np.testing.assert_allclose(a[0], b[0], rtol=0, atol=1e-13)
    np.testing.assert_allclose(a[1], b[1], rtol=0, atol=1e-13)


# ------------------------------------------------------------ page migration

def test_migrate_copies_bytes_and_touches_nothing_else():
    rng = np.random.default_rng(30)
    src = rng.integers(0, 2**16, size=(12, 16, D_QK), dtype=np.uint16)
    dst = rng.integers(0, 2**16, size=(9, 16, D_QK), dtype=np.uint16)
    before = dst.copy()
    s_ids = np.array([3, 11, 0, 7], np.int32)
    d_ids = np.array([8, 1, 4, 2], np.int32)
    oracle.kv_migrate(src, dst, s_ids, d_ids)
    expect = before.copy()
    expect[d_ids] = src[s_ids]
    assert np.array_equal(dst, expect)


def test_migrate_rejects_out_of_range_ids():
    src = np.zeros((4, 16, D_QK), np.uint16)
    dst = np.ones((4, 16, D_QK), np.uint16)
    with pytest.raises(ValueError):
        oracle.kv_migrate(src, dst, np.array([0, 4], np.int32), np.array([0, 1], np.int32))
    assert np.all(dst == 1)


def test_migrated_pages_decode_identically():
    """A handoff moves pages and rewrites block-table rows; attention is unchanged."""
    rng = np.random.default_rng(31)
    case = random_case(rng, [50, 20], num_heads=4, page_size=16)
    o1, l1 = _run(case)
    pool2 = np.full((10, 16, D_QK), 0x7FC0, np.uint16)          # NaN-filled second pool
    src_ids = np.array(case["page_ids"][0], np.int32)
    dst_ids = np.array([9, 2, 5, 0], np.int32)
    oracle.kv_migrate(case["pool"], pool2, src_ids, dst_ids)
    bt2 = np.full((1, case["bt"].shape[1]), -1, np.int32)
    bt2[0, :4] = dst_ids
    o2, l2 = oracle.decode_attn(case["q"][:1], pool2, bt2, case["ctx"][:1], SCALE)
    assert np.array_equal(o2[0], o1[0]) and np.array_equal(l2[0], l1[0])
