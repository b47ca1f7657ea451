"""GPU parity of the LSE merge and of KV-page migration (marked gpu)."""
import numpy as np
import pytest
import torch

import oracle
from layout_agnostic_paged_gb300 import splash as S

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.mark.parametrize("S_,B,H,d_v", [(1, 3, 5, 512), (8, 16, 128, 512), (3, 7, 9, 4), (5, 2, 3, 96)])
def test_lse_merge_matches_oracle(S_, B, H, d_v):
    g = torch.Generator(device=DEV).manual_seed(S_ * 100 + B)
    po = torch.randn(S_, B, H, d_v, generator=g, device=DEV)
    pl = torch.randn(S_, B, H, generator=g, device=DEV) * 4
    if S_ > 1:
        pl[0, 0, :] = float("-inf")              # one empty part
        po[0, 0, :] = 0
        pl[:, -1, -1] = float("-inf")            # a row with every part empty
        po[:, -1, -1] = 0
    out = torch.full((B, H, d_v), float("nan"), device=DEV)
    lse = torch.full((B, H), float("nan"), device=DEV)
    S.splash_lse_merge(po, pl, out, lse)
    ro, rl = oracle.lse_merge(po.cpu().double().numpy(), pl.cpu().double().numpy())
    np.testing.assert_allclose(out.cpu().double().numpy(), ro, rtol=0, atol=2e-6)
    fin = np.isfinite(rl)
    np.testing.assert_allclose(lse.cpu().double().numpy()[fin], rl[fin], rtol=0, atol=2e-6)
    assert np.array_equal(np.isneginf(lse.cpu().numpy()), np.isneginf(rl))


def _pools(n_src, n_dst, P=64, seed=0):
    g = torch.Generator(device=DEV).manual_seed(seed)
    src = torch.randint(-32768, 32767, (n_src, P, 576), generator=g, device=DEV,
                        dtype=torch.int16).view(torch.bfloat16)
    dst = torch.randint(-32768, 32767, (n_dst, P, 576), generator=g, device=DEV,
                        dtype=torch.int16).view(torch.bfloat16)
    return src, dst


def test_migrate_is_bit_exact_and_touches_only_targets():
    src, dst = _pools(300, 200, seed=1)
    rng = np.random.default_rng(1)
    s_ids = rng.choice(300, 120, replace=False).astype(np.int32)
    d_ids = rng.choice(200, 120, replace=False).astype(np.int32)
    before = dst.view(torch.int16).cpu().numpy().copy()
    S.splash_kv_migrate(src, dst, torch.from_numpy(s_ids).to(DEV), torch.from_numpy(d_ids).to(DEV))
    expect = oracle.kv_migrate(src.view(torch.int16).cpu().numpy().view(np.uint16),
                               before.view(np.uint16).copy(), s_ids, d_ids)
    assert np.array_equal(dst.view(torch.int16).cpu().numpy().view(np.uint16), expect)


@pytest.mark.parametrize("P", [16, 128])
def test_migrate_other_page_sizes(P):
    src, dst = _pools(40, 40, P=P, seed=P)
    s_ids = torch.arange(0, 40, 2, dtype=torch.int32, device=DEV)
    d_ids = torch.arange(39, 0, -2, dtype=torch.int32, device=DEV)
    before = dst.clone()
    S.splash_kv_migrate(src, dst, s_ids, d_ids)
    expect = before.clone()
    expect[d_ids.long()] = src[s_ids.long()]
    assert torch.equal(dst.view(torch.int16), expect.view(torch.int16))


def test_migrate_within_one_pool_disjoint_sets():
    pool, _ = _pools(64, 1, seed=3)
    before = pool.clone()
    s_ids = torch.arange(0, 16, dtype=torch.int32, device=DEV)
    d_ids = torch.arange(40, 56, dtype=torch.int32, device=DEV)
    S.splash_kv_migrate(pool, pool, s_ids, d_ids)
    expect = before.clone()
    expect[40:56] = before[0:16]
    assert torch.equal(pool.view(torch.int16), expect.view(torch.int16))


def test_migrate_skips_out_of_range_pairs():
    src, dst = _pools(10, 10, seed=4)
    before = dst.clone()
    s_ids = torch.tensor([0, 99, 2, -1], dtype=torch.int32, device=DEV)
    d_ids = torch.tensor([5, 1, 77, 3], dtype=torch.int32, device=DEV)
    S.splash_kv_migrate(src, dst, s_ids, d_ids)
    expect = before.clone()
    expect[5] = src[0]
    assert torch.equal(dst.view(torch.int16), expect.view(torch.int16))
