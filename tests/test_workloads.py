"""Seeded input generators: determinism, layout and poison (CPU only)."""
import numpy as np
import torch

import oracle
from layout_agnostic_paged_gb300 import workloads as W


def test_generator_is_deterministic_and_shuffled():
    a = W.make_decode_inputs([64, 100], 8, 16, seed=5)
    b = W.make_decode_inputs([64, 100], 8, 16, seed=5)
    assert torch.equal(a.q.view(torch.int16), b.q.view(torch.int16))
    assert torch.equal(a.pool.view(torch.int16), b.pool.view(torch.int16))
    assert torch.equal(a.block_table, b.block_table)
    used = sum(a.pages_per_req)
    assert a.num_pages == used + int(np.ceil(0.10 * used))
    ids = a.block_table[a.block_table >= 0]
    assert ids.unique().numel() == used                  # distinct physical ids
    assert not torch.equal(ids.sort().values, ids)       # not in storage order


def test_poison_sits_exactly_in_tails_and_spares():
    inp = W.make_decode_inputs([64, 100], 8, 16, seed=6)
    nan_rows = torch.isnan(inp.pool.float()).all(dim=-1)
    bt = inp.block_table
    # request 1: 100 tokens -> 7 pages, last page holds 4 tokens
    last = int(bt[1, 6])
    assert not nan_rows[last, :4].any() and nan_rows[last, 4:].all()
    used = set(int(x) for x in bt[bt >= 0])
    spare = [p for p in range(inp.num_pages) if p not in used]
    assert spare and all(nan_rows[p].all() for p in spare)


def test_page_placement_does_not_change_logical_content():
    a = W.make_decode_inputs([50, 33], 4, 16, seed=7, perm_seed=1)
    b = W.make_decode_inputs([50, 33], 4, 16, seed=7, perm_seed=2)
    assert not torch.equal(a.block_table, b.block_table)
    for r, L in enumerate([50, 33]):
        for t in range(L):
            pa = int(a.block_table[r, t // 16])
            pb = int(b.block_table[r, t // 16])
            assert torch.equal(a.pool[pa, t % 16].view(torch.int16), b.pool[pb, t % 16].view(torch.int16))


def test_oracle_runs_on_tiny_workload_and_is_finite():
    w = W.tiny()
    inp = W.make_workload_inputs(w)
    out, lse = oracle.decode_attn(oracle.bf16_bits(inp.q), oracle.bf16_bits(inp.pool),
                                  inp.block_table.numpy(), inp.ctx_lens.numpy(), w.scale)
    assert out.shape == (2, 8, 512) and np.isfinite(out).all() and np.isfinite(lse).all()


def test_ragged_lengths_are_log_uniform_and_seeded():
    a = W.ragged_ctx_lens(256, 512, 131072, seed=1004)
    assert a == W.ragged_ctx_lens(256, 512, 131072, seed=1004)
    x = np.array(a)
    assert x.min() >= 512 and x.max() <= 131072
    # log-uniform: the median of log-length sits near the middle of [ln 512, ln 131072]
    mid = 0.5 * (np.log(512) + np.log(131072))
    assert abs(np.median(np.log(x)) - mid) < 0.6


def test_migration_plan_is_distinct_and_complete():
    inp = W.make_decode_inputs([40, 70, 16, 90], 2, 16, seed=8)
    m = W.make_migration(inp, 0.5, seed=8)
    assert len(m.requests) == 2
    assert m.src_ids.numel() == sum(inp.pages_per_req[r] for r in m.requests)
    assert m.dst_ids.unique().numel() == m.dst_ids.numel()
    assert int(m.dst_ids.max()) < m.dst_num_pages
