"""bench.py's reference arm (the fp64 oracle on the host) runs on CPU and prints
one JSON line with the contract's keys."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_prints_contract_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--workload", "tiny", "--steps", "2", "--warmup", "1"],
                       capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
              "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
              "cpu_baseline", "e2e", "impl"):
        assert k in d, k
    assert d["impl"] == "reference" and d["value"] > 0
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["cpu_baseline"]["kind"] == "oracle"


def test_bench_module_imports_without_gpu():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.UNIT == "KV-tokens/s"
    assert len(bench.kernel_source_hash()) == 16


def test_kernel_source_hash_ignores_comments_but_not_code(tmp_path, monkeypatch):
    """The stored ncu counters follow the code: comments and whitespace do not change the
    hash, a changed token does."""
    bench = _bench()
    src = os.path.join(ROOT, "layout_agnostic_paged_gb300", "csrc")
    dst = tmp_path / "layout_agnostic_paged_gb300" / "csrc"
    dst.mkdir(parents=True)
    for name in ("decode_tc.cu", "common.cuh", "plan.cuh"):
        (dst / name).write_text(open(os.path.join(src, name)).read())
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    h0 = bench.kernel_source_hash()
    f = dst / "decode_tc.cu"
    text = f.read_text()
    f.write_text(text.replace("namespace splash {", "// a note\nnamespace   splash /* x */ {", 1))
    assert bench.kernel_source_hash() == h0
    f.write_text(text.replace("kTau = 8.0f", "kTau = 9.0f", 1))
    assert bench.kernel_source_hash() != h0


def _bench():
    sys.path.insert(0, ROOT)
    import bench
    return bench


def test_step_patterns_follow_each_configuration():
    """Each workload's step is the calls its configuration defines: ragged + handoff =
    whole-batch decode, migration, decode rerun as two request-subset calls on the two
    pools; CP = token-share calls then the merge; head shards = one call per shard;
    full heads and tiny = one call."""
    bench = _bench()
    from layout_agnostic_paged_gb300 import workloads as W
    w = W.ragged_handoff()
    moved = [3, 7, 100]
    ph = bench.step_pattern(w, moved)
    assert [p[0] for p in ph] == ["decode", "migrate", "decode"]
    (pre,), post = ph[0][1], ph[2][1]
    assert pre.rows is None and pre.out == "pre" and (pre.head_lo, pre.head_hi) == (0, 128)
    assert [c.pool for c in post] == ["pool1", "pool2"]
    assert post[1].rows == (3, 7, 100) and len(post[0].rows) == w.batch - 3
    assert set(post[0].rows) | set(post[1].rows) == set(range(w.batch))
    # the step decodes the batch twice, for every head
    assert bench.decoded_tokens(w, ph) == 2 * w.kv_tokens
    cp = bench.step_pattern(W.cp_long())
    assert [p[0] for p in cp] == ["decode", "merge"] and cp[1][1] == 8
    assert [(c.tok_lo, c.tok_hi) for c in cp[0][1]][:2] == [(0, 8192), (8192, 16384)]
    assert cp[0][1][-1].tok_hi == -1
    assert bench.decoded_tokens(W.cp_long(), cp) == W.cp_long().kv_tokens
    hs = bench.step_pattern(W.head_shard())
    assert [(c.head_lo, c.head_hi) for c in hs[0][1]] == [(16 * i, 16 * i + 16) for i in range(8)]
    assert bench.decoded_tokens(W.head_shard(), hs) == W.head_shard().kv_tokens
    for name in ("full_heads", "tiny"):
        p = bench.step_pattern(W.ALL[name]())
        assert len(p) == 1 and len(p[0][1]) == 1 and p[0][1][0].rows is None


def test_small_two_call_phases_get_half_the_sms():
    """A phase of several calls whose calls each fit in one wave (128-token tiles x
    64-head groups <= SMs) gives every call half the SMs; larger calls and single calls
    keep every SM."""
    bench = _bench()
    from layout_agnostic_paged_gb300 import workloads as W
    C = bench.CallSpec
    fh = W.full_heads()                       # 16 x 1024 tokens, 128 heads
    halves = [C(0, 128, rows=list(range(8))), C(0, 128, rows=list(range(8, 16)))]
    assert not bench.token_share_phase(halves)         # request subsets, not token shares
    assert [bench.call_cta_tiles(fh, c) for c in halves] == [8 * 8 * 2, 8 * 8 * 2]
    assert bench.pick_call_sms(fh, halves, 152) == 76
    assert bench.pick_call_sms(fh, halves, 100) == 0   # 128 CTA-tiles no longer fit in one wave
    assert bench.pick_call_sms(fh, halves[:1], 152) == 0
    hs = W.head_shard()                       # 16-head shards: one head group per call
    assert bench.call_cta_tiles(hs, C(0, 16)) == 128 * 32
    hs_calls = bench.step_pattern(hs)[0][1]
    assert not bench.token_share_phase(hs_calls)       # same tokens, other heads
    assert bench.pick_lanes(hs_calls) == 2 and bench.pick_call_sms(hs, hs_calls, 152) == 0
    rh = W.ragged_handoff()
    post = bench.step_pattern(rh, list(range(64)))[2][1]
    assert not bench.token_share_phase(post)           # other requests
    assert bench.pick_call_sms(rh, post, 152) == 0     # the rerun calls are large


def test_cp_token_shares_run_at_once_on_an_even_sm_split():
    """The 8 token shares of a CP group read disjoint KV: they run as the group's ranks
    would, all at once, each on its own stream with a quarter of the SMs (four run, the
    rest start as SMs free up).  The scalar
    shares of the long-context batch (the last one open-ended) and the per-request shares
    of the ragged batch both qualify; overlapping or repeated shares do not."""
    bench = _bench()
    from layout_agnostic_paged_gb300 import workloads as W
    C = bench.CallSpec
    cp = W.cp_long()
    cp_calls = bench.step_pattern(cp)[0][1]
    assert cp_calls[-1].tok_hi < 0 and bench.token_share_phase(cp_calls)
    assert bench.pick_lanes(cp_calls) == 8 and bench.pick_call_sms(cp, cp_calls, 152) == 38
    rc = W.ragged_cp()
    rc_calls = bench.step_pattern(rc)[0][1]
    assert bench.token_share_phase(rc_calls) and bench.pick_lanes(rc_calls) == 8
    assert not bench.token_share_phase([C(0, 128, 0, 100), C(0, 128, 50, 200), C(0, 128, 200, -1)])
    assert not bench.token_share_phase([C(0, 128, share=0), C(0, 128, share=0), C(0, 128, share=1)])
    assert not bench.token_share_phase([C(0, 64, 0, 100), C(64, 128, 100, 200), C(0, 128, 200, -1)])
    assert bench.token_share_phase([C(0, 128, 0, 100), C(0, 128, 100, 200), C(0, 128, 200, -1)])
    gq = W.gqa()                              # two token shares: half the SMs each
    gq_calls = bench.step_pattern(gq)[0][1]
    assert bench.token_share_phase(gq_calls) and bench.pick_lanes(gq_calls) == 2
    assert bench.pick_call_sms(gq, gq_calls, 152) == 76
    assert not bench.token_share_phase(gq_calls[:1])


def test_per_request_ranges_count_their_own_tiles():
    bench = _bench()
    import torch
    from layout_agnostic_paged_gb300 import workloads as W
    w = W.Workload("ragged shares", (300, 1000, 0), 128, 64, seed=1, token_splits=2,
                   per_request_splits=True)
    calls = bench.step_pattern(w)[0][1]
    rng = W.per_request_ranges(w)             # share i of request r: [L_r i / 2, L_r (i + 1) / 2)
    # share 0: [0,150) -> tiles 0-1, [0,500) -> tiles 0-3, empty;
    # share 1: [150,300) -> tiles 1-2, [500,1000) -> tiles 3-7, empty
    assert bench.call_cta_tiles(w, calls[0], rng.tolist()) == (2 + 4) * 2
    assert bench.call_cta_tiles(w, calls[1], rng.tolist()) == (2 + 5) * 2
    assert torch.equal(rng[0, 1], torch.tensor([150, 500, 0], dtype=torch.int32))
    # the two shares' tokens add up to the batch's
    assert sum(bench.call_tokens_pages(w, c, rng.tolist())[0] for c in calls) == 1300


def test_reference_step_restricted_to_a_sample_matches_the_oracle_per_phase():
    """The reference arm's step: the workload's phases run by the oracle over a sample of
    the requests.  On a small ragged handoff batch the rerun output (pool 1 for the
    remaining requests, pool 2 for the moved ones, after the oracle's page copy) equals
    the oracle on the original pool."""
    bench = _bench()
    import numpy as np
    import oracle
    from layout_agnostic_paged_gb300 import workloads as W
    w = W.Workload("small handoff", (300, 77, 1000, 129), 8, 16, seed=5, migrate_frac=0.5)
    inp = W.make_workload_inputs(w)
    mig = W.make_migration(inp, w.migrate_frac, seed=w.seed)
    ph = bench.step_pattern(w, mig.requests)
    q, pool = oracle.bf16_bits(inp.q), oracle.bf16_bits(inp.pool).copy()
    bt, ctx = inp.block_table.numpy(), inp.ctx_lens.numpy()
    pool2 = np.zeros((mig.dst_num_pages,) + pool.shape[1:], dtype=np.uint16)
    bt2 = np.full(bt.shape, -1, dtype=np.int32)
    bt2[mig.requests] = mig.new_block_table.numpy()
    out, lse = bench.reference_step(w, ph, q, pool, bt, ctx, np.arange(4), mig, pool2, bt2, None)
    ro, rl = oracle.decode_attn(q, pool, bt, ctx, w.scale)
    assert np.allclose(out, ro, rtol=0, atol=1e-12) and np.allclose(lse, rl, rtol=0, atol=1e-12)


def _free_port():
    import socket
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _reduce_worker(rank, world, port, results):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        sys.path.insert(0, ROOT)
        import bench
        bench.barrier(world)
        results[rank] = (bench.max_over_ranks(rank + 1.5, world, "cpu"),
                         bench.sum_over_ranks(rank + 1.5, world, "cpu"))
    finally:
        dist.destroy_process_group()


def test_timing_reductions_over_two_gloo_ranks():
    """The benchmark's cross-rank reductions (max of the times, sum of the tokens) and
    barrier, on two CPU ranks over gloo."""
    import torch.multiprocessing as mp
    world = 2
    with mp.Manager() as m:
        results = m.dict()
        mp.spawn(_reduce_worker, args=(world, _free_port(), results), nprocs=world, join=True)
        got = dict(results)
    assert got == {0: (2.5, 4.0), 1: (2.5, 4.0)}


def test_reference_arm_prints_once_under_two_ranks():
    """Launched as two ranks, the reference arm runs on rank 0 only: one JSON line, and
    every rank exits 0."""
    r = subprocess.run([sys.executable, "-m", "torch.distributed.run", "--nnodes", "1",
                        "--nproc-per-node", "2", "--master-addr", "127.0.0.1", "--master-port",
                        str(_free_port()), os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--workload", "tiny", "--steps", "1", "--warmup", "1"],
                       capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
