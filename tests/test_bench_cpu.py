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


def _fake_step(w, calls, ranges=None):
    """A bench Step holding only what the call-size logic reads (no device buffers)."""
    sys.path.insert(0, ROOT)
    import bench
    st = bench.Step.__new__(bench.Step)
    st.w, st.calls, st.ranges = w, calls, ranges
    return st


def test_small_two_call_steps_get_half_the_sms():
    """A multi-call step whose calls each fit in one wave (128-token tiles x 64-head
    groups <= SMs) gives every call half the SMs; larger calls and single calls keep
    every SM."""
    sys.path.insert(0, ROOT)
    import bench
    from layout_agnostic_paged_gb300 import workloads as W
    Step = bench.Step
    fh = W.full_heads()                       # 16 x 1024 tokens, 128 heads
    shares = [(0, 128, 0, 512, "out0", None), (0, 128, 512, -1, "out1", None)]
    st = _fake_step(fh, shares)
    assert [Step.call_cta_tiles(st, c) for c in shares] == [16 * 4 * 2, 16 * 4 * 2]
    assert Step.pick_call_sms(st, 152) == 76
    assert Step.pick_call_sms(st, 100) == 0   # 128 CTA-tiles no longer fit in one wave
    one = _fake_step(fh, shares[:1])
    assert Step.pick_call_sms(one, 152) == 0
    cp = W.cp_long()                          # 8 shares of 8,192 tokens: 2,048 CTA-tiles each
    cp_calls = [(0, 128, i * 8192, (i + 1) * 8192, f"out{i}", None) for i in range(8)]
    assert Step.pick_call_sms(_fake_step(cp, cp_calls), 152) == 0
    hs = W.head_shard()                       # 16-head shards: one head group per call
    hs_calls = [(i * 16, (i + 1) * 16, 0, -1, f"out{i}", None) for i in range(8)]
    assert Step.call_cta_tiles(_fake_step(hs, hs_calls), hs_calls[0]) == 128 * 32


def test_per_request_ranges_count_their_own_tiles():
    sys.path.insert(0, ROOT)
    import bench
    import torch
    from layout_agnostic_paged_gb300 import workloads as W
    w = W.Workload("ragged shares", (300, 1000, 0), 128, 64, seed=1, token_splits=2,
                   per_request_splits=True)
    calls = [(0, 128, 0, -1, "out0", None), (0, 128, 0, -1, "out1", None)]
    rng = W.per_request_ranges(w)             # share i of request r: [L_r i / 2, L_r (i + 1) / 2)
    st = _fake_step(w, calls, rng)
    # share 0: [0,150) -> tiles 0-1, [0,500) -> tiles 0-3, empty;
    # share 1: [150,300) -> tiles 1-2, [500,1000) -> tiles 3-7, empty
    assert bench.Step.call_cta_tiles(st, calls[0]) == (2 + 4) * 2
    assert bench.Step.call_cta_tiles(st, calls[1]) == (2 + 5) * 2
    assert torch.equal(rng[0, 1], torch.tensor([150, 500, 0], dtype=torch.int32))


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
