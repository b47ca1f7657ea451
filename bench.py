#!/usr/bin/env python3
"""Benchmark of the paged MLA decode hot path on GB300: KV-tokens/s, with the
decode kernel's roofline fraction and the fp64 CPU oracle as a baseline.

One step = one pass of every hot-path row over one synthetic batch (by default
the full-heads workload: B=16, ctx 1,024, 128 query heads, one shared 576-wide
latent KV head, page 64, shuffled page ids):
  * CP layout: two token-share decode calls ([0, L/2) and [L/2, L)), each = split
    plan + tensor-core decode + split combine, producing partial out + LSE; the
    calls are independent and alternate between two streams, one workspace each,
    and calls that fit in one wave of the GPU are held to half the SMs each so that
    the two run side by side (--call-sms);
  * splash_lse_merge of the two shares into the final out / LSE;
  * a layout handoff: splash_kv_migrate of 25% of the requests' pages into a
    second block pool (the migrated requests' block-table rows are prepared once;
    switching tables is a pointer swap, not a kernel).
value = KV tokens of the batch / step time (each KV token is read once per step).

Timing: W untimed warm-up steps, then K timed steps; before every step a 512 MB
buffer is written to flush the 129 MB L2 (outside the timed events); each step
is one CUDA graph replay bracketed by CUDA events on the launching stream and the
K step times are summed; ranks meet at a barrier (+ synchronize) before and after
and the max over ranks is reported.  A second pass of instrumented graphs gives
the per-row breakdown, and a third the decode calls with a background page
migration.  `--impl reference` times the fp64 C oracle instead.
"""
from __future__ import annotations

import argparse
import hashlib
import io
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "paged decode attn KV-tokens/s; achieved TB/s & TFLOP/s as % of roofline"
UNIT = "KV-tokens/s"
L2_FLUSH_BYTES = 512 << 20


def parse_args():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="full_heads",
                    help="tiny | full_heads | cp_long | head_shard | ragged_handoff")
    ap.add_argument("--reserved-sms", type=int, default=16,
                    help="SMs left to the background page migration in the handoff-overlap "
                         "measurement")
    ap.add_argument("--call-sms", type=int, default=-1,
                    help="SM budget of each decode call of a multi-call step (-1: half the "
                         "SMs when every call fits in one wave, else all; 0: all)")
    ap.add_argument("--cpu-seconds", type=float, default=12.0,
                    help="target CPU time of the oracle baseline sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-clocks", action="store_true")
    return ap.parse_args()


# ----------------------------------------------------------------------------- helpers

def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), "measured"
    return 6800.0, 1900.0, "fallback"


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    for name in ("decode_tc.cu", "common.cuh"):
        with open(os.path.join(ROOT, "layout_agnostic_paged_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def ncu_traffic(workload: str):
    """DRAM bytes per decode launch from the committed ncu summary, if it was taken
    on the current kernel source (else None)."""
    p = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    e = d.get(workload)
    if not e or e.get("kernel_source_hash") != kernel_source_hash():
        return None
    return float(e["dram_bytes_per_launch"])


class ClockSampler:
    """SM clock and clock-event reasons sampled every millisecond during the timed
    region, through NVML (libnvidia-ml via ctypes), in a background thread."""
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, cuda_index: int, enabled: bool = True):
        self.enabled = enabled
        self.samples = []
        self.error = None
        self.max_mhz = None
        self._stop = None
        self._thread = None
        if not enabled:
            return
        try:
            import ctypes
            self.nvml = ctypes.CDLL("libnvidia-ml.so.1")
            if self.nvml.nvmlInit_v2() != 0:
                raise OSError("nvmlInit failed")
            self.h = ctypes.c_void_p()
            bus = self._pci_bus_id(cuda_index)
            if bus and self.nvml.nvmlDeviceGetHandleByPciBusId_v2(bus.encode(), ctypes.byref(self.h)) == 0:
                pass
            elif self.nvml.nvmlDeviceGetHandleByIndex_v2(cuda_index, ctypes.byref(self.h)) != 0:
                raise OSError("no NVML handle")
            mx = ctypes.c_uint()
            if self.nvml.nvmlDeviceGetMaxClockInfo(self.h, 1, ctypes.byref(mx)) == 0:
                self.max_mhz = mx.value
            self._fn_reasons = getattr(self.nvml, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
                self.nvml.nvmlDeviceGetCurrentClocksThrottleReasons
        except Exception as e:  # noqa: BLE001 - reported in the JSON line
            self.error = f"nvml unavailable: {e}"
            self.enabled = False

    @staticmethod
    def _pci_bus_id(i):
        try:
            import torch
            p = torch.cuda.get_device_properties(i)
            return f"{p.pci_domain_id:08x}:{p.pci_bus_id:02x}:{p.pci_device_id:02x}.0"
        except Exception:  # noqa: BLE001
            return None

    def sample(self):
        import ctypes
        c = ctypes.c_uint()
        r = ctypes.c_ulonglong()
        if self.nvml.nvmlDeviceGetClockInfo(self.h, 1, ctypes.byref(c)) == 0 and \
                self._fn_reasons(self.h, ctypes.byref(r)) == 0:
            self.samples.append((c.value, r.value))

    def _run(self):
        while not self._stop.is_set():
            self.sample()
            self._stop.wait(0.001)

    def __enter__(self):
        if self.enabled:
            import threading
            self._stop = threading.Event()
            self.sample()
            self._thread = threading.Thread(target=self._run, daemon=True)
            self._thread.start()
        return self

    def __exit__(self, *exc):
        if self.enabled:
            self.sample()
            self._stop.set()
            self._thread.join()

    def summary(self):
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": self.max_mhz, "reasons": [],
                    "samples": 0, "note": self.error or "no samples"}
        mhz = [c for c, _ in self.samples]
        bits = 0
        for _, r in self.samples:
            bits |= r
        return {"sm_mhz": statistics.median(mhz), "sm_max_mhz": self.max_mhz,
                "reasons": sorted(n for b, n in self.REASONS.items() if bits & b),
                "samples": len(self.samples), "source": "nvml"}


def dist_setup(args):
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int, device) -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(x: float, world: int, device) -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


# ----------------------------------------------------------------------------- the step

class Step:
    """Buffers and calls of one step over one batch (see the module docstring).

    The step pattern follows the workload's layout:
      * CP (tiny, full_heads, cp_long): max(2, token_splits) token-share calls, then
        splash_lse_merge of the shares;
      * TP / DOP head shards (head_shard): one call per head shard, rows concatenate;
      * DP-attention / DOP whole requests (ragged_handoff): one call over the batch.
    Every pattern ends with the handoff: splash_kv_migrate of migrate_frac (default
    25%) of the requests' pages into a second pool.
    """

    def __init__(self, w, inp, device, ranges=None, call_sms=-1):
        import torch
        from layout_agnostic_paged_gb300 import splash as S
        from layout_agnostic_paged_gb300 import workloads as W
        self.S = S
        self.w = w
        self.inp = inp
        B, H = w.batch, w.num_heads
        self.B, self.H = B, H
        # out and lse share one buffer so that the end-to-end leg reads them back at once
        self.out_pack, (self.out, self.lse) = pack(
            [torch.empty(B, H, 512), torch.empty(B, H)], device)
        self.calls = []          # (head_lo, head_hi, tok_lo, tok_hi, out, lse)
        self.merge = False
        if w.head_shards > 1:
            hs = H // w.head_shards
            for i in range(w.head_shards):
                self.calls.append((i * hs, (i + 1) * hs, 0, -1, self.out, self.lse))
            self.pattern = f"{w.head_shards} head-shard calls of {hs} heads"
        elif w.migrate_frac > 0 and w.token_splits == 1:
            self.calls.append((0, H, 0, -1, self.out, self.lse))
            self.pattern = "one whole-request call over the batch"
        else:
            n = max(2, w.token_splits)
            L = max(w.ctx_lens)
            span = -(-L // n)
            self.po = torch.empty(n, B, H, 512, device=device)
            self.pl = torch.empty(n, B, H, device=device)
            for i in range(n):
                self.calls.append((0, H, i * span, (i + 1) * span if i + 1 < n else -1,
                                   self.po[i], self.pl[i]))
            self.merge = True
            self.pattern = f"{n} CP token-share calls + LSE merge"
            if w.per_request_splits:
                # share i of request r: [L_r i / n, L_r (i + 1) / n), per-request ranges
                self.ranges = ranges if ranges is not None else W.per_request_ranges(w).to(device)
                self.pattern = (f"{n} CP calls with per-request token shares "
                                f"(splash_decode_attn_ex) + LSE merge")
        hs0 = self.calls[0][1] - self.calls[0][0]
        self.ws = S.decode_workspace(inp.q, inp.pool, inp.block_table, w.scale, 0, hs0)
        # the step's decode calls are independent: odd calls go to a second stream with a
        # workspace of their own, so one call's tail overlaps the next call's start
        self.ws_b = (S.decode_workspace(inp.q, inp.pool, inp.block_table, w.scale, 0, hs0)
                     if len(self.calls) > 1 else None)
        self.stream_b = torch.cuda.Stream(device)
        frac = w.migrate_frac if w.migrate_frac > 0 else 0.25
        self.mig = W.make_migration(inp, frac, seed=w.seed)
        self.pool2 = torch.empty((self.mig.dst_num_pages,) + tuple(inp.pool.shape[1:]),
                                 dtype=inp.pool.dtype, device=device)
        self.src_ids = self.mig.src_ids.to(device)
        self.dst_ids = self.mig.dst_ids.to(device)
        self.page_bytes = int(inp.pool[0].numel() * inp.pool.element_size())
        self.pattern += f" + {int(round(100 * frac))}% KV-page handoff ({self.src_ids.numel()} pages)"
        if len(self.calls) > 1:
            self.pattern += "; decode calls alternate between two streams, one workspace each"
            if self.migrate_bytes() <= (64 << 20):
                self.pattern += "; the (small) migration runs on the second stream alongside the merge"
        self.launches_per_step = 3 * len(self.calls) + (1 if self.merge else 0) + 1
        if not hasattr(self, "ranges"):
            self.ranges = None
        sms = torch.cuda.get_device_properties(device).multi_processor_count
        self.call_sms = self.pick_call_sms(sms) if call_sms < 0 else call_sms
        if self.call_sms:
            self.pattern += (f"; each call limited to {self.call_sms} of {sms} SMs, so the two "
                             f"streams' calls run side by side")

    def call_cta_tiles(self, c):
        """(128-token tiles x 64-head groups) one decode call must process."""
        hl, hh, lo, hi, _, _ = c
        i = next(k for k, x in enumerate(self.calls) if x is c)
        rng = self.ranges[i].cpu().tolist() if self.ranges is not None else None
        tiles = 0
        for r, L in enumerate(self.w.ctx_lens):
            if rng is not None:
                lo, hi = rng[0][r], rng[1][r]
            a, b = max(lo, 0), (L if hi < 0 else min(hi, L))
            if b > a:
                tiles += (b - 1) // 128 - a // 128 + 1
        return tiles * -(-(hh - hl) // 64)

    def pick_call_sms(self, sms):
        """A call whose tiles fill at most one wave of the GPU leaves SMs idle while the
        other stream's call waits for them; two such calls each get half the SMs and run
        side by side (two CP ranks sharing one GPU).  Larger calls keep every SM."""
        if len(self.calls) < 2:
            return 0
        if all(self.call_cta_tiles(c) <= sms for c in self.calls):
            return sms // 2
        return 0

    def call_algorithmic(self, c):
        """(bytes, flops) one decode call must move / do."""
        hl, hh, lo, hi, _, _ = c
        Hs = hh - hl
        toks = pages = 0
        P = self.w.page_size
        i = next(k for k, x in enumerate(self.calls) if x is c)
        rng = self.ranges[i].cpu().tolist() if self.ranges is not None else None
        for r, L in enumerate(self.w.ctx_lens):
            if rng is not None:
                lo, hi = rng[0][r], rng[1][r]
            a, b = lo, (L if hi < 0 else min(hi, L))
            if b > a:
                toks += b - a
                pages += (b - 1) // P - a // P + 1
        rows = self.B * Hs
        # with several KV heads a call reads the KV heads its query heads map to
        Hkv = self.w.num_kv_heads
        kv_read = 1 if Hkv == 1 else len({h // (self.H // Hkv) for h in range(hl, hh)})
        return algorithmic(Hs, toks, rows, pages, kv_read)

    def decode(self, c, q=None, bt=None, ctx=None, max_sms=0, ws=None):
        inp = self.inp
        ws = self.ws if ws is None else ws
        hl, hh, lo, hi, out, lse = c
        q = q if q is not None else inp.q
        bt = bt if bt is not None else inp.block_table
        ctx = ctx if ctx is not None else inp.ctx_lens
        if self.ranges is not None or max_sms or inp.pool.dim() == 4:
            i = next(k for k, x in enumerate(self.calls) if x is c)
            rl = self.ranges[i, 0] if self.ranges is not None else None
            rh = self.ranges[i, 1] if self.ranges is not None else None
            self.S.splash_decode_attn_ex(q, inp.pool, bt, ctx, hl, hh, lo, hi, out, lse, ws,
                                         self.w.scale, tok_lo_r=rl, tok_hi_r=rh,
                                         max_sms=max_sms)
        else:
            self.S.splash_decode_attn(q, inp.pool, bt, ctx, hl, hh, lo, hi, out, lse, ws,
                                      self.w.scale)

    def run(self, q=None, bt=None, ctx=None, decode_events=None, row_events=None):
        """One step.  decode_events: a (start, end) pair recorded around the step's
        back-to-back decode calls; row_events: pairs around the merge and the migration."""
        import torch
        if decode_events is not None:
            decode_events[0].record()
        cur = torch.cuda.current_stream()
        if len(self.calls) > 1:
            fork = torch.cuda.Event()
            fork.record(cur)
            self.stream_b.wait_event(fork)
        for k, c in enumerate(self.calls):
            if k % 2:
                with torch.cuda.stream(self.stream_b):
                    self.decode(c, q, bt, ctx, max_sms=self.call_sms, ws=self.ws_b)
            else:
                self.decode(c, q, bt, ctx, max_sms=self.call_sms)
        if len(self.calls) > 1:
            join = torch.cuda.Event()
            join.record(self.stream_b)
            cur.wait_event(join)
        if decode_events is not None:
            decode_events[1].record()
        # the handoff's migration does not depend on the merge: a small one runs on the
        # second stream alongside the merge; a large one would contend with the merge and
        # the decode tail for SMs and HBM (see the background-handoff measurement), so it
        # runs after them
        two = len(self.calls) > 1 and self.migrate_bytes() <= (64 << 20)
        mig_stream = self.stream_b if two else cur
        with torch.cuda.stream(mig_stream):
            if row_events is not None:
                row_events["kv_migrate"][0].record()
            self.S.splash_kv_migrate(self.inp.pool, self.pool2, self.src_ids, self.dst_ids)
            if row_events is not None:
                row_events["kv_migrate"][1].record()
        if self.merge:
            if row_events is not None:
                row_events["lse_merge"][0].record()
            self.S.splash_lse_merge(self.po, self.pl, self.out, self.lse)
            if row_events is not None:
                row_events["lse_merge"][1].record()
        if two:
            done = torch.cuda.Event()
            done.record(self.stream_b)
            cur.wait_event(done)

    def run_background_handoff(self, side2, max_sms, dec_events, join_event):
        """The step's decode calls on the current stream with at most max_sms SMs, while
        the handoff's page migration runs on stream side2 (forked from the current
        stream; joined back at the end).  dec_events brackets the decode calls."""
        import torch
        cur = torch.cuda.current_stream()
        fork = torch.cuda.Event()
        fork.record(cur)
        side2.wait_event(fork)
        with torch.cuda.stream(side2):
            self.S.splash_kv_migrate(self.inp.pool, self.pool2, self.src_ids, self.dst_ids)
            join_event.record(side2)
        dec_events[0].record()
        for c in self.calls:
            self.decode(c, max_sms=max_sms)
        dec_events[1].record()
        cur.wait_event(join_event)

    def merge_bytes(self):
        """Bytes splash_lse_merge must move: every share's fp32 rows read once, one written."""
        n = self.po.shape[0] if self.merge else 0
        return (n + 1) * self.B * self.H * (512 * 4 + 4)

    def migrate_bytes(self):
        return 2 * self.page_bytes * int(self.src_ids.numel())


def pack(tensors, device):
    """One byte buffer on `device` holding copies of `tensors` at 256-byte aligned
    offsets, and views of it with the tensors' dtypes and shapes: a step's inputs (or
    outputs) then move between host and device in one copy."""
    import torch
    offs, total = [], 0
    for t in tensors:
        offs.append(total)
        total += (t.numel() * t.element_size() + 255) // 256 * 256
    buf = torch.empty(total, dtype=torch.uint8, device=device)
    views = []
    for t, o in zip(tensors, offs):
        n = t.numel() * t.element_size()
        v = buf[o:o + n].view(t.dtype).view(t.shape)
        v.copy_(t)
        views.append(v)
    return buf, views


def algorithmic(Hs, tokens_in_call, rows, pages, kv_heads_read=1):
    """Bytes and flops one decode call must move / do: every KV token once (576 bf16
    per KV head the call reads), q rows (576 bf16), fp32 out rows + lse, 4 bytes per
    page id."""
    bytes_ = (tokens_in_call * 576 * 2 * kv_heads_read + rows * 576 * 2 + rows * (512 * 4 + 4)
              + pages * 4)
    flops = 2.0 * tokens_in_call * Hs * (576 + 512)
    return bytes_, flops


# ----------------------------------------------------------------------------- arms

def run_ours(args, world, rank, local):
    import torch
    from layout_agnostic_paged_gb300 import splash as S
    from layout_agnostic_paged_gb300 import workloads as W

    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    S.load_library()
    w = W.ALL[args.workload]()
    # weak scaling: every rank owns its own batch of the workload (own seed)
    inp = W.make_decode_inputs(w.ctx_lens, w.num_heads, w.page_size, w.seed + 1000 * rank,
                               device=device, spare_frac=w.spare_frac, num_kv_heads=w.num_kv_heads)
    # q, block table and context lengths share one buffer: the end-to-end leg copies
    # them in with one transfer
    ins = [inp.q, inp.block_table, inp.ctx_lens]
    if w.per_request_splits:
        ins.append(W.per_request_ranges(w))
    in_pack, views = pack(ins, device)
    inp.q, inp.block_table, inp.ctx_lens = views[:3]
    step = Step(w, inp, device, ranges=views[3] if w.per_request_splits else None,
                call_sms=args.call_sms)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=device)
    K, Wm = args.steps, args.warmup

    # one eager pass (caches the per-device state), then two sets of CUDA graphs of one
    # step each: plain graphs for the headline timing, and instrumented graphs with
    # in-graph events around the decode calls, the merge and the migration for the
    # per-row breakdown.  Event nodes inside a graph end the programmatic-dependent-
    # launch overlap between neighbouring kernels and add latency, so they stay out of
    # the headline graphs.
    step.run()
    torch.cuda.synchronize()

    def new_event():
        try:
            return torch.cuda.Event(enable_timing=True, external=True)
        except TypeError:
            return None

    side = torch.cuda.Stream(device)

    def capture(**kw):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=side):
            step.run(**kw)
        return g

    graphs = [capture() for _ in range(max(K, 1))]
    inst, dec_ev, row_ev = [], [], []
    for k in range(max(K, 1)):
        evs = (new_event(), new_event())
        rows = {n: (new_event(), new_event()) for n in ("lse_merge", "kv_migrate")}
        if None in evs or any(e is None for pair in rows.values() for e in pair):
            break
        inst.append(capture(decode_events=evs, row_events=rows))
        dec_ev.append(evs)
        row_ev.append(rows)
    stream = torch.cuda.current_stream(device)
    for k in range(Wm):
        flush.zero_()
        graphs[k % len(graphs)].replay()
    torch.cuda.synchronize()

    # timed region: K plain steps, the L2 flushed before each
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    barrier(world)
    torch.cuda.synchronize()
    with ClockSampler(local, enabled=not args.no_clocks) as clk:
        for k in range(K):
            flush.zero_()
            ev[k][0].record(stream)
            graphs[k].replay()
            ev[k][1].record(stream)
        torch.cuda.synchronize()
    barrier(world)
    step_ms = [ev[k][0].elapsed_time(ev[k][1]) for k in range(K)]

    # breakdown: K instrumented steps, same flush
    ncalls = len(step.calls)
    if len(inst) == max(K, 1):
        for k in range(K):
            flush.zero_()
            inst[k].replay()
        torch.cuda.synchronize()
        dec_ms = [dec_ev[k][0].elapsed_time(dec_ev[k][1]) / ncalls for k in range(K)]
        dec_src = (f"CUDA events captured inside instrumented step graphs around the step's "
                   f"{ncalls} back-to-back decode call(s) (a second timed pass of K steps); "
                   f"per call = their span / {ncalls}")
    else:   # events cannot be captured: time graph replays of single decode calls
        row_ev = [None]
        dec_ms = []
        for c in step.calls[:2]:
            g1 = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g1, stream=side):
                step.decode(c)
            for k in range(K):
                flush.zero_()
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record(stream)
                g1.replay()
                b.record(stream)
                torch.cuda.synchronize()
                dec_ms.append(a.elapsed_time(b))
        dec_src = "CUDA events around graph replays of one decode call"
    # background handoff: the decode calls on all but RESERVED SMs while the page
    # migration runs on a second stream, against the decode calls alone on every SM
    handoff = None
    if len(inst) == max(K, 1):
        reserved = args.reserved_sms
        side2 = torch.cuda.Stream(device)
        g_alone, g_bg, ev_alone, ev_bg, ev_span = [], [], [], [], []
        for k in range(K):
            ea = (new_event(), new_event())
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=side):
                ea[0].record()
                for c in step.calls:
                    step.decode(c)
                ea[1].record()
            g_alone.append(g)
            ev_alone.append(ea)
            eb, es = (new_event(), new_event()), (new_event(), new_event())
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=side):
                es[0].record()
                step.run_background_handoff(side2, torch.cuda.get_device_properties(device)
                                            .multi_processor_count - reserved, eb,
                                            torch.cuda.Event())
                es[1].record()
            g_bg.append(g)
            ev_bg.append(eb)
            ev_span.append(es)
        for graphs_ in (g_alone, g_bg):
            for k in range(K):
                flush.zero_()
                graphs_[k].replay()
        torch.cuda.synchronize()
        t_alone = statistics.mean(a.elapsed_time(b) for a, b in ev_alone) * 1e3
        t_dec_bg = statistics.mean(a.elapsed_time(b) for a, b in ev_bg) * 1e3
        t_span = statistics.mean(a.elapsed_time(b) for a, b in ev_span) * 1e3
        t_mig = statistics.mean(row_ev[k]["kv_migrate"][0].elapsed_time(row_ev[k]["kv_migrate"][1])
                                for k in range(K)) * 1e3
        handoff = {
            "reserved_sms": reserved, "migrate_bytes": step.migrate_bytes(),
            "decode_us_alone": t_alone, "decode_us_with_background_migrate": t_dec_bg,
            "decode_slowdown_pct": 100.0 * (t_dec_bg - t_alone) / t_alone,
            "overlapped_us": t_span, "serial_us": t_alone + t_mig,
            "note": "decode calls with max_sms = SMs - reserved on one stream, splash_kv_migrate "
                    "on a second stream of the same graph; serial = decode alone + migrate alone",
        }
    rows_report = {}
    if row_ev[0] is not None:
        mig_us = statistics.mean(row_ev[k]["kv_migrate"][0].elapsed_time(row_ev[k]["kv_migrate"][1])
                                 for k in range(K)) * 1e3
        rows_report["kv_migrate"] = {"us": mig_us, "bytes": step.migrate_bytes(),
                                     "gb_s": step.migrate_bytes() / mig_us / 1e3}
        if step.merge:
            mer_us = statistics.mean(row_ev[k]["lse_merge"][0].elapsed_time(row_ev[k]["lse_merge"][1])
                                     for k in range(K)) * 1e3
            rows_report["lse_merge"] = {"us": mer_us, "bytes": step.merge_bytes(),
                                        "gb_s": step.merge_bytes() / mer_us / 1e3}
    total_ms = max_over_ranks(sum(step_ms), world, device)
    status = S.splash_workspace_status(step.ws)
    if step.ws_b is not None:
        status |= S.splash_workspace_status(step.ws_b)
    if status != 0:
        raise RuntimeError(f"device status word set: {status}")

    # end to end through the public API with host buffers: the pinned q / block table /
    # context lengths copied in (one transfer of the packed inputs), the step, and the
    # merged out / lse copied back (one transfer), every step
    in_h = in_pack.cpu().pin_memory()
    out_h = torch.empty(step.out_pack.shape, dtype=torch.uint8).pin_memory()
    h2d = in_h.numel()
    d2h = out_h.numel()
    e2e_ms = []
    for k in range(Wm + K):
        flush.zero_()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        in_pack.copy_(in_h, non_blocking=True)      # the graphs read the views of in_pack
        graphs[k % len(graphs)].replay()
        out_h.copy_(step.out_pack, non_blocking=True)
        stream.synchronize()
        if k >= Wm:
            e2e_ms.append((time.perf_counter() - t0) * 1e3)
    e2e_total = max_over_ranks(sum(e2e_ms), world, device)

    tokens = w.kv_tokens
    total_tokens = sum_over_ranks(float(tokens), world, device)
    value = total_tokens * K / (total_ms / 1e3)
    e2e_value = total_tokens * K / (e2e_total / 1e3)

    # roofline of the dominant kernel: the decode call (plan + tcgen05 decode + combine)
    hbm_peak, bf16_peak, peak_src = measured_peaks()
    call_bytes = [step.call_algorithmic(c) for c in step.calls]
    alg_bytes = sum(b for b, _ in call_bytes) / len(call_bytes)
    alg_flops = sum(f for _, f in call_bytes) / len(call_bytes)
    dec_avg_s = statistics.mean(dec_ms) / 1e3
    achieved_gbs = alg_bytes / dec_avg_s / 1e9
    achieved_tfs = alg_flops / dec_avg_s / 1e12
    traffic = ncu_traffic(args.workload)
    clocks = clk.summary()

    line = None
    if rank == 0:
        cpu = None
        if not args.no_cpu_baseline and world == 1:
            cpu = cpu_baseline(w, inp, args.cpu_seconds)
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": K,
            "warmup": Wm, "ms_per_step": total_ms / K, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {
                "workload": w.name, "global_batch": w.batch * world, "seq_len": max(w.ctx_lens),
                "heads": w.num_heads, "page_size": w.page_size, "kv_tokens_per_rank": tokens,
                "parallelism": f"replicas{world}" if world > 1 else "single",
                "step": step.pattern + "; captured as one CUDA graph",
                "l2": "512 MB flush write before every timed step",
            },
            "clocks": clocks,
            "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h, "ms_per_step": e2e_total / K},
            "gpu_launches": step.launches_per_step * K,
            "roofline": {"bound": "hbm", "achieved": achieved_gbs, "peak": hbm_peak,
                         "unit": "GB/s", "frac": achieved_gbs / hbm_peak, "traffic": traffic,
                         "kernel": "splash_decode_attn call (plan + tcgen05 decode + combine)",
                         "alg_bytes_per_launch": alg_bytes, "launch_us": dec_avg_s * 1e6,
                         "timing": dec_src, "peak_source": f"{peak_src} hbm_gbs",
                         "tflops": achieved_tfs,
                         "tensor_frac_of_bf16_peak": achieved_tfs / bf16_peak},
            "other_rows": {k: dict(v, frac_of_hbm=v["gb_s"] / hbm_peak) for k, v in rows_report.items()},
            "background_handoff": handoff,
            "cpu_baseline": cpu,
        }
        print(json.dumps(line), flush=True)
    return line


def cpu_baseline(w, inp, seconds: float):
    """The fp64 oracle, as it stands, on this host's cores over a bounded sample of the
    same workload (whole requests, all heads), in KV-tokens/s."""
    import numpy as np
    import oracle
    q = oracle.bf16_bits(inp.q)
    pool = oracle.bf16_bits(inp.pool)
    bt = inp.block_table.cpu().numpy()
    ctx = inp.ctx_lens.cpu().numpy()
    B = len(ctx)
    # grow the sample (requests, cycling) until it takes about `seconds`
    t_total, toks, n = 0.0, 0, 0
    r = 0
    while t_total < seconds and n < 1000 * B:
        t0 = time.perf_counter()
        oracle.decode_attn(q[r:r + 1], pool, bt[r:r + 1], ctx[r:r + 1], w.scale)
        t_total += time.perf_counter() - t0
        toks += int(ctx[r])
        n += 1
        r = (r + 1) % B
    return {"value": toks / t_total, "unit": UNIT, "cores": oracle.num_threads(), "kind": "oracle",
            "sample": f"{n} whole requests (all {w.num_heads} heads, cycling over the batch), "
                      f"{toks} KV tokens, {t_total:.1f} s"}


def run_reference(args, world, rank, local):
    """The fp64 C oracle as the reference arm, timed on the host cores."""
    if rank != 0:
        return None
    import torch
    import oracle
    from layout_agnostic_paged_gb300 import workloads as W
    w = W.ALL[args.workload]()
    inp = W.make_decode_inputs(w.ctx_lens, w.num_heads, w.page_size, w.seed, device="cpu"
                               if w.kv_tokens <= 2_000_000 else "cuda:0", spare_frac=w.spare_frac,
                               num_kv_heads=w.num_kv_heads)
    q = oracle.bf16_bits(inp.q)
    pool = oracle.bf16_bits(inp.pool)
    bt = inp.block_table.cpu().numpy()
    ctx = inp.ctx_lens.cpu().numpy()
    # each step: a bounded sample of whole requests (all heads) sized so that
    # warm-up + steps stay within a few minutes
    t0 = time.perf_counter()
    oracle.decode_attn(q[:1], pool, bt[:1], ctx[:1], w.scale)
    per_req = max(time.perf_counter() - t0, 1e-3)
    budget = 120.0 / max(1, args.steps + args.warmup)
    n_req = max(1, min(len(ctx), int(budget / per_req)))
    times, toks = [], int(ctx[:n_req].sum())
    for k in range(args.warmup + args.steps):
        t0 = time.perf_counter()
        oracle.decode_attn(q[:n_req], pool, bt[:n_req], ctx[:n_req], w.scale)
        dt = time.perf_counter() - t0
        if k >= args.warmup:
            times.append(dt)
    total = sum(times)
    value = toks * args.steps / total
    sample = f"{n_req} of {len(ctx)} requests (all {w.num_heads} heads) per step, {toks} KV tokens"
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": total / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": {"workload": w.name, "global_batch": w.batch,
                                        "seq_len": max(w.ctx_lens), "heads": w.num_heads,
                                        "page_size": w.page_size},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": oracle.num_threads(),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return line


def main():
    args = parse_args()
    if args.impl == "reference":
        world = int(os.environ.get("WORLD_SIZE", "1"))
        rank = int(os.environ.get("RANK", "0"))
        run_reference(args, world, rank, int(os.environ.get("LOCAL_RANK", "0")))
        return
    world, rank, local = dist_setup(args)
    try:
        run_ours(args, world, rank, local)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
