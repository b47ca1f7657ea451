#!/usr/bin/env python3
"""Benchmark of the paged MLA decode hot path on GB300: KV-tokens/s, with the
decode kernel's roofline fraction and the fp64 CPU oracle as a baseline.

One step = one pass of the workload's hot-path rows over one synthetic batch
(step_pattern).  The default workload is the largest single-GPU configuration,
the ragged mixed batch with a layout handoff: 256 requests with log-uniform
contexts of 512..131,072 tokens, 128 query heads over one shared 576-wide latent
KV head, page 64, shuffled page ids.  Its step is
  * one decode call over the whole batch (tcgen05 decode, which computes its own
    split plan, + combine of requests cut across CTA groups);
  * the handoff: splash_kv_migrate of a seeded 25% of the requests' pages into a
    second block pool at fresh page ids (their block-table rows are rewritten on
    the host, once: an input of the step);
  * the decode rerun as two calls, each owning its requests as storage rows of the
    same batch: the remaining requests on pool 1 and the moved ones on pool 2.
Other workloads (--workload): tiny and full_heads (one call), cp_long (8 token
shares + splash_lse_merge), head_shard (8 calls of 16 heads), ragged_cp and gqa.
value = KV tokens decoded for every query head per step (the ragged step decodes
the batch twice) / step time.

Timing: W untimed warm-up steps, then K timed steps; before every step a 512 MB
buffer is written to flush the 129 MB L2 (outside the timed events); each step
is one CUDA graph replay bracketed by CUDA events on the launching stream and the
K step times are summed; ranks meet at a barrier (+ synchronize) before and after
and the max over ranks is reported.  A second pass of instrumented graphs gives
the per-phase breakdown, and a third the first decode phase with a background
page migration.  `--impl reference` times the fp64 C oracle instead, running the
same step pattern over a bounded sample of the requests.
"""
from __future__ import annotations

import argparse
import hashlib
import io
import json
import math
import os
import re
import statistics
import subprocess
import sys
import tempfile
import time
from dataclasses import dataclass

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
    ap.add_argument("--workload", default="ragged_handoff",
                    help="ragged_handoff | tiny | full_heads | cp_long | head_shard | ragged_cp | gqa")
    ap.add_argument("--reserved-sms", type=int, default=16,
                    help="SMs left to the background page migration in the handoff-overlap "
                         "measurement")
    ap.add_argument("--call-sms", type=int, default=-1,
                    help="SM budget of each decode call of a multi-call phase (-1: half the "
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
    """Hash of the decode kernel's sources with comments and whitespace removed, so that
    the stored ncu counters stay attached to the code they were taken on and to nothing
    else (the sources hold no string literal containing a comment marker)."""
    h = hashlib.sha256()
    for name in ("decode_tc.cu", "common.cuh", "plan.cuh"):
        with open(os.path.join(ROOT, "layout_agnostic_paged_gb300", "csrc", name)) as f:
            text = f.read()
        text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
        text = re.sub(r"//[^\n]*", " ", text)
        h.update(" ".join(text.split()).encode())
    return h.hexdigest()[:16]


def ncu_traffic(workload: str, alg_bytes_per_step: float):
    """DRAM bytes of the step's decode launches from the committed ncu summary, if it
    was taken on the current kernel source (else None).  An entry either gives the bytes
    of the workload's own decode launches in one step (dram_bytes_per_step) or the ratio
    of DRAM bytes to algorithmic bytes measured on a scaled-down case of the same
    workload (dram_over_algorithmic), applied to the step's algorithmic bytes."""
    p = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    e = d.get(workload)
    if not e or e.get("kernel_source_hash") != kernel_source_hash():
        return None
    if "dram_over_algorithmic" in e:
        return float(e["dram_over_algorithmic"]) * alg_bytes_per_step
    return float(e["dram_bytes_per_step"])


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

@dataclass
class CallSpec:
    """One decode call of a step: the ownership slice it computes and where it writes.

    rows: the requests (storage rows) the call owns, None for the whole batch;
    pool: "pool1" (the batch's pool) or "pool2" (the handoff's destination pool);
    share: index of the per-request token share (None: the scalar tok_lo / tok_hi);
    out: "out" (the step's result), "pre" (the output before the handoff) or "part<i>"
    (CP partial i, merged afterwards)."""
    head_lo: int
    head_hi: int
    tok_lo: int = 0
    tok_hi: int = -1
    rows: tuple | None = None
    pool: str = "pool1"
    share: int | None = None
    out: str = "out"


def step_pattern(w, moved=None):
    """The phases of one step of workload w, in order: ("decode", [CallSpec, ...]) (the
    calls of a phase are independent), ("merge", n) or ("migrate",).

      * TP / DOP head shards (head_shards > 1): one call per head shard;
      * ragged + handoff (migrate_frac > 0): one call over the batch, the migration of
        the moved requests' pages to the second pool, then the decode rerun as two calls
        (the remaining requests on pool 1, the moved ones on pool 2), each owning its
        requests as storage rows of the same batch;
      * CP (token_splits > 1): one call per token share, then the merge of the shares;
      * otherwise one call over the batch.
    moved: the requests the handoff moves (required when migrate_frac > 0)."""
    B, H = w.batch, w.num_heads
    if w.head_shards > 1:
        hs = H // w.head_shards
        return [("decode", [CallSpec(i * hs, (i + 1) * hs) for i in range(w.head_shards)])]
    if w.migrate_frac > 0:
        mv = set(moved)
        keep = tuple(r for r in range(B) if r not in mv)
        return [("decode", [CallSpec(0, H, out="pre")]), ("migrate",),
                ("decode", [CallSpec(0, H, rows=keep, pool="pool1"),
                            CallSpec(0, H, rows=tuple(sorted(mv)), pool="pool2")])]
    if w.token_splits > 1:
        n = w.token_splits
        if w.per_request_splits:
            calls = [CallSpec(0, H, share=i, out=f"part{i}") for i in range(n)]
        else:
            span = -(-max(w.ctx_lens) // n)
            calls = [CallSpec(0, H, i * span, (i + 1) * span if i + 1 < n else -1, out=f"part{i}")
                     for i in range(n)]
        return [("decode", calls), ("merge", n)]
    return [("decode", [CallSpec(0, H)])]


def describe_pattern(w, phases):
    parts = []
    for ph in phases:
        if ph[0] == "decode":
            cs = ph[1]
            if len(cs) == 1 and cs[0].rows is None:
                parts.append("one decode call over the batch"
                             + ("" if cs[0].out != "pre" else " (before the handoff)"))
            elif w.head_shards > 1:
                parts.append(f"{len(cs)} head-shard calls of {cs[0].head_hi - cs[0].head_lo} heads")
            elif cs[0].rows is not None:
                parts.append(f"decode rerun as {len(cs)} calls owning request subsets in place "
                             f"({', '.join(f'{len(c.rows)} on {c.pool}' for c in cs)})")
            else:
                kind = "per-request token-share" if cs[0].share is not None else "token-share"
                parts.append(f"{len(cs)} CP {kind} calls")
        elif ph[0] == "merge":
            parts.append(f"splash_lse_merge of {ph[1]} shares")
        else:
            parts.append(f"splash_kv_migrate of {int(round(100 * w.migrate_frac))}% of the "
                         f"requests' pages to a second pool")
    return " -> ".join(parts)


def call_tokens_pages(w, c, ranges=None):
    """(KV tokens, pages) call c reads (ranges: the per-request share bounds, [n][2][B])."""
    toks = pages = 0
    P = w.page_size
    rows = range(w.batch) if c.rows is None else c.rows
    for r in rows:
        L = w.ctx_lens[r]
        if c.share is not None:
            lo, hi = int(ranges[c.share][0][r]), int(ranges[c.share][1][r])
        else:
            lo, hi = c.tok_lo, c.tok_hi
        a, b = max(lo, 0), (L if hi < 0 else min(hi, L))
        if b > a:
            toks += b - a
            pages += (b - 1) // P - a // P + 1
    return toks, pages


def call_cta_tiles(w, c, ranges=None):
    """(128-token tiles x 64-head groups) one decode call must process."""
    tiles = 0
    rows = range(w.batch) if c.rows is None else c.rows
    for r in rows:
        L = w.ctx_lens[r]
        if c.share is not None:
            lo, hi = int(ranges[c.share][0][r]), int(ranges[c.share][1][r])
        else:
            lo, hi = c.tok_lo, c.tok_hi
        a, b = max(lo, 0), (L if hi < 0 else min(hi, L))
        if b > a:
            tiles += (b - 1) // 128 - a // 128 + 1
    return tiles * -(-(c.head_hi - c.head_lo) // 64)


def token_share_phase(calls):
    """Whether a phase's calls are the token shares of one CP group: the same heads and
    requests, each call a different share of every request's tokens (scalar ranges that
    do not overlap, or distinct per-request shares).  Such calls read disjoint KV."""
    if len(calls) < 2:
        return False
    c0 = calls[0]
    if any(c.head_lo != c0.head_lo or c.head_hi != c0.head_hi or c.rows != c0.rows
           or c.pool != c0.pool for c in calls):
        return False
    if all(c.share is not None for c in calls):
        return len({c.share for c in calls}) == len(calls)
    if any(c.share is not None for c in calls):
        return False
    spans = sorted((c.tok_lo, c.tok_hi if c.tok_hi >= 0 else math.inf) for c in calls)
    return all(a[1] <= b[0] for a, b in zip(spans, spans[1:]))


def pick_lanes(calls):
    """Streams a decode phase's calls run on.  The token shares of a CP group run at once,
    as the group's ranks would, each call on its own stream (those that find no free SMs
    start as the first ones finish); other multi-call phases alternate between two
    streams."""
    if token_share_phase(calls):
        return len(calls)
    return 2 if len(calls) > 1 else 1


def pick_call_sms(w, calls, sms, ranges=None):
    """SM budget of each call of a phase (0: all).  The concurrent token shares of a CP
    group each get 1/min(n, 4) of the SMs: four at a time of an eight-way group (a
    quarter each; an eighth would leave SMs idle, as a 64-head call's CTAs come in pairs,
    and measured slower on both CP workloads), two halves for two shares.  A phase of
    several calls whose tiles each fill at most one wave of the GPU would leave SMs idle
    while the other stream's call waits for them; such calls each get half the SMs and
    run side by side (two ranks sharing one GPU).  Larger calls, and a phase of one call,
    keep every SM."""
    if len(calls) < 2:
        return 0
    if token_share_phase(calls):
        return sms // min(len(calls), 4)
    if all(call_cta_tiles(w, c, ranges) <= sms for c in calls):
        return sms // 2
    return 0


def algorithmic(Hs, tokens_in_call, rows, pages, kv_heads_read=1):
    """Bytes and flops one decode call must move / do: every KV token once (576 bf16
    per KV head the call reads), q rows (576 bf16), fp32 out rows + lse, 4 bytes per
    page id."""
    bytes_ = (tokens_in_call * 576 * 2 * kv_heads_read + rows * 576 * 2 + rows * (512 * 4 + 4)
              + pages * 4)
    flops = 2.0 * tokens_in_call * Hs * (576 + 512)
    return bytes_, flops


def call_algorithmic(w, c, ranges=None):
    toks, pages = call_tokens_pages(w, c, ranges)
    Hs = c.head_hi - c.head_lo
    nreq = w.batch if c.rows is None else len(c.rows)
    Hkv = w.num_kv_heads
    kv_read = 1 if Hkv == 1 else len({h // (w.num_heads // Hkv) for h in range(c.head_lo, c.head_hi)})
    return algorithmic(Hs, toks, nreq * Hs, pages, kv_read)


def decoded_tokens(w, phases, ranges=None):
    """KV tokens a step decodes for every query head: the sum over its calls of the
    call's tokens times the share of the heads it covers."""
    t = 0.0
    for ph in phases:
        if ph[0] == "decode":
            for c in ph[1]:
                t += call_tokens_pages(w, c, ranges)[0] * (c.head_hi - c.head_lo) / w.num_heads
    return int(round(t))


def workload_config(w, phases, world):
    """The `config` object of the JSON line (the same for both arms)."""
    return {"workload": w.name, "global_batch": w.batch * world, "seq_len": max(w.ctx_lens),
            "heads": w.num_heads, "page_size": w.page_size,
            "kv_tokens_per_rank": w.kv_tokens,
            "decoded_kv_tokens_per_step_per_rank": decoded_tokens(
                w, phases, per_request_ranges_or_none(w)),
            "parallelism": f"replicas{world}" if world > 1 else "single",
            "step": describe_pattern(w, phases),
            "l2": "inputs larger than L2 where the workload's cache is; a 512 MB flush write "
                  "before every timed step in every case"}


def per_request_ranges_or_none(w):
    if not w.per_request_splits:
        return None
    from layout_agnostic_paged_gb300 import workloads as W
    return W.per_request_ranges(w).tolist()


class Step:
    """Device buffers and calls of one step over one batch (see step_pattern)."""

    def __init__(self, w, inp, device, call_sms=-1, migration=None):
        import torch
        from layout_agnostic_paged_gb300 import splash as S
        from layout_agnostic_paged_gb300 import workloads as W
        self.S, self.w, self.inp = S, w, inp
        B, H = w.batch, w.num_heads
        self.B, self.H = B, H
        self.mig = None
        if w.migrate_frac > 0:
            self.mig = migration or W.make_migration(inp, w.migrate_frac, seed=w.seed)
        self.phases = step_pattern(w, self.mig.requests if self.mig else None)
        self.pattern = describe_pattern(w, self.phases)
        # host inputs that the end-to-end leg copies in every step: q, block table(s),
        # context lengths, request rows, per-request ranges -- packed in one buffer
        ins = {"q": inp.q, "bt1": inp.block_table, "ctx": inp.ctx_lens}
        if self.mig is not None:
            bt2 = torch.full(tuple(inp.block_table.shape), -1, dtype=torch.int32)
            bt2[torch.tensor(self.mig.requests, dtype=torch.long)] = self.mig.new_block_table
            ins["bt2"] = bt2
        self.rows_key = {}
        for ph in self.phases:
            if ph[0] == "decode":
                for k, c in enumerate(ph[1]):
                    if c.rows is not None:
                        key = f"rows_{c.pool}"
                        ins[key] = torch.tensor(c.rows, dtype=torch.int32)
                        self.rows_key[id(c)] = key
        self.ranges_host = per_request_ranges_or_none(w)
        if self.ranges_host is not None:
            ins["ranges"] = W.per_request_ranges(w)
        self.in_pack, views = pack(list(ins.values()), device)
        self.dev = dict(zip(ins.keys(), views))
        inp.q, inp.block_table, inp.ctx_lens = self.dev["q"], self.dev["bt1"], self.dev["ctx"]
        # outputs: the step's result (read back by the end-to-end leg) and scratch outputs
        self.out_pack, (self.out, self.lse) = pack(
            [torch.empty(B, H, 512), torch.empty(B, H)], device)
        self.outs = {"out": (self.out, self.lse)}
        n_parts = max([ph[1] for ph in self.phases if ph[0] == "merge"], default=0)
        if n_parts:
            self.po = torch.empty(n_parts, B, H, 512, device=device)
            self.pl = torch.empty(n_parts, B, H, device=device)
            for i in range(n_parts):
                self.outs[f"part{i}"] = (self.po[i], self.pl[i])
        if any(c.out == "pre" for ph in self.phases if ph[0] == "decode" for c in ph[1]):
            self.outs["pre"] = (torch.empty(B, H, 512, device=device),
                                torch.empty(B, H, device=device))
        self.pool2 = None
        if self.mig is not None:
            self.pool2 = torch.empty((self.mig.dst_num_pages,) + tuple(inp.pool.shape[1:]),
                                     dtype=inp.pool.dtype, device=device)
            self.src_ids = self.mig.src_ids.to(device)
            self.dst_ids = self.mig.dst_ids.to(device)
            self.page_bytes = int(inp.pool[0].numel() * inp.pool.element_size())
        # call k of a decode phase runs on lane k % lanes: lane 0 is the current stream,
        # the others streams of their own; each lane has its own workspace (sized for the
        # largest call it runs)
        self.lanes = [pick_lanes(ph[1]) if ph[0] == "decode" else 1 for ph in self.phases]
        n_lanes = max(self.lanes)
        self.streams = [None] + [torch.cuda.Stream(device) for _ in range(n_lanes - 1)]
        need = [0] * n_lanes
        desc = S.make_desc(inp.q, inp.pool, inp.block_table, w.scale)
        with torch.cuda.device(device):
            for ph, lanes in zip(self.phases, self.lanes):
                if ph[0] == "decode":
                    for k, c in enumerate(ph[1]):
                        desc.num_reqs = B if c.rows is None else len(c.rows)
                        n = S.splash_decode_workspace_size(desc, c.head_lo, c.head_hi)
                        if n == 0:
                            raise S.SplashError(S.SPLASH_ERR_UNSUPPORTED, "splash_decode_workspace_size")
                        need[k % lanes] = max(need[k % lanes], n)
        self.wss = [torch.empty(n, dtype=torch.uint8, device=device) for n in need if n]
        self.ws = self.wss[0]
        sms = torch.cuda.get_device_properties(device).multi_processor_count
        self.sms = sms
        self.call_sms = {}
        for ph in self.phases:
            if ph[0] == "decode":
                s = pick_call_sms(w, ph[1], sms, self.ranges_host) if call_sms < 0 else call_sms
                for c in ph[1]:
                    self.call_sms[id(c)] = s
        # a decode call launches the decode kernel (which computes its own split plan)
        # and the combine kernel
        self.launches_per_step = sum(2 * len(ph[1]) if ph[0] == "decode" else 1
                                     for ph in self.phases)

    def decode_calls(self):
        return [c for ph in self.phases if ph[0] == "decode" for c in ph[1]]

    def decode(self, c, ws, max_sms=None):
        inp, d = self.inp, self.dev
        pool = inp.pool if c.pool == "pool1" else self.pool2
        bt = d["bt1"] if c.pool == "pool1" else d["bt2"]
        out, lse = self.outs[c.out]
        sms = self.call_sms[id(c)] if max_sms is None else max_sms
        rows = d[self.rows_key[id(c)]] if id(c) in self.rows_key else None
        rl = rh = None
        if c.share is not None:
            rl, rh = d["ranges"][c.share, 0], d["ranges"][c.share, 1]
        if rows is not None or rl is not None or sms or pool.dim() == 4:
            self.S.splash_decode_attn_ex(inp.q, pool, bt, d["ctx"], c.head_lo, c.head_hi, c.tok_lo,
                                         c.tok_hi, out, lse, ws, self.w.scale, tok_lo_r=rl,
                                         tok_hi_r=rh, rows=rows, max_sms=sms)
        else:
            self.S.splash_decode_attn(inp.q, pool, bt, d["ctx"], c.head_lo, c.head_hi, c.tok_lo,
                                      c.tok_hi, out, lse, ws, self.w.scale)

    def run_phase(self, ph, max_sms=None):
        import torch
        if ph[0] == "decode":
            calls = ph[1]
            lanes = self.lanes[self.phases.index(ph)]
            cur = torch.cuda.current_stream()
            if lanes > 1:
                fork = torch.cuda.Event()
                fork.record(cur)
                for st in self.streams[1:lanes]:
                    st.wait_event(fork)
            for k, c in enumerate(calls):
                lane = k % lanes
                if lane:
                    with torch.cuda.stream(self.streams[lane]):
                        self.decode(c, self.wss[lane], max_sms)
                else:
                    self.decode(c, self.ws, max_sms)
            for st in self.streams[1:lanes]:
                join = torch.cuda.Event()
                join.record(st)
                cur.wait_event(join)
        elif ph[0] == "merge":
            self.S.splash_lse_merge(self.po[:ph[1]], self.pl[:ph[1]], self.out, self.lse)
        else:
            self.migrate()

    def migrate(self):
        self.S.splash_kv_migrate(self.inp.pool, self.pool2, self.src_ids, self.dst_ids)

    def run(self, events=None):
        """One step; events: one (start, end) pair per phase, recorded around it."""
        for i, ph in enumerate(self.phases):
            if events is not None:
                events[i][0].record()
            self.run_phase(ph)
            if events is not None:
                events[i][1].record()

    def run_background_handoff(self, side2, max_sms, dec_events, join_event):
        """The step's first decode phase on the current stream with at most max_sms SMs,
        while the handoff's page migration runs on stream side2 (forked from the current
        stream; joined back at the end).  dec_events brackets the decode phase."""
        import torch
        cur = torch.cuda.current_stream()
        fork = torch.cuda.Event()
        fork.record(cur)
        side2.wait_event(fork)
        with torch.cuda.stream(side2):
            self.migrate()
            join_event.record(side2)
        dec_events[0].record()
        self.run_phase(self.phases[0], max_sms=max_sms)
        dec_events[1].record()
        cur.wait_event(join_event)

    def merge_bytes(self, n):
        """Bytes splash_lse_merge must move: every share's fp32 rows read once, one written."""
        return (n + 1) * self.B * self.H * (512 * 4 + 4)

    def migrate_bytes(self):
        return 2 * self.page_bytes * int(self.src_ids.numel()) if self.mig is not None else 0


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
    step = Step(w, inp, device, call_sms=args.call_sms)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=device)
    K, Wm = args.steps, args.warmup
    nph = len(step.phases)

    # one eager pass (caches the per-device state), then two sets of CUDA graphs of one
    # step each: plain graphs for the headline timing, and instrumented graphs with
    # in-graph events around every phase for the per-row breakdown.  Event nodes inside
    # a graph end the programmatic-dependent-launch overlap between neighbouring kernels
    # and add latency, so they stay out of the headline graphs.
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
    inst, ph_ev = [], []
    for k in range(max(K, 1)):
        evs = [(new_event(), new_event()) for _ in range(nph)]
        if any(e is None for pair in evs for e in pair):
            break
        inst.append(capture(events=evs))
        ph_ev.append(evs)
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

    # breakdown: K instrumented steps, same flush; mean time of every phase
    ph_us = None
    if len(inst) == max(K, 1):
        for k in range(K):
            flush.zero_()
            inst[k].replay()
        torch.cuda.synchronize()
        ph_us = [statistics.mean(ph_ev[k][i][0].elapsed_time(ph_ev[k][i][1]) for k in range(K)) * 1e3
                 for i in range(nph)]
        dec_src = ("CUDA events captured inside instrumented step graphs around every decode "
                   "phase (a second timed pass of K steps)")
    else:   # events cannot be captured: time graph replays of each decode phase alone
        ph_us = []
        for ph in step.phases:
            g1 = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g1, stream=side):
                step.run_phase(ph)
            t = []
            for k in range(K):
                flush.zero_()
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record(stream)
                g1.replay()
                b.record(stream)
                torch.cuda.synchronize()
                t.append(a.elapsed_time(b) * 1e3)
            ph_us.append(statistics.mean(t))
        dec_src = "CUDA events around graph replays of each decode phase alone"

    # background handoff: the first decode phase on all but RESERVED SMs while the page
    # migration runs on a second stream, against that phase alone on every SM
    handoff = None
    if step.mig is not None and len(inst) == max(K, 1):
        reserved = args.reserved_sms
        side2 = torch.cuda.Stream(device)
        g_alone, g_bg, ev_alone, ev_bg, ev_span = [], [], [], [], []
        for k in range(K):
            ea = (new_event(), new_event())
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=side):
                ea[0].record()
                step.run_phase(step.phases[0])
                ea[1].record()
            g_alone.append(g)
            ev_alone.append(ea)
            eb, es = (new_event(), new_event()), (new_event(), new_event())
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=side):
                es[0].record()
                step.run_background_handoff(side2, step.sms - reserved, eb, torch.cuda.Event())
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
        t_mig = ph_us[[i for i, ph in enumerate(step.phases) if ph[0] == "migrate"][0]]
        handoff = {
            "reserved_sms": reserved, "migrate_bytes": step.migrate_bytes(),
            "decode_us_alone": t_alone, "decode_us_with_background_migrate": t_dec_bg,
            "decode_slowdown_pct": 100.0 * (t_dec_bg - t_alone) / t_alone,
            "overlapped_us": t_span, "serial_us": t_alone + t_mig,
            "note": "first decode phase with max_sms = SMs - reserved on one stream, "
                    "splash_kv_migrate on a second stream of the same graph; serial = decode "
                    "alone + migrate alone",
        }
    total_ms = max_over_ranks(sum(step_ms), world, device)
    status = 0
    for ws in step.wss:
        status |= S.splash_workspace_status(ws)
    if status != 0:
        raise RuntimeError(f"device status word set: {status}")

    # end to end through the public API with host buffers: the pinned inputs (q, block
    # tables, context lengths, request rows, ranges) copied in with one transfer, the
    # step, and its out / lse copied back with one transfer, every step
    in_h = step.in_pack.cpu().pin_memory()
    out_h = torch.empty(step.out_pack.shape, dtype=torch.uint8).pin_memory()
    h2d = in_h.numel()
    d2h = out_h.numel()
    e2e_ms = []
    for k in range(Wm + K):
        flush.zero_()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        step.in_pack.copy_(in_h, non_blocking=True)   # the graphs read views of in_pack
        graphs[k % len(graphs)].replay()
        out_h.copy_(step.out_pack, non_blocking=True)
        stream.synchronize()
        if k >= Wm:
            e2e_ms.append((time.perf_counter() - t0) * 1e3)
    e2e_total = max_over_ranks(sum(e2e_ms), world, device)

    tokens = decoded_tokens(w, step.phases, step.ranges_host)
    total_tokens = sum_over_ranks(float(tokens), world, device)
    value = total_tokens * K / (total_ms / 1e3)
    e2e_value = total_tokens * K / (e2e_total / 1e3)

    # roofline of the dominant kernel, the decode call (tcgen05 decode + combine):
    # the algorithmic bytes of every decode call of the step / the decode phases' time
    hbm_peak, bf16_peak, peak_src = measured_peaks()
    dec_idx = [i for i, ph in enumerate(step.phases) if ph[0] == "decode"]
    calls = step.decode_calls()
    alg = [call_algorithmic(w, c, step.ranges_host) for c in calls]
    alg_bytes = sum(b for b, _ in alg)
    alg_flops = sum(f for _, f in alg)
    dec_s = sum(ph_us[i] for i in dec_idx) / 1e6
    achieved_gbs = alg_bytes / dec_s / 1e9
    achieved_tfs = alg_flops / dec_s / 1e12
    traffic = ncu_traffic(args.workload, alg_bytes)
    clocks = clk.summary()
    rows_report = {}
    for i, ph in enumerate(step.phases):
        if ph[0] == "migrate":
            b = step.migrate_bytes()
            rows_report["kv_migrate"] = {"us": ph_us[i], "bytes": b, "gb_s": b / ph_us[i] / 1e3,
                                         "frac_of_hbm": b / ph_us[i] / 1e3 / hbm_peak}
        elif ph[0] == "merge":
            b = step.merge_bytes(ph[1])
            rows_report["lse_merge"] = {"us": ph_us[i], "bytes": b, "gb_s": b / ph_us[i] / 1e3,
                                        "frac_of_hbm": b / ph_us[i] / 1e3 / hbm_peak}
    phases_report = []
    for i, ph in enumerate(step.phases):
        e = {"phase": ph[0], "us": ph_us[i]}
        if ph[0] == "decode":
            pa = [call_algorithmic(w, c, step.ranges_host) for c in ph[1]]
            e["calls"] = len(ph[1])
            e["alg_bytes"] = sum(b for b, _ in pa)
            e["frac_of_hbm"] = e["alg_bytes"] / ph_us[i] / 1e3 / hbm_peak
        phases_report.append(e)

    line = None
    if rank == 0:
        cpu = None
        if not args.no_cpu_baseline and world == 1:
            cpu = cpu_baseline(w, inp, args.cpu_seconds)
        if any(ph[0] == "decode" and token_share_phase(ph[1]) for ph in step.phases):
            launch = ("the token shares of the CP group run at once, each call on its own stream "
                      "and workspace (calls beyond the SM budget start as SMs free up)")
        elif any(ph[0] == "decode" and len(ph[1]) > 1 for ph in step.phases):
            launch = "calls of a decode phase alternate between two streams, one workspace each"
        else:
            launch = "one stream"
        small = sorted({s for s in step.call_sms.values() if s})
        if small:
            launch += f"; each call limited to {small[0]} of {step.sms} SMs"
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": K,
            "warmup": Wm, "ms_per_step": total_ms / K, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": workload_config(w, step.phases, world),
            "launch": launch + "; each step captured as one CUDA graph",
            "clocks": clocks,
            "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h, "ms_per_step": e2e_total / K},
            "gpu_launches": step.launches_per_step * K,
            "roofline": {"bound": "hbm", "achieved": achieved_gbs, "peak": hbm_peak,
                         "unit": "GB/s", "frac": achieved_gbs / hbm_peak, "traffic": traffic,
                         "kernel": "splash_decode_attn call (tcgen05 decode with its split plan + combine)",
                         "alg_bytes_per_step": alg_bytes, "decode_us_per_step": dec_s * 1e6,
                         "decode_calls_per_step": len(calls),
                         "timing": dec_src, "peak_source": f"{peak_src} hbm_gbs",
                         "tflops": achieved_tfs,
                         "tensor_frac_of_bf16_peak": achieved_tfs / bf16_peak},
            "phases": phases_report,
            "other_rows": rows_report,
            "background_handoff": handoff,
            "cpu_baseline": cpu,
        }
        print(json.dumps(line), flush=True)
    return line


def cpu_baseline(w, inp, seconds: float):
    """The fp64 oracle, as it stands, on this host's cores over a bounded sample of the
    same workload (whole requests, all heads), in KV-tokens/s."""
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
    cores = oracle.num_threads()
    # the same oracle on one core, over the same requests in the same order, for a
    # quarter of the time (at most as many requests as the sample above)
    one = None
    oracle.set_num_threads(1)
    try:
        t1, toks1, n1 = 0.0, 0, 0
        while t1 < seconds / 4 and n1 < n:
            r = n1 % B
            # stop before a request that would overrun the budget by half (the time per
            # token so far predicts it)
            if toks1 > 0 and t1 + int(ctx[r]) * (t1 / toks1) > 1.5 * seconds / 4:
                break
            t0 = time.perf_counter()
            oracle.decode_attn(q[r:r + 1], pool, bt[r:r + 1], ctx[r:r + 1], w.scale)
            t1 += time.perf_counter() - t0
            toks1 += int(ctx[r])
            n1 += 1
        if t1 > 0:
            one = {"value": toks1 / t1, "cores": 1,
                   "sample": f"the first {n1} of those requests, {toks1} KV tokens, {t1:.1f} s"}
    finally:
        oracle.set_num_threads(cores)
    return {"value": toks / t_total, "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": f"{n} whole requests (all {w.num_heads} heads, cycling over the batch), "
                      f"{toks} KV tokens, {t_total:.1f} s",
            "one_core": one}


def reference_step(w, phases, q, pool, bt, ctx, sample, mig, pool2, bt2, ranges):
    """One step of the workload's pattern run by the fp64 oracle over the requests in
    `sample` (all heads): the same phases as the GPU step, restricted to the sample."""
    import numpy as np
    import oracle
    B, H = len(ctx), w.num_heads
    out = np.full((B, H, 512), np.nan)
    lse = np.full((B, H), np.nan)
    parts = {}
    sample = np.asarray(sample)
    for ph in phases:
        if ph[0] == "decode":
            for c in ph[1]:
                rows = sample if c.rows is None else np.intersect1d(sample, np.asarray(c.rows))
                if rows.size == 0:
                    continue
                p, t = (pool, bt) if c.pool == "pool1" else (pool2, bt2)
                if c.share is not None:
                    lo = np.asarray(ranges[c.share][0])[rows]
                    hi = np.asarray(ranges[c.share][1])[rows]
                    res = [oracle.decode_attn(q[r:r + 1], p, t[r:r + 1], ctx[r:r + 1], w.scale,
                                              c.head_lo, c.head_hi, int(a), int(b))
                           for r, a, b in zip(rows, lo, hi)]
                    o = np.concatenate([x[0] for x in res])
                    l = np.concatenate([x[1] for x in res])
                else:
                    o, l = oracle.decode_attn(q[rows], p, t[rows], ctx[rows], w.scale, c.head_lo,
                                              c.head_hi, c.tok_lo, c.tok_hi)
                if c.out.startswith("part"):
                    parts[c.out] = (rows, o, l)
                else:
                    out[rows, c.head_lo:c.head_hi] = o[:, c.head_lo:c.head_hi]
                    lse[rows, c.head_lo:c.head_hi] = l[:, c.head_lo:c.head_hi]
        elif ph[0] == "merge":
            rows = parts["part0"][0]
            po = np.stack([parts[f"part{i}"][1] for i in range(ph[1])])
            pl = np.stack([parts[f"part{i}"][2] for i in range(ph[1])])
            out[rows], lse[rows] = oracle.lse_merge(po, pl)
        else:
            moved = [r for r in mig.requests if r in set(sample.tolist())]
            if moved:
                src = np.concatenate([bt[r, :(ctx[r] + w.page_size - 1) // w.page_size]
                                      for r in moved]).astype(np.int32)
                dst = np.concatenate([bt2[r, :(ctx[r] + w.page_size - 1) // w.page_size]
                                      for r in moved]).astype(np.int32)
                oracle.kv_migrate(pool, pool2, src, dst)
    return out, lse


def run_reference(args, world, rank, local):
    """The fp64 C oracle as the reference arm, timed on the host cores: every step runs
    the workload's own step pattern (step_pattern) over a bounded sample of its
    requests."""
    if rank != 0:
        return None
    import numpy as np
    import torch
    import oracle
    from layout_agnostic_paged_gb300 import workloads as W
    w = W.ALL[args.workload]()
    dev = "cuda:0" if (w.kv_tokens > 2_000_000 and torch.cuda.is_available()) else "cpu"
    inp = W.make_decode_inputs(w.ctx_lens, w.num_heads, w.page_size, w.seed, device=dev,
                               spare_frac=w.spare_frac, num_kv_heads=w.num_kv_heads)
    mig = W.make_migration(inp, w.migrate_frac, seed=w.seed) if w.migrate_frac > 0 else None
    phases = step_pattern(w, mig.requests if mig else None)
    q = oracle.bf16_bits(inp.q)
    pool = oracle.bf16_bits(inp.pool)
    bt = inp.block_table.cpu().numpy()
    ctx = inp.ctx_lens.cpu().numpy()
    pool2 = bt2 = None
    if mig is not None:
        pool2 = np.zeros((mig.dst_num_pages,) + pool.shape[1:], dtype=np.uint16)
        bt2 = np.full(bt.shape, -1, dtype=np.int32)
        bt2[mig.requests] = mig.new_block_table.numpy()
    del inp
    ranges = per_request_ranges_or_none(w)
    # size the sample (whole requests, in a seeded order, every kind of call covered) so
    # that warm-up + steps stay within about two minutes
    order = np.random.default_rng(w.seed + 29).permutation(len(ctx))
    if mig is not None:   # alternate moved and remaining requests so both reruns run
        mv = [r for r in order if r in set(mig.requests)]
        kp = [r for r in order if r not in set(mig.requests)]
        order = np.array([x for pair in zip(kp, mv) for x in pair] + kp[len(mv):] + mv[len(kp):])
    t0 = time.perf_counter()
    reference_step(w, phases, q, pool, bt, ctx, order[:2], mig, pool2, bt2, ranges)
    per_tok = max(time.perf_counter() - t0, 1e-3) / max(1, int(ctx[order[:2]].sum()))
    budget = 120.0 / max(1, args.steps + args.warmup)
    n_req, acc = 0, 0
    while n_req < len(order) and (acc + ctx[order[n_req]]) * per_tok <= budget:
        acc += int(ctx[order[n_req]])
        n_req += 1
    n_req = max(n_req, min(2, len(order)))
    sample = np.sort(order[:n_req])
    sw = W.Workload(w.name, tuple(int(ctx[r]) for r in sample), w.num_heads, w.page_size, w.seed)
    sub_phases = [(ph[0], [CallSpec(c.head_lo, c.head_hi, c.tok_lo, c.tok_hi,
                                    None if c.rows is None else tuple(
                                        i for i, r in enumerate(sample) if r in set(c.rows)),
                                    c.pool, c.share, c.out) for c in ph[1]])
                  if ph[0] == "decode" else ph for ph in phases]
    toks = decoded_tokens(sw, sub_phases, None if ranges is None else
                          [[[row[r] for r in sample] for row in share] for share in ranges])
    times = []
    for k in range(args.warmup + args.steps):
        t0 = time.perf_counter()
        reference_step(w, phases, q, pool, bt, ctx, sample, mig, pool2, bt2, ranges)
        dt = time.perf_counter() - t0
        if k >= args.warmup:
            times.append(dt)
    total = sum(times)
    value = toks * args.steps / total
    desc = (f"{n_req} of {len(ctx)} requests (all {w.num_heads} heads) per step through the "
            f"step's phases, {toks} decoded KV tokens")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": total / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": workload_config(w, phases, world),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": oracle.num_threads(),
                         "kind": "oracle", "sample": desc},
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
