"""Helpers shared by the GPU parity tests: run the CUDA path through the binding,
run the oracle on the same bits, compare with the stated tolerances."""
from __future__ import annotations

import numpy as np
import torch

import oracle
from layout_agnostic_paged_gb300 import splash as S
from layout_agnostic_paged_gb300 import workloads as W

# Attention tolerances (bf16 inputs, fp32 accumulation): max-abs over every
# compared output element and relative L2 over the compared set; LSE max-abs.
OUT_MAX_ABS = 2e-2
OUT_REL_L2 = 5e-3
LSE_MAX_ABS = 1e-3


def gpu_decode(inp: W.DecodeInputs, scale: float, head_lo=0, head_hi=None, tok_lo=0, tok_hi=-1,
               out=None, lse=None, ws=None):
    B, H, _ = inp.q.shape
    head_hi = H if head_hi is None else head_hi
    dev = inp.q.device
    if out is None:
        out = torch.full((B, H, 512), float("nan"), dtype=torch.float32, device=dev)
    if lse is None:
        lse = torch.full((B, H), float("nan"), dtype=torch.float32, device=dev)
    if ws is None:
        ws = S.decode_workspace(inp.q, inp.pool, inp.block_table, scale, head_lo, head_hi)
    S.splash_decode_attn(inp.q, inp.pool, inp.block_table, inp.ctx_lens, head_lo, head_hi, tok_lo,
                         tok_hi, out, lse, ws, scale)
    return out, lse, ws


def oracle_full(inp: W.DecodeInputs, scale: float, **kw):
    return oracle.decode_attn(oracle.bf16_bits(inp.q), oracle.bf16_bits(inp.pool),
                              inp.block_table.cpu().numpy(), inp.ctx_lens.cpu().numpy(), scale, **kw)


def oracle_rows(inp: W.DecodeInputs, scale: float, r: int, head_lo: int, head_hi: int, tok_lo=0,
                tok_hi=-1):
    """Oracle for request r and heads [head_lo, head_hi): gathers only that request's
    pages into a compact host pool (a page permutation, which the oracle's pins
    show does not change the result)."""
    n = inp.pages_per_req[r]
    ids = inp.block_table[r, :n].long()
    pool = inp.pool.index_select(0, ids) if n else inp.pool[:1]
    bt = np.arange(max(n, 1), dtype=np.int32)[None, :]
    q = inp.q[r:r + 1, head_lo:head_hi]
    o, l = oracle.decode_attn(oracle.bf16_bits(q), oracle.bf16_bits(pool), bt,
                              inp.ctx_lens[r:r + 1].cpu().numpy(), scale, tok_lo=tok_lo,
                              tok_hi=tok_hi)
    return o[0], l[0]


def assert_attn_close(out, ref_out, lse, ref_lse, what=""):
    out = np.asarray(out, dtype=np.float64)
    lse = np.asarray(lse, dtype=np.float64)
    assert out.shape == ref_out.shape and lse.shape == ref_lse.shape
    assert np.isfinite(out).all(), f"{what}: non-finite output"
    err = np.abs(out - ref_out)
    mx = float(err.max()) if err.size else 0.0
    den = float(np.linalg.norm(ref_out))
    rel = float(np.linalg.norm(out - ref_out)) / den if den > 0 else float(np.linalg.norm(out))
    assert mx <= OUT_MAX_ABS, f"{what}: max-abs {mx:.3e} > {OUT_MAX_ABS}"
    assert rel <= OUT_REL_L2, f"{what}: rel-L2 {rel:.3e} > {OUT_REL_L2}"
    fin = np.isfinite(ref_lse)
    assert np.array_equal(np.isfinite(lse), fin), f"{what}: lse finiteness differs"
    assert np.array_equal(lse[~fin], ref_lse[~fin]), f"{what}: empty-set lse differs"
    if fin.any():
        lmx = float(np.abs(lse[fin] - ref_lse[fin]).max())
        assert lmx <= LSE_MAX_ABS, f"{what}: lse max-abs {lmx:.3e} > {LSE_MAX_ABS}"
    return mx, rel
