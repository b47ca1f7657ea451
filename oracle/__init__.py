"""fp64 CPU oracle for paged MLA decode attention, LSE merge and KV-page migration.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference legs of ``bench.py`` may import this package.  The
product path (``layout_agnostic_paged_gb300``) never imports it and shares no
code with it; both sides only receive the same seeded inputs.

The arithmetic lives in ``splash_oracle.c`` (plain C, IEEE double, OpenMP over
(request, head)); this module compiles it with gcc and marshals numpy arrays.
Source for what is computed: "SPLASH: Switching Parallel Layouts of Attention
with Seamless Handoff for LLM Serving" -- Abstract (layouts differ only in who
owns weights and cache; a switch moves KV state and hands off at a batch
boundary) and Appendix, Table 2 (TP head shares, CP token shares, DP-attention /
DOP request ownership).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "splash_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libsplash_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (OpenMP, -O2, strict IEEE) and return the .so path."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-fno-fast-math", "-ffp-contract=off", "-fopenmp", "-fPIC",
           "-shared", "-std=c11", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _bind(lib):
    i32, i64, dbl, vp = ctypes.c_int, ctypes.c_int64, ctypes.c_double, ctypes.c_void_p
    lib.oracle_decode_attn.argtypes = [i32, i32, i32, i32, i32, i32, i32, dbl, vp, vp, vp, vp,
                                       i32, i32, i64, i64, vp, vp]
    lib.oracle_decode_attn.restype = i32
    lib.oracle_decode_attn_kv.argtypes = [i32, i32, i32, i32, i32, i32, i32, i32, dbl, vp, vp, vp,
                                          vp, i32, i32, i64, i64, vp, vp]
    lib.oracle_decode_attn_kv.restype = i32
    lib.oracle_lse_merge.argtypes = [i32, i64, i32, vp, vp, vp, vp]
    lib.oracle_lse_merge.restype = i32
    lib.oracle_kv_migrate.argtypes = [vp, vp, i64, vp, vp, i32, ctypes.c_int32, ctypes.c_int32]
    lib.oracle_kv_migrate.restype = i32
    lib.oracle_num_threads.argtypes = []
    lib.oracle_num_threads.restype = i32
    lib.oracle_set_num_threads.argtypes = [i32]
    lib.oracle_set_num_threads.restype = None
    return lib


def _load():
    global _lib
    with _lock:
        if _lib is None:
            _lib = _bind(ctypes.CDLL(build()))
        return _lib


class OracleLib:
    """The oracle's three operations bound to one compiled copy of the C source.

    The default instance uses the committed source; tests may compile a copy
    with a planted mistake and check that the pins catch it.
    """

    def __init__(self, so_path: str | None = None):
        self._so = _bind(ctypes.CDLL(so_path)) if so_path else None

    @property
    def lib(self):
        return self._so if self._so is not None else _load()

    def decode_attn(self, *a, **k):
        return decode_attn(*a, _lib=self.lib, **k)

    def lse_merge(self, *a, **k):
        return lse_merge(*a, _lib=self.lib, **k)

    def kv_migrate(self, *a, **k):
        return kv_migrate(*a, _lib=self.lib, **k)


def compile_variant(src_text: str, out_dir: str, name: str = "variant") -> str:
    """Compile C source text with the oracle's flags into out_dir; returns the .so path."""
    c_path = os.path.join(out_dir, name + ".c")
    so_path = os.path.join(out_dir, name + ".so")
    with open(c_path, "w") as f:
        f.write(src_text)
    subprocess.run(["gcc", "-O2", "-fno-fast-math", "-ffp-contract=off", "-fopenmp", "-fPIC",
                    "-shared", "-std=c11", c_path, "-o", so_path, "-lm"], check=True)
    return so_path


def source_text() -> str:
    with open(_SRC) as f:
        return f.read()


def _c(a: np.ndarray, dtype) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=dtype)


def _ptr(a: np.ndarray):
    return ctypes.c_void_p(a.ctypes.data)


def num_threads() -> int:
    """Threads the oracle uses (OMP_NUM_THREADS or all cores)."""
    return int(_load().oracle_num_threads())


def set_num_threads(n: int) -> None:
    _load().oracle_set_num_threads(int(n))


def bf16_bits(x) -> np.ndarray:
    """uint16 view of a bf16 tensor / array (the exact bits both sides read)."""
    if hasattr(x, "view") and hasattr(x, "dtype") and str(x.dtype) == "torch.bfloat16":
        import torch
        return x.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)
    a = np.asarray(x)
    if a.dtype != np.uint16:
        raise TypeError("expected bf16 bits as uint16")
    return a


def decode_attn(q_bits, pool_bits, block_table, ctx_lens, scale: float, head_lo: int = 0,
                head_hi: int | None = None, tok_lo: int = 0, tok_hi: int = -1,
                out: np.ndarray | None = None, lse: np.ndarray | None = None, _lib=None):
    """fp64 paged decode attention of one ownership slice.

    q_bits uint16 [B][H][d_qk], pool_bits uint16 [num_pages][P][d_qk] (bf16 bits;
    one shared KV head) or [num_pages][Hkv][P][d_qk] (Hkv KV heads, query head h
    reading KV head h / (H / Hkv)), block_table int32 [B][max_pages], ctx_lens int32
    [B].  Returns (out, lse) as float64 [B][H][d_v] / [B][H] with d_v = 512 (the
    latent prefix of the key); rows outside [head_lo, head_hi) are left as given
    (NaN when freshly made).
    """
    q = _c(q_bits, np.uint16)
    pool = _c(pool_bits, np.uint16)
    bt = _c(block_table, np.int32)
    cl = _c(ctx_lens, np.int32)
    B, H, d_qk = q.shape
    if pool.ndim == 4:
        num_pages, Hkv, P, d_qk2 = pool.shape
    else:
        (num_pages, P, d_qk2), Hkv = pool.shape, 0
    assert d_qk2 == d_qk
    d_v = 512 if d_qk == 576 else d_qk
    if head_hi is None:
        head_hi = H
    if out is None:
        out = np.full((B, H, d_v), np.nan, dtype=np.float64)
    if lse is None:
        lse = np.full((B, H), np.nan, dtype=np.float64)
    assert out.dtype == np.float64 and out.flags.c_contiguous
    assert lse.dtype == np.float64 and lse.flags.c_contiguous
    max_pages = bt.shape[1] if bt.ndim == 2 else 0
    lib = _lib or _load()
    if Hkv:
        rc = lib.oracle_decode_attn_kv(B, H, Hkv, d_qk, d_v, P, num_pages, max_pages, float(scale),
                                       _ptr(q), _ptr(pool), _ptr(bt), _ptr(cl), int(head_lo),
                                       int(head_hi), int(tok_lo), int(tok_hi), _ptr(out), _ptr(lse))
    else:
        rc = lib.oracle_decode_attn(B, H, d_qk, d_v, P, num_pages, max_pages, float(scale),
                                    _ptr(q), _ptr(pool), _ptr(bt), _ptr(cl), int(head_lo),
                                    int(head_hi), int(tok_lo), int(tok_hi), _ptr(out), _ptr(lse))
    if rc != 0:
        raise ValueError(f"oracle_decode_attn rejected its arguments (status {rc})")
    return out, lse


def lse_merge(part_out: np.ndarray, part_lse: np.ndarray, _lib=None):
    """Merge S partials: part_out [S][..rows..][d_v], part_lse [S][..rows..] -> (out, lse)."""
    po = _c(part_out, np.float64)
    pl = _c(part_lse, np.float64)
    S = po.shape[0]
    d_v = po.shape[-1]
    rows_shape = po.shape[1:-1]
    R = int(np.prod(rows_shape)) if rows_shape else 1
    assert pl.shape == (S,) + rows_shape
    out = np.empty(rows_shape + (d_v,), dtype=np.float64)
    lse = np.empty(rows_shape, dtype=np.float64)
    rc = (_lib or _load()).oracle_lse_merge(S, R, d_v, _ptr(po), _ptr(pl), _ptr(out), _ptr(lse))
    if rc != 0:
        raise ValueError(f"oracle_lse_merge rejected its arguments (status {rc})")
    return out, lse


def kv_migrate(src_pool: np.ndarray, dst_pool: np.ndarray, src_ids, dst_ids, _lib=None
               ) -> np.ndarray:
    """Copy pages src_pool[src_ids[i]] -> dst_pool[dst_ids[i]] in place; returns dst_pool."""
    assert src_pool.flags.c_contiguous and dst_pool.flags.c_contiguous
    page_bytes = src_pool[0].nbytes if src_pool.shape[0] else dst_pool[0].nbytes
    assert dst_pool[0].nbytes == page_bytes
    s = _c(src_ids, np.int32)
    d = _c(dst_ids, np.int32)
    assert s.shape == d.shape
    rc = (_lib or _load()).oracle_kv_migrate(_ptr(src_pool), _ptr(dst_pool), page_bytes, _ptr(s), _ptr(d),
                                   int(s.shape[0]), int(src_pool.shape[0]), int(dst_pool.shape[0]))
    if rc != 0:
        raise ValueError("oracle_kv_migrate: page id out of range")
    return dst_pool
