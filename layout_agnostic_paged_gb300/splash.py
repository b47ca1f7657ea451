"""Thin Python binding of the C ABI in include/splash.h (argument marshalling only).

Every function here forwards torch tensors' device pointers, sizes and the
current CUDA stream to ``libsplash_gb300.so``; every step of the computation
runs in that library's CUDA kernels.  There is no fallback: if the library is
missing or the tensors are not on a CUDA device the call raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "_build", "libsplash_gb300.so")

SPLASH_OK = 0
SPLASH_ERR_INVALID_ARG = -1
SPLASH_ERR_UNSUPPORTED = -2
SPLASH_ERR_WORKSPACE = -3
SPLASH_ERR_CUDA = -4
SPLASH_DEVICE_TIMEOUT = 1
SPLASH_DEVICE_BAD_INPUT = 2

EXPORTED = ("splash_decode_workspace_size", "splash_decode_attn", "splash_decode_attn_ex",
            "splash_decode_attn_noalloc", "splash_noalloc_status",
            "splash_lse_merge", "splash_kv_migrate", "splash_workspace_status",
            "splash_status_string")


class SplashError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {splash_status_string(code)} ({code})")


class SplashAttnDesc(ctypes.Structure):
    _fields_ = [("num_reqs", ctypes.c_int32), ("num_heads", ctypes.c_int32),
                ("d_qk", ctypes.c_int32), ("d_v", ctypes.c_int32), ("page_size", ctypes.c_int32),
                ("num_pages", ctypes.c_int32), ("max_pages_per_req", ctypes.c_int32),
                ("scale", ctypes.c_float)]


class SplashDecodeExt(ctypes.Structure):
    _fields_ = [("tok_lo", ctypes.c_void_p), ("tok_hi", ctypes.c_void_p),
                ("rows", ctypes.c_void_p), ("num_rows", ctypes.c_int32),
                ("max_sms", ctypes.c_int32), ("num_kv_heads", ctypes.c_int32)]


_lock = threading.Lock()
_lib = None


def load_library(path: str | None = None):
    """Loads (once) and returns the ctypes handle; raises if the library is missing."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        p = path or LIB_PATH
        if not os.path.exists(p):
            raise RuntimeError(f"{p} is missing: build it with layout_agnostic_paged_gb300.build.build()")
        lib = ctypes.CDLL(p)
        vp, i32, i64, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t
        dp = ctypes.POINTER(SplashAttnDesc)
        lib.splash_decode_workspace_size.argtypes = [dp, i32, i32]
        lib.splash_decode_workspace_size.restype = sz
        lib.splash_decode_attn.argtypes = [dp, vp, vp, vp, vp, i32, i32, i64, i64, vp, vp, vp, sz, vp]
        lib.splash_decode_attn.restype = i32
        lib.splash_decode_attn_ex.argtypes = [dp, ctypes.POINTER(SplashDecodeExt), vp, vp, vp, vp,
                                              i32, i32, i64, i64, vp, vp, vp, sz, vp]
        lib.splash_decode_attn_ex.restype = i32
        lib.splash_decode_attn_noalloc.argtypes = [dp, vp, vp, vp, vp, i32, i32, i64, i64, vp, vp, vp]
        lib.splash_decode_attn_noalloc.restype = i32
        lib.splash_noalloc_status.argtypes = [ctypes.POINTER(ctypes.c_uint32), vp]
        lib.splash_noalloc_status.restype = i32
        lib.splash_lse_merge.argtypes = [vp, vp, i32, i32, i32, i32, vp, vp, vp]
        lib.splash_lse_merge.restype = i32
        lib.splash_kv_migrate.argtypes = [vp, vp, sz, vp, vp, i32, ctypes.c_int32, ctypes.c_int32, vp]
        lib.splash_kv_migrate.restype = i32
        lib.splash_workspace_status.argtypes = [vp, ctypes.POINTER(ctypes.c_uint32), vp]
        lib.splash_workspace_status.restype = i32
        lib.splash_status_string.argtypes = [i32]
        lib.splash_status_string.restype = ctypes.c_char_p
        _lib = lib
        return lib


def splash_status_string(code: int) -> str:
    return load_library().splash_status_string(int(code)).decode()


def _ptr(t: torch.Tensor | None):
    return ctypes.c_void_p(0 if t is None else t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(int(stream.cuda_stream) if hasattr(stream, "cuda_stream") else int(stream))


def _check_cuda(*ts):
    for t in ts:
        if not t.is_cuda:
            raise ValueError("splash: tensors must live on a CUDA device")
        if not t.is_contiguous():
            raise ValueError("splash: tensors must be contiguous")


def make_desc(q: torch.Tensor, kv_pool: torch.Tensor, block_table: torch.Tensor,
              scale: float) -> SplashAttnDesc:
    B, H, d_qk = q.shape
    if kv_pool.dim() == 4:   # [num_pages][Hkv][P][576]: several KV heads
        num_pages, _, P, d_qk2 = kv_pool.shape
    else:
        num_pages, P, d_qk2 = kv_pool.shape
    if d_qk2 != d_qk:
        raise ValueError("q and kv_pool disagree on the key width")
    return SplashAttnDesc(B, H, d_qk, 512, P, num_pages, block_table.shape[1], float(scale))


def splash_decode_workspace_size(desc: SplashAttnDesc, head_lo: int, head_hi: int) -> int:
    return int(load_library().splash_decode_workspace_size(ctypes.byref(desc), int(head_lo),
                                                           int(head_hi)))


def decode_workspace(q, kv_pool, block_table, scale, head_lo=0, head_hi=None,
                     num_reqs=None) -> torch.Tensor:
    """Allocates (with torch, on q's device) a workspace large enough for the slice
    (num_reqs: requests in the call, when they are a subset of q's rows)."""
    desc = make_desc(q, kv_pool, block_table, scale)
    if num_reqs is not None:
        desc.num_reqs = int(num_reqs)
    head_hi = q.shape[1] if head_hi is None else head_hi
    with torch.cuda.device(q.device):
        n = splash_decode_workspace_size(desc, head_lo, head_hi)
    if n == 0:
        raise SplashError(SPLASH_ERR_UNSUPPORTED, "splash_decode_workspace_size")
    return torch.empty(n, dtype=torch.uint8, device=q.device)


def splash_decode_attn(q: torch.Tensor, kv_pool: torch.Tensor, block_table: torch.Tensor,
                       ctx_lens: torch.Tensor, head_lo: int, head_hi: int, tok_lo: int,
                       tok_hi: int, out: torch.Tensor, lse: torch.Tensor,
                       workspace: torch.Tensor, scale: float, stream=None) -> None:
    """Paged decode attention of one ownership slice (see splash.h); writes out / lse rows."""
    _check_cuda(q, kv_pool, block_table, ctx_lens, out, lse, workspace)
    if kv_pool.dim() != 3:
        raise ValueError("splash_decode_attn: one shared KV head [num_pages][P][576]; "
                         "use splash_decode_attn_ex for several KV heads")
    if (q.dtype != torch.bfloat16 or kv_pool.dtype != torch.bfloat16 or out.dtype != torch.float32
            or lse.dtype != torch.float32 or block_table.dtype != torch.int32
            or ctx_lens.dtype != torch.int32):
        raise ValueError("splash_decode_attn: dtype mismatch")
    B, H, _ = q.shape
    if out.shape != (B, H, 512) or lse.shape != (B, H) or ctx_lens.shape != (B,):
        raise ValueError("splash_decode_attn: shape mismatch")
    desc = make_desc(q, kv_pool, block_table, scale)
    with torch.cuda.device(q.device):
        rc = load_library().splash_decode_attn(
            ctypes.byref(desc), _ptr(q), _ptr(kv_pool), _ptr(block_table), _ptr(ctx_lens),
            int(head_lo), int(head_hi), int(tok_lo), int(tok_hi), _ptr(out), _ptr(lse),
            _ptr(workspace), workspace.numel() * workspace.element_size(), _stream(stream))
    if rc != SPLASH_OK:
        raise SplashError(rc, "splash_decode_attn")


def splash_decode_attn_ex(q: torch.Tensor, kv_pool: torch.Tensor, block_table: torch.Tensor,
                          ctx_lens: torch.Tensor, head_lo: int, head_hi: int, tok_lo: int,
                          tok_hi: int, out: torch.Tensor, lse: torch.Tensor,
                          workspace: torch.Tensor, scale: float, tok_lo_r=None, tok_hi_r=None,
                          rows=None, max_sms: int = 0, stream=None) -> None:
    """splash_decode_attn with optional per-request token ranges (int32 [B] tensors
    tok_lo_r / tok_hi_r), storage rows (int32 [B] tensor `rows` into q, block_table,
    ctx_lens, out and lse; B is len(rows) when rows is given, else q's rows) and an SM
    budget for the decode grid (max_sms, 0 = all).  A kv_pool of shape
    [num_pages][Hkv][P][576] selects grouped-query attention over Hkv KV heads."""
    opt = [t for t in (tok_lo_r, tok_hi_r, rows) if t is not None]
    _check_cuda(q, kv_pool, block_table, ctx_lens, out, lse, workspace, *opt)
    if (q.dtype != torch.bfloat16 or kv_pool.dtype != torch.bfloat16 or out.dtype != torch.float32
            or lse.dtype != torch.float32 or block_table.dtype != torch.int32
            or ctx_lens.dtype != torch.int32 or any(t.dtype != torch.int32 for t in opt)):
        raise ValueError("splash_decode_attn_ex: dtype mismatch")
    R, H, _ = q.shape
    if out.shape != (R, H, 512) or lse.shape != (R, H) or ctx_lens.shape != (R,):
        raise ValueError("splash_decode_attn_ex: shape mismatch")
    B = int(rows.numel()) if rows is not None else R
    if any(t.shape != (B,) for t in opt):
        raise ValueError("splash_decode_attn_ex: per-request arrays must have one entry per request")
    desc = make_desc(q, kv_pool, block_table, scale)
    desc.num_reqs = B
    ext = SplashDecodeExt(tok_lo_r.data_ptr() if tok_lo_r is not None else None,
                          tok_hi_r.data_ptr() if tok_hi_r is not None else None,
                          rows.data_ptr() if rows is not None else None,
                          R if rows is not None else 0, int(max_sms),
                          int(kv_pool.shape[1]) if kv_pool.dim() == 4 else 0)
    with torch.cuda.device(q.device):
        rc = load_library().splash_decode_attn_ex(
            ctypes.byref(desc), ctypes.byref(ext), _ptr(q), _ptr(kv_pool), _ptr(block_table),
            _ptr(ctx_lens), int(head_lo), int(head_hi), int(tok_lo), int(tok_hi), _ptr(out),
            _ptr(lse), _ptr(workspace), workspace.numel() * workspace.element_size(),
            _stream(stream))
    if rc != SPLASH_OK:
        raise SplashError(rc, "splash_decode_attn_ex")


def splash_decode_attn_noalloc(q: torch.Tensor, kv_pool: torch.Tensor, block_table: torch.Tensor,
                               ctx_lens: torch.Tensor, head_lo: int, head_hi: int, tok_lo: int,
                               tok_hi: int, out: torch.Tensor, lse: torch.Tensor, scale: float,
                               stream=None) -> None:
    """splash_decode_attn with the library's own fixed scratch instead of a caller
    workspace (for callers that cannot allocate device memory where they decode,
    e.g. under stream capture); see splash.h for its size limit and sharing rules."""
    _check_cuda(q, kv_pool, block_table, ctx_lens, out, lse)
    if (q.dtype != torch.bfloat16 or kv_pool.dtype != torch.bfloat16 or out.dtype != torch.float32
            or lse.dtype != torch.float32 or block_table.dtype != torch.int32
            or ctx_lens.dtype != torch.int32):
        raise ValueError("splash_decode_attn_noalloc: dtype mismatch")
    B, H, _ = q.shape
    if out.shape != (B, H, 512) or lse.shape != (B, H) or ctx_lens.shape != (B,):
        raise ValueError("splash_decode_attn_noalloc: shape mismatch")
    desc = make_desc(q, kv_pool, block_table, scale)
    with torch.cuda.device(q.device):
        rc = load_library().splash_decode_attn_noalloc(
            ctypes.byref(desc), _ptr(q), _ptr(kv_pool), _ptr(block_table), _ptr(ctx_lens),
            int(head_lo), int(head_hi), int(tok_lo), int(tok_hi), _ptr(out), _ptr(lse),
            _stream(stream))
    if rc != SPLASH_OK:
        raise SplashError(rc, "splash_decode_attn_noalloc")


def splash_noalloc_status(device=None, stream=None) -> int:
    """Synchronises the stream and returns the SPLASH_DEVICE_* bits of the last
    splash_decode_attn_noalloc call on the device."""
    flags = ctypes.c_uint32(0)
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    with torch.cuda.device(dev):
        rc = load_library().splash_noalloc_status(ctypes.byref(flags), _stream(stream))
    if rc != SPLASH_OK:
        raise SplashError(rc, "splash_noalloc_status")
    return int(flags.value)


def splash_lse_merge(part_out: torch.Tensor, part_lse: torch.Tensor, out: torch.Tensor,
                     lse: torch.Tensor, stream=None) -> None:
    """part_out [S][B][H][d_v], part_lse [S][B][H] -> out [B][H][d_v], lse [B][H]."""
    _check_cuda(part_out, part_lse, out, lse)
    S, B, H, d_v = part_out.shape
    if part_lse.shape != (S, B, H) or out.shape != (B, H, d_v) or lse.shape != (B, H):
        raise ValueError("splash_lse_merge: shape mismatch")
    if any(t.dtype != torch.float32 for t in (part_out, part_lse, out, lse)):
        raise ValueError("splash_lse_merge: tensors must be float32")
    with torch.cuda.device(out.device):
        rc = load_library().splash_lse_merge(_ptr(part_out), _ptr(part_lse), S, B, H, d_v, _ptr(out),
                                             _ptr(lse), _stream(stream))
    if rc != SPLASH_OK:
        raise SplashError(rc, "splash_lse_merge")


def splash_kv_migrate(src_pool: torch.Tensor, dst_pool: torch.Tensor, src_ids: torch.Tensor,
                      dst_ids: torch.Tensor, stream=None) -> None:
    """dst_pool[dst_ids[i]] <- src_pool[src_ids[i]] byte for byte (pages = leading dim)."""
    _check_cuda(src_pool, dst_pool, src_ids, dst_ids)
    if src_ids.dtype != torch.int32 or dst_ids.dtype != torch.int32 or src_ids.shape != dst_ids.shape:
        raise ValueError("splash_kv_migrate: ids must be int32 of equal length")
    page_bytes = src_pool[0].numel() * src_pool.element_size() if src_pool.shape[0] else 0
    if dst_pool.shape[0] and dst_pool[0].numel() * dst_pool.element_size() != page_bytes:
        raise ValueError("splash_kv_migrate: pools disagree on the page size")
    with torch.cuda.device(dst_pool.device):
        rc = load_library().splash_kv_migrate(_ptr(src_pool), _ptr(dst_pool), page_bytes,
                                              _ptr(src_ids), _ptr(dst_ids), src_ids.numel(),
                                              src_pool.shape[0], dst_pool.shape[0], _stream(stream))
    if rc != SPLASH_OK:
        raise SplashError(rc, "splash_kv_migrate")


def splash_workspace_status(workspace: torch.Tensor, stream=None) -> int:
    """Synchronises the stream and returns the SPLASH_DEVICE_* bits of the last decode call."""
    flags = ctypes.c_uint32(0)
    with torch.cuda.device(workspace.device):
        rc = load_library().splash_workspace_status(_ptr(workspace), ctypes.byref(flags),
                                                    _stream(stream))
    if rc != SPLASH_OK:
        raise SplashError(rc, "splash_workspace_status")
    return int(flags.value)
