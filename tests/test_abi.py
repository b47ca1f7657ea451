"""The C-ABI library: it loads, exports every symbol include/splash.h declares, and
rejects bad arguments on the host before enqueuing anything (CPU only: no call
here reaches a kernel)."""
import ctypes
import glob
import os
import re
import subprocess

import pytest

from layout_agnostic_paged_gb300 import build as B
from layout_agnostic_paged_gb300 import splash as S

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    B.build()
    return S.load_library()


def declared_functions():
    names = []
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        names += re.findall(r"SPLASH_API\s+[\w\s\*]+?\b(splash_\w+)\s*\(", open(h).read())
    return sorted(set(names))


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ("splash_decode_attn", "splash_lse_merge", "splash_kv_migrate",
              "splash_decode_workspace_size", "splash_status_string"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    names = declared_functions()
    out = subprocess.run(["nm", "-D", "--defined-only", S.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r"\bT\s+(\w+)$", out, re.M))
    for n in names:
        assert n in exported, n
        assert hasattr(lib, n)
    assert set(S.EXPORTED) <= set(names)
    # nothing else with the public prefix leaks out
    assert {e for e in exported if e.startswith("splash_")} == set(names)


def test_status_strings(lib):
    for code in (0, -1, -2, -3, -4):
        assert S.splash_status_string(code).startswith("SPLASH_")
    assert "unknown" in S.splash_status_string(7)


def _desc(**kw):
    d = dict(num_reqs=2, num_heads=8, d_qk=576, d_v=512, page_size=16, num_pages=11,
             max_pages_per_req=7, scale=0.0721)
    d.update(kw)
    return S.SplashAttnDesc(**d)


FAKE = 0x10000  # never dereferenced: every call below fails host validation first


def _decode(lib, desc, head_lo=0, head_hi=8, tok_lo=0, tok_hi=-1, q=FAKE, ws=FAKE, ws_bytes=1 << 30,
            out=FAKE, pool=FAKE):
    vp = ctypes.c_void_p
    return lib.splash_decode_attn(ctypes.byref(desc), vp(q), vp(pool), vp(FAKE), vp(FAKE), head_lo,
                                  head_hi, tok_lo, tok_hi, vp(out), vp(FAKE), vp(ws), ws_bytes,
                                  vp(0))


@pytest.mark.parametrize("kw,code", [
    (dict(d_qk=512), S.SPLASH_ERR_UNSUPPORTED),
    (dict(d_v=576), S.SPLASH_ERR_UNSUPPORTED),
    (dict(page_size=48), S.SPLASH_ERR_UNSUPPORTED),
    (dict(page_size=256), S.SPLASH_ERR_UNSUPPORTED),
    (dict(num_heads=0), S.SPLASH_ERR_INVALID_ARG),
    (dict(num_reqs=-1), S.SPLASH_ERR_INVALID_ARG),
    (dict(scale=float("nan")), S.SPLASH_ERR_INVALID_ARG),
    (dict(num_pages=1 << 27, page_size=64), S.SPLASH_ERR_UNSUPPORTED),
])
def test_decode_rejects_bad_shapes(lib, kw, code):
    assert _decode(lib, _desc(**kw)) == code


@pytest.mark.parametrize("args", [
    dict(head_lo=3, head_hi=3), dict(head_lo=-1), dict(head_hi=9), dict(tok_lo=-5),
    dict(tok_lo=10, tok_hi=4), dict(ws=0), dict(ws=FAKE + 16), dict(q=FAKE + 2),
    dict(out=FAKE + 4), dict(q=0), dict(pool=FAKE + 8),
])
def test_decode_rejects_bad_arguments(lib, args):
    assert _decode(lib, _desc(), **args) == S.SPLASH_ERR_INVALID_ARG


def _decode_ex(lib, desc, ext, head_lo=0, head_hi=8, tok_lo=0, tok_hi=-1):
    vp = ctypes.c_void_p
    return lib.splash_decode_attn_ex(ctypes.byref(desc), ext, vp(FAKE), vp(FAKE), vp(FAKE),
                                     vp(FAKE), head_lo, head_hi, tok_lo, tok_hi, vp(FAKE),
                                     vp(FAKE), vp(FAKE), 1 << 30, vp(0))


@pytest.mark.parametrize("ext", [
    dict(rows=FAKE, num_rows=0), dict(rows=FAKE, num_rows=-3), dict(tok_lo=FAKE + 2),
    dict(tok_hi=FAKE + 1), dict(rows=FAKE + 2, num_rows=4), dict(max_sms=-1), dict(kv=-1),
    dict(kv=3),   # 8 query heads over 3 KV heads
])
def test_decode_ex_rejects_bad_extensions(lib, ext):
    e = S.SplashDecodeExt(ext.get("tok_lo"), ext.get("tok_hi"), ext.get("rows"),
                          ext.get("num_rows", 0), ext.get("max_sms", 0), ext.get("kv", 0))
    assert _decode_ex(lib, _desc(), ctypes.byref(e)) == S.SPLASH_ERR_INVALID_ARG


def test_decode_ex_rejects_unsupported_kv_head_groupings(lib):
    e = S.SplashDecodeExt(None, None, None, 0, 0, 2)
    # 8 query heads over 2 KV heads: groups of 4, so head_lo must be a multiple of 4
    assert _decode_ex(lib, _desc(), ctypes.byref(e), head_lo=2, head_hi=8) == S.SPLASH_ERR_UNSUPPORTED


def test_decode_ex_validates_like_decode_without_extension(lib):
    assert _decode_ex(lib, _desc(), None, head_lo=3, head_hi=3) == S.SPLASH_ERR_INVALID_ARG
    assert _decode_ex(lib, _desc(d_qk=512), None) == S.SPLASH_ERR_UNSUPPORTED


def test_workspace_size_is_zero_for_invalid_shapes(lib):
    assert lib.splash_decode_workspace_size(ctypes.byref(_desc(d_qk=128)), 0, 8) == 0
    assert lib.splash_decode_workspace_size(ctypes.byref(_desc()), 4, 2) == 0
    assert lib.splash_decode_workspace_size(None, 0, 8) == 0


def test_merge_rejects_bad_arguments(lib):
    vp = ctypes.c_void_p
    f = lib.splash_lse_merge
    assert f(vp(FAKE), vp(FAKE), 0, 2, 2, 512, vp(FAKE << 4), vp(FAKE), vp(0)) == S.SPLASH_ERR_INVALID_ARG
    assert f(vp(FAKE), vp(FAKE), 2, 2, 2, 6, vp(FAKE << 4), vp(FAKE), vp(0)) == S.SPLASH_ERR_INVALID_ARG
    assert f(vp(0), vp(FAKE), 2, 2, 2, 512, vp(FAKE << 4), vp(FAKE), vp(0)) == S.SPLASH_ERR_INVALID_ARG
    assert f(vp(FAKE + 4), vp(FAKE), 2, 2, 2, 512, vp(FAKE << 4), vp(FAKE), vp(0)) == S.SPLASH_ERR_INVALID_ARG
    # out overlapping part_out
    assert f(vp(FAKE), vp(FAKE), 2, 2, 2, 512, vp(FAKE + 1024), vp(FAKE), vp(0)) == S.SPLASH_ERR_INVALID_ARG
    # nothing to do is not an error
    assert f(vp(0), vp(0), 2, 0, 2, 512, vp(0), vp(0), vp(0)) == S.SPLASH_OK


def test_migrate_rejects_bad_arguments(lib):
    vp = ctypes.c_void_p
    f = lib.splash_kv_migrate
    assert f(vp(FAKE), vp(FAKE), 10, vp(FAKE), vp(FAKE), 3, 8, 8, vp(0)) == S.SPLASH_ERR_INVALID_ARG
    assert f(vp(FAKE), vp(FAKE), 0, vp(FAKE), vp(FAKE), 3, 8, 8, vp(0)) == S.SPLASH_ERR_INVALID_ARG
    assert f(vp(FAKE), vp(FAKE), 4096, vp(FAKE), vp(FAKE), -1, 8, 8, vp(0)) == S.SPLASH_ERR_INVALID_ARG
    assert f(vp(FAKE + 8), vp(FAKE), 4096, vp(FAKE), vp(FAKE), 3, 8, 8, vp(0)) == S.SPLASH_ERR_INVALID_ARG
    assert f(vp(0), vp(FAKE), 4096, vp(FAKE), vp(FAKE), 3, 8, 8, vp(0)) == S.SPLASH_ERR_INVALID_ARG
    assert f(vp(0), vp(0), 4096, vp(0), vp(0), 0, 8, 8, vp(0)) == S.SPLASH_OK


def test_status_reader_rejects_null(lib):
    flags = ctypes.c_uint32(0)
    assert lib.splash_workspace_status(None, ctypes.byref(flags), None) == S.SPLASH_ERR_INVALID_ARG
    assert lib.splash_workspace_status(ctypes.c_void_p(FAKE), None, None) == S.SPLASH_ERR_INVALID_ARG
    # the no-allocation entry point's status reader checks its output pointer first
    assert lib.splash_noalloc_status(None, None) == S.SPLASH_ERR_INVALID_ARG


def test_noalloc_rejects_invalid_shapes_before_touching_the_scratch(lib):
    vp = ctypes.c_void_p
    f = lib.splash_decode_attn_noalloc
    args = (vp(FAKE), vp(FAKE), vp(FAKE), vp(FAKE), 0, 8, 0, -1, vp(FAKE), vp(FAKE), vp(0))
    assert f(ctypes.byref(_desc(d_qk=512)), *args) == S.SPLASH_ERR_UNSUPPORTED
    assert f(ctypes.byref(_desc(num_heads=0)), *args) == S.SPLASH_ERR_INVALID_ARG


def test_binding_fails_loudly_without_cuda_tensors():
    import torch
    q = torch.zeros(1, 8, 576, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        S.splash_decode_attn(q, q, q, q, 0, 8, 0, -1, q, q, q, 0.1)
