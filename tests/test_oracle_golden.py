"""Oracle against the hand-derived closed-form fixtures in tests/golden/ (CPU only).

Each fixture states its citation and derivation; expected values are written as
closed-form expressions and evaluated here, never produced by any implementation.
"""
import glob
import json
import math
import os

import numpy as np
import pytest

import oracle
from tests.oracle_cases import D_QK, D_V, paged, to_bf16_bits

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
ENV = {"e": math.e, "log": math.log, "exp": math.exp, "sqrt": math.sqrt}


def _val(expr):
    return float(eval(str(expr), {"__builtins__": {}}, ENV))


def _dense(sparse, width):
    row = np.zeros(width, np.float32)
    for k, v in sparse.items():
        row[int(k)] = v
    return row


def _expect_row(spec, width):
    default = _val(spec.get("*", "nan"))
    row = np.full(width, default)
    for k, v in spec.items():
        if k != "*":
            row[int(k)] = _val(v)
    return row


ATTN = [p for p in sorted(glob.glob(os.path.join(GOLDEN, "*.json")))
        if "tokens" in json.load(open(p))]


@pytest.mark.parametrize("path", ATTN, ids=[os.path.basename(p) for p in ATTN])
def test_attention_fixture(path):
    fx = json.load(open(path))
    assert fx["citation"] and fx["derivation"]
    toks = [np.stack([_dense(t, D_QK) for t in req]) for req in fx["tokens"]]
    q = np.stack([_dense(r, D_QK) for r in fx["q"]])[:, None, :]
    pool, bt, ctx = paged(toks, fx["page_size"], fx.get("page_ids"))
    out, lse = oracle.decode_attn(to_bf16_bits(q), pool, bt, ctx, fx["scale"])
    for r in range(len(toks)):
        np.testing.assert_allclose(out[r, 0], _expect_row(fx["expect_out"][r], D_V), rtol=0,
                                   atol=1e-14)
        assert abs(lse[r, 0] - _val(fx["expect_lse"][r])) <= 1e-14


def test_merge_fixture():
    fx = json.load(open(os.path.join(GOLDEN, "lse_merge_weights.json")))
    assert fx["citation"] and fx["derivation"]
    po = np.stack([np.full((1, D_V), _val(v)) for v in fx["parts_out"]])
    pl = np.array([[_val(v)] for v in fx["parts_lse"]])
    out, lse = oracle.lse_merge(po, pl)
    np.testing.assert_allclose(out, np.full((1, D_V), _val(fx["expect_out"])), rtol=0, atol=1e-14)
    assert abs(lse[0] - _val(fx["expect_lse"])) <= 1e-14
