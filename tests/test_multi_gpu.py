"""GPU parity of several new tokens per sequence (mqa_kv_append_multi, mqa_decode_attention_multi,
mqa_decode_step_multi) against the fp64 oracle on the same seeded inputs.

The oracle's side: oracle.kv_append_multi (token t at row pos + t) and oracle.decode_attention_multi
(token t attends the first seq_lens - T + 1 + t rows). Rows at or past each sequence's old context
hold NaN, so a row read past a token's causal limit would show. Caches are compared bit for bit,
outputs within the contract's tolerances.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from query_grouped_decode_kv_b300 import inputs
from tests import _parity as P

pytestmark = pytest.mark.gpu

BOUNDS = 4


@pytest.fixture(scope="module")
def mqa():
    import query_grouped_decode_kv_b300 as m
    m.debug_override(0, 0)
    yield m
    m.debug_override(0, 0)


def multi_case(b, T, h, g, d_h, ctx_lo, ctx_hi, seed_id, ctx=None):
    """ctx: the rows cached before this step (default: seeded lengths); the new tokens go to rows
    ctx .. ctx + T - 1, and n_max leaves room for them."""
    w = inputs.custom(f"multi{seed_id}", b, h, g, d_h, ctx_lo, ctx_hi + T - 1, wid=seed_id)
    c = inputs.context_lengths(w) if ctx is None else torch.tensor(ctx, dtype=torch.int32)
    c = torch.clamp(c, max=ctx_hi)
    k, v = inputs.cache(w, 0, "cpu", tail="nan", lengths=c)
    q, kn, vn = inputs.multi_step_inputs(w, T, 0, "cpu")
    return dict(w=w, T=T, q=q, k_new=kn, v_new=vn, k=k, v=v, pos=c.clone(),
                lens=(c + T).to(torch.int32), scale=w.scale)


def oracle_multi(case):
    kb, vb = P.bits(case["k"]).copy(), P.bits(case["v"]).copy()
    st = oracle.kv_append_multi(P.bits(case["k_new"]), P.bits(case["v_new"]), kb, vb,
                                case["pos"].numpy())
    out, ast = oracle.decode_attention_multi(P.bits(case["q"]), kb, vb, case["lens"].numpy(),
                                             case["scale"], return_status=True)
    return kb, vb, out, st, ast


def gpu_multi(case, mqa, fused=True):
    dev = torch.device("cuda")
    q = case["q"].to(dev)
    kn, vn = case["k_new"].to(dev), case["v_new"].to(dev)
    k, v = case["k"].to(dev), case["v"].to(dev)
    pos, lens = case["pos"].to(dev), case["lens"].to(dev)
    if fused:
        out = mqa.decode_step_multi(q, kn, vn, k, v, pos, lens, scale=case["scale"])
    else:
        mqa.kv_append_multi(kn, vn, k, v, pos)
        out = mqa.decode_attention_multi(q, k, v, lens, scale=case["scale"])
    return k, v, out


SHAPES = [
    # b, T, h, g, d_h, ctx_lo, ctx_hi
    (2, 2, 16, 2, 128, 100, 700),     # T=2, G=8: 16 rows
    (3, 4, 64, 8, 128, 0, 513),       # T=4, G=8 (the 70B-class grouping): 32 rows
    (2, 8, 64, 8, 128, 60, 300),      # T=8, G=8: 64 rows
    (2, 3, 8, 2, 128, 1, 200),        # T=3, G=4: 12 rows
    (2, 4, 4, 4, 128, 60, 70),        # T=4, MHA (G=1): 4 rows
    (2, 2, 32, 1, 128, 1, 1000),      # T=2, G=32: 64 rows
    (3, 5, 9, 3, 64, 10, 129),        # T=5, G=3, d_h=64: 15 rows
    (1, 16, 8, 2, 128, 0, 64),        # T=16, G=4: 64 rows, a prompt chunk from an empty cache
]


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "b{}T{}h{}g{}d{}_{}-{}".format(*s))
@pytest.mark.parametrize("fused", [True, False], ids=["fused", "two_launches"])
def test_multi_step_matches_oracle(mqa, shape, fused):
    case = multi_case(*shape, seed_id=1600 + SHAPES.index(shape))
    k_ref, v_ref, out_ref, st, ast = oracle_multi(case)
    assert st == oracle.OK and ast == oracle.OK
    k, v, out = gpu_multi(case, mqa, fused)
    torch.cuda.synchronize()
    assert mqa.get_device_status() == 0
    assert np.array_equal(P.bits(k), k_ref) and np.array_equal(P.bits(v), v_ref)
    P.assert_close(out, out_ref, f"T tokens {shape}")


@pytest.mark.parametrize("ctas", [1, 2, 3, 7, 64, 148, 1000])
@pytest.mark.parametrize("shape", [(2, 4, 32, 4, 128, 0, 700), (2, 2, 64, 2, 128, 60, 400)],
                         ids=["T4G8", "T2G32"])
def test_multi_any_cta_split(mqa, shape, ctas):
    # split pieces that hold only a sequence's last tile give the earlier tokens no key at all
    case = multi_case(*shape, seed_id=1620)
    k_ref, v_ref, out_ref, _, _ = oracle_multi(case)
    mqa.debug_override(ctas, 0)
    try:
        k, v, out = gpu_multi(case, mqa)
        assert mqa.get_device_status() == 0
    finally:
        mqa.debug_override(0, 0)
    assert np.array_equal(P.bits(k), k_ref) and np.array_equal(P.bits(v), v_ref)
    P.assert_close(out, out_ref, f"T tokens {shape} ctas={ctas}")


@pytest.mark.parametrize("ctas", [0, 1, 5])
def test_multi_rows_across_tile_edges(mqa, ctas):
    # the new rows start at 62 (cross tiles 0/1), 127 (1/2), 0 (empty cache), 64 (a tile start)
    case = multi_case(4, 4, 16, 2, 128, 0, 200, seed_id=1630, ctx=[62, 127, 0, 64])
    k_ref, v_ref, out_ref, st, _ = oracle_multi(case)
    assert st == oracle.OK
    mqa.debug_override(ctas, 0)
    try:
        k, v, out = gpu_multi(case, mqa)
        assert mqa.get_device_status() == 0
    finally:
        mqa.debug_override(0, 0)
    assert np.array_equal(P.bits(k), k_ref) and np.array_equal(P.bits(v), v_ref)
    P.assert_close(out, out_ref, f"tile edges ctas={ctas}")


def test_multi_with_one_token_equals_the_decode_step(mqa):
    case = multi_case(3, 1, 32, 4, 128, 50, 900, seed_id=1640)
    dev = torch.device("cuda")
    k1, v1 = case["k"].to(dev), case["v"].to(dev)
    k2, v2 = case["k"].to(dev), case["v"].to(dev)
    pos, lens = case["pos"].to(dev), case["lens"].to(dev)
    o1 = mqa.decode_step_multi(case["q"].to(dev), case["k_new"].to(dev), case["v_new"].to(dev),
                               k1, v1, pos, lens, scale=case["scale"])
    o2 = mqa.decode_step(case["q"][:, 0].contiguous().to(dev),
                         case["k_new"][:, 0].contiguous().to(dev),
                         case["v_new"][:, 0].contiguous().to(dev), k2, v2, pos, lens,
                         scale=case["scale"])
    torch.cuda.synchronize()
    assert mqa.get_device_status() == 0
    assert torch.equal(o1[:, 0].view(torch.int16), o2.view(torch.int16))
    assert torch.equal(k1.view(torch.int16), k2.view(torch.int16))


def test_multi_invalid_lengths_and_positions(mqa):
    # sequence 1: length below T (zeros, latched); sequence 2: rows past the cache (no append)
    case = multi_case(3, 4, 16, 2, 128, 20, 100, seed_id=1650)
    n_max = case["w"].n_max
    lens, pos = case["lens"].clone(), case["pos"].clone()
    lens[1] = 3
    pos[2] = n_max - 2
    case["lens"], case["pos"] = lens, pos
    k_ref, v_ref, out_ref, st, ast = oracle_multi(case)
    assert st == oracle.ERR_BOUNDS and ast == oracle.ERR_BOUNDS
    for fused in (True, False):
        k, v, out = gpu_multi(case, mqa, fused)
        assert mqa.get_device_status() == BOUNDS
        assert np.array_equal(P.bits(k), k_ref) and np.array_equal(P.bits(v), v_ref)
        assert np.all(P.bits(out)[1] == 0)
        P.assert_close(out[[0]], out_ref[[0]], f"valid sequence next to invalid ones, {fused}")
