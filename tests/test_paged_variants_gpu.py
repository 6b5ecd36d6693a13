"""GPU parity of the paged calls combined with fp8 codes or with several new tokens
(mqa_*_paged_fp8, mqa_*_paged_multi) against the fp64 oracle, on the same seeded inputs.

The oracle's side: the append through the page table (oracle.kv_append_paged_fp8 /
oracle.kv_append_paged_multi), the gather of the rows the table maps (oracle.gather_pages_u8 /
oracle.gather_pages) and the attention over them (oracle.decode_attention_fp8 over the dequantized
codes / oracle.decode_attention_multi with its causal mask). Pools are compared byte for byte,
spare pages of NaN codes or NaN values included; outputs within the contract's tolerances. The same
rows laid out contiguously must give the same outputs bit for bit (the paged producer lands every
page's rows where a whole tile's copy would).
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from query_grouped_decode_kv_b300 import inputs
from tests import _parity as P
from tests.test_fp8_gpu import fp8_case
from tests.test_multi_gpu import multi_case

pytestmark = pytest.mark.gpu

BOUNDS, UNSUPPORTED = 4, 2


@pytest.fixture(scope="module")
def mqa():
    import query_grouped_decode_kv_b300 as m
    m.debug_override(0, 0)
    yield m
    m.debug_override(0, 0)


def _page(case, k, v, rows, page_size, seed):
    kp, vp, table = inputs.page_pool(k, v, rows, page_size, seed=seed, spare_pages=3)
    case.update(k_pool=kp, v_pool=vp, table=table, page_size=page_size)
    return case


# ---- fp8 codes in pages -------------------------------------------------------------------------
FP8_SHAPES = [
    # b, h, g, d_h, ctx_lo, ctx_hi
    (2, 4, 4, 128, 60, 70),       # G = 1 (MHA), around the tile edge
    (3, 8, 4, 128, 0, 300),       # G = 2, lengths from 1
    (2, 16, 2, 128, 100, 700),    # G = 8
    (2, 32, 1, 128, 1, 1000),     # G = 32, eight consumer warps
]


@pytest.mark.parametrize("page_size", [8, 16, 64])
@pytest.mark.parametrize("shape", FP8_SHAPES, ids=lambda s: "b{}h{}g{}d{}_{}-{}".format(*s))
@pytest.mark.parametrize("fused", [True, False], ids=["fused", "two_launches"])
def test_paged_fp8_step_matches_the_oracle(mqa, shape, page_size, fused):
    case = fp8_case(shape, seed_id=1700 + page_size)
    rows = torch.maximum(case["lens"], case["pos"] + 1)
    _page(case, case["k8"], case["v8"], rows, page_size, seed=1701 + page_size)
    ks, vs = case["k_scale"], case["v_scale"]
    # oracle: the quantized append through the table, the gather, the attention
    kp, vp = case["k_pool"].numpy().copy(), case["v_pool"].numpy().copy()
    tb = case["table"].numpy()
    assert oracle.kv_append_paged_fp8(P.bits(case["k_new"]), P.bits(case["v_new"]), kp, vp,
                                      case["pos"].numpy(), tb, ks, vs) == oracle.OK
    kc, _ = oracle.gather_pages_u8(kp, tb, page_size)
    vc, _ = oracle.gather_pages_u8(vp, tb, page_size)
    ref = oracle.decode_attention_fp8(P.bits(case["q"]), kc, vc, case["lens"].numpy(), ks, vs,
                                      case["scale"])
    # GPU
    dev = torch.device("cuda")
    q, kn, vn = case["q"].to(dev), case["k_new"].to(dev), case["v_new"].to(dev)
    kpd, vpd = case["k_pool"].to(dev), case["v_pool"].to(dev)
    pos, lens, table = case["pos"].to(dev), case["lens"].to(dev), case["table"].to(dev)
    if fused:
        out = mqa.decode_step_paged_fp8(q, kn, vn, kpd, vpd, pos, table, lens, ks, vs,
                                        scale=case["scale"])
    else:
        mqa.kv_append_paged_fp8(kn, vn, kpd, vpd, pos, table, ks, vs)
        out = mqa.decode_attention_paged_fp8(q, kpd, vpd, table, lens, ks, vs,
                                             scale=case["scale"])
    torch.cuda.synchronize()
    assert mqa.get_device_status() == 0
    assert np.array_equal(kpd.cpu().numpy(), kp) and np.array_equal(vpd.cpu().numpy(), vp)
    P.assert_close(out, ref, f"paged fp8 {shape} page {page_size}")
    # the same codes laid out contiguously give the same bits
    kc8, vc8 = case["k8"].to(dev), case["v8"].to(dev)
    out_c = mqa.decode_step_fp8(q, kn, vn, kc8, vc8, pos, lens, ks, vs, scale=case["scale"])
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), out_c.view(torch.int16))


@pytest.mark.parametrize("ctas", [1, 3, 148, 1000])
@pytest.mark.parametrize("page_size", [8, 16])
def test_paged_fp8_any_cta_split_equals_contiguous(mqa, page_size, ctas):
    """Two producer warps share a CTA's tiles over paged caches (alternate tiles, each with its
    own page lookups): one CTA walks every tile, 1000 CTAs leave most with one tile or none.
    The same split over the same codes laid out contiguously gives the same bits."""
    case = fp8_case((3, 16, 2, 128, 1, 1500), seed_id=1740 + page_size)
    rows = torch.maximum(case["lens"], case["pos"] + 1)
    _page(case, case["k8"], case["v8"], rows, page_size, seed=1741 + page_size)
    dev = torch.device("cuda")
    q, kn, vn = case["q"].to(dev), case["k_new"].to(dev), case["v_new"].to(dev)
    pos, lens, table = case["pos"].to(dev), case["lens"].to(dev), case["table"].to(dev)
    ks, vs = case["k_scale"], case["v_scale"]
    mqa.debug_override(ctas, 0)
    try:
        kpd, vpd = case["k_pool"].to(dev), case["v_pool"].to(dev)
        out = mqa.decode_step_paged_fp8(q, kn, vn, kpd, vpd, pos, table, lens, ks, vs,
                                        scale=case["scale"])
        kc8, vc8 = case["k8"].to(dev), case["v8"].to(dev)
        out_c = mqa.decode_step_fp8(q, kn, vn, kc8, vc8, pos, lens, ks, vs, scale=case["scale"])
        torch.cuda.synchronize()
    finally:
        mqa.debug_override(0, 0)
    assert mqa.get_device_status() == 0
    assert torch.equal(out.view(torch.int16), out_c.view(torch.int16))
    # the appended rows landed in the pools where the table maps them
    kp, vp = case["k_pool"].numpy().copy(), case["v_pool"].numpy().copy()
    assert oracle.kv_append_paged_fp8(P.bits(case["k_new"]), P.bits(case["v_new"]), kp, vp,
                                      case["pos"].numpy(), case["table"].numpy(), ks,
                                      vs) == oracle.OK
    assert np.array_equal(kpd.cpu().numpy(), kp) and np.array_equal(vpd.cpu().numpy(), vp)


def test_paged_fp8_bad_page_latches_and_skips_the_append(mqa):
    case = fp8_case((3, 16, 2, 128, 100, 400), seed_id=1720)
    rows = torch.maximum(case["lens"], case["pos"] + 1)
    _page(case, case["k8"], case["v8"], rows, 16, seed=1721)
    bad = case["table"].clone()
    bad[1, int(case["pos"][1]) // 16] = 10 ** 6   # the page holding sequence 1's new row
    dev = torch.device("cuda")
    kpd, vpd = case["k_pool"].to(dev), case["v_pool"].to(dev)
    mqa.kv_append_paged_fp8(case["k_new"].to(dev), case["v_new"].to(dev), kpd, vpd,
                            case["pos"].to(dev), bad.to(dev), case["k_scale"], case["v_scale"])
    torch.cuda.synchronize()
    assert mqa.get_device_status() == BOUNDS
    kp, vp = case["k_pool"].numpy().copy(), case["v_pool"].numpy().copy()
    assert oracle.kv_append_paged_fp8(P.bits(case["k_new"]), P.bits(case["v_new"]), kp, vp,
                                      case["pos"].numpy(), bad.numpy(), case["k_scale"],
                                      case["v_scale"]) == oracle.ERR_BOUNDS
    assert np.array_equal(kpd.cpu().numpy(), kp) and np.array_equal(vpd.cpu().numpy(), vp)


# ---- several tokens in pages --------------------------------------------------------------------
MULTI_SHAPES = [
    # b, T, h, g, d_h, ctx_lo, ctx_hi
    (2, 2, 16, 2, 128, 100, 700),     # T = 2, G = 8
    (3, 4, 64, 8, 128, 0, 513),       # T = 4, G = 8 (the 70B-class grouping)
    (2, 8, 64, 8, 128, 60, 300),      # T = 8, G = 8: 64 rows
    (2, 3, 8, 2, 128, 1, 200),        # T = 3, G = 4
    (3, 5, 9, 3, 64, 10, 129),        # T = 5, G = 3, d_h = 64
]


@pytest.mark.parametrize("page_size", [8, 16, 64])
@pytest.mark.parametrize("shape", MULTI_SHAPES,
                         ids=lambda s: "b{}T{}h{}g{}d{}_{}-{}".format(*s))
@pytest.mark.parametrize("fused", [True, False], ids=["fused", "two_launches"])
def test_paged_multi_step_matches_the_oracle(mqa, shape, page_size, fused):
    case = multi_case(*shape, seed_id=1800 + page_size)
    _page(case, case["k"], case["v"], case["lens"], page_size, seed=1801 + page_size)
    kp, vp = P.bits(case["k_pool"]).copy(), P.bits(case["v_pool"]).copy()
    tb = case["table"].numpy()
    assert oracle.kv_append_paged_multi(P.bits(case["k_new"]), P.bits(case["v_new"]), kp, vp,
                                        case["pos"].numpy(), tb) == oracle.OK
    kc, _ = oracle.gather_pages(kp, tb, page_size)
    vc, _ = oracle.gather_pages(vp, tb, page_size)
    ref = oracle.decode_attention_multi(P.bits(case["q"]), kc, vc, case["lens"].numpy(),
                                        case["scale"])
    dev = torch.device("cuda")
    q, kn, vn = case["q"].to(dev), case["k_new"].to(dev), case["v_new"].to(dev)
    kpd, vpd = case["k_pool"].to(dev), case["v_pool"].to(dev)
    pos, lens, table = case["pos"].to(dev), case["lens"].to(dev), case["table"].to(dev)
    if fused:
        out = mqa.decode_step_paged_multi(q, kn, vn, kpd, vpd, pos, table, lens,
                                          scale=case["scale"])
    else:
        mqa.kv_append_paged_multi(kn, vn, kpd, vpd, pos, table)
        out = mqa.decode_attention_paged_multi(q, kpd, vpd, table, lens, scale=case["scale"])
    torch.cuda.synchronize()
    assert mqa.get_device_status() == 0
    assert np.array_equal(P.bits(kpd), kp) and np.array_equal(P.bits(vpd), vp)
    P.assert_close(out, ref, f"paged multi {shape} page {page_size}")
    # the same rows laid out contiguously give the same bits
    kcd, vcd = case["k"].to(dev), case["v"].to(dev)
    out_c = mqa.decode_step_multi(q, kn, vn, kcd, vcd, pos, lens, scale=case["scale"])
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), out_c.view(torch.int16))


def test_paged_multi_append_skips_a_row_on_a_bad_page(mqa):
    # the 4 new rows of sequence 0 straddle two 8-row pages; the second page is out of range
    case = multi_case(2, 4, 16, 2, 128, 20, 20, seed_id=1820, ctx=[14, 30])
    _page(case, case["k"], case["v"], case["lens"], 8, seed=1821)
    bad = case["table"].clone()
    bad[0, 2] = -5                          # rows 16 .. 23 of sequence 0
    dev = torch.device("cuda")
    kpd, vpd = case["k_pool"].to(dev), case["v_pool"].to(dev)
    mqa.kv_append_paged_multi(case["k_new"].to(dev), case["v_new"].to(dev), kpd, vpd,
                              case["pos"].to(dev), bad.to(dev))
    torch.cuda.synchronize()
    assert mqa.get_device_status() == BOUNDS
    kp, vp = P.bits(case["k_pool"]).copy(), P.bits(case["v_pool"]).copy()
    assert oracle.kv_append_paged_multi(P.bits(case["k_new"]), P.bits(case["v_new"]), kp, vp,
                                        case["pos"].numpy(), bad.numpy()) == oracle.ERR_BOUNDS
    assert np.array_equal(P.bits(kpd), kp) and np.array_equal(P.bits(vpd), vp)


def test_paged_multi_past_one_tile_of_rows_is_refused(mqa):
    # T * h / g = 9 * 8 = 72 rows: beyond the decode kernel's 64, and the prefill kernel reads
    # contiguous caches only
    case = multi_case(2, 9, 16, 2, 128, 50, 100, seed_id=1830)
    _page(case, case["k"], case["v"], case["lens"], 16, seed=1831)
    dev = torch.device("cuda")
    with pytest.raises(mqa.MqaError) as e:
        mqa.decode_attention_paged_multi(case["q"].to(dev), case["k_pool"].to(dev),
                                         case["v_pool"].to(dev), case["table"].to(dev),
                                         case["lens"].to(dev), scale=case["scale"])
    assert e.value.status == UNSUPPORTED
