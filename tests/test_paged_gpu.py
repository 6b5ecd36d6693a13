"""GPU parity of the paged-cache calls (mqa_kv_append_paged, mqa_decode_attention_paged,
mqa_decode_step_paged) against the fp64 oracle, on the same seeded inputs.

The oracle's side: append through the page table (oracle.kv_append_paged), gather the cache the
table describes (oracle.gather_pages) and attend over it (oracle.decode_attention). The pools are
compared bit for bit, guard pages included; the outputs within the contract's tolerances. The
pages of every sequence are scattered over the pool in a seeded random order, with spare pages
full of NaN that no table entry names, and table entries past a sequence's pages are -1.
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


def paged_case(shape, page_size, seed_id, spare_pages=3, lens=None, pos=None):
    """A contiguous case laid out as page pools: every sequence gets the pages that its
    attended rows and its append row need."""
    case = P.make_case(*shape, seed_id=seed_id)
    if lens is not None:
        case["lens"] = torch.tensor(lens, dtype=torch.int32)
        case["pos"] = torch.tensor(pos, dtype=torch.int32)
        case["k"], case["v"] = inputs.cache(case["w"], 0, "cpu", tail="nan", lengths=case["lens"])
    n_max = case["w"].n_max
    rows = torch.maximum(case["lens"], torch.clamp(case["pos"] + 1, max=n_max))
    kp, vp, table = inputs.page_pool(case["k"], case["v"], rows, page_size, seed=seed_id * 7 + 1,
                                     spare_pages=spare_pages)
    case.update(k_pool=kp, v_pool=vp, table=table, page_size=page_size)
    return case


def oracle_paged_step(case, append=True):
    """(k_pool, v_pool, out, append status, gather status) from the oracle."""
    kp, vp = P.bits(case["k_pool"]).copy(), P.bits(case["v_pool"]).copy()
    table = case["table"].numpy()
    st = oracle.OK
    if append:
        st = oracle.kv_append_paged(P.bits(case["k_new"]), P.bits(case["v_new"]), kp, vp,
                                    case["pos"].numpy(), table)
    kc, gst = oracle.gather_pages(kp, table, case["page_size"])
    vc, _ = oracle.gather_pages(vp, table, case["page_size"])
    out = oracle.decode_attention(P.bits(case["q"]), kc, vc, case["lens"].numpy(), case["scale"])
    return kp, vp, out, st, gst


def gpu_paged(case, mqa, fused=True, stream=None):
    dev = torch.device("cuda")
    q = case["q"].to(dev)
    kn, vn = case["k_new"].to(dev), case["v_new"].to(dev)
    kp, vp = case["k_pool"].to(dev), case["v_pool"].to(dev)
    pos, lens, table = case["pos"].to(dev), case["lens"].to(dev), case["table"].to(dev)
    if fused:
        out = mqa.decode_step_paged(q, kn, vn, kp, vp, pos, table, lens, scale=case["scale"],
                                    stream=stream)
    else:
        mqa.kv_append_paged(kn, vn, kp, vp, pos, table, stream=stream)
        out = mqa.decode_attention_paged(q, kp, vp, table, lens, scale=case["scale"],
                                         stream=stream)
    return kp, vp, out


SHAPES = [
    # b, h, g, d_h, ctx_lo, ctx_hi
    (1, 8, 1, 64, 128, 128),      # tiny MQA step, G = 8 (mma.sync)
    (3, 8, 2, 64, 0, 300),        # G = 4 (mma.sync), lengths from 1
    (2, 16, 2, 128, 100, 700),    # G = 8, mma.sync
    (2, 32, 1, 128, 1, 1000),     # G = 32, eight consumer warps
    (4, 32, 8, 128, 0, 513),      # GQA 8B-class heads, short ragged contexts
    (2, 7, 1, 128, 60, 200),      # G = 7
    (3, 4, 2, 128, 0, 300),       # G = 2, CUDA cores, lengths from 1
]
PAGE_SIZES = [8, 16, 32, 64, 128]


@pytest.mark.parametrize("page_size", PAGE_SIZES)
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "b{}h{}g{}d{}_{}-{}".format(*s))
@pytest.mark.parametrize("fused", [True, False], ids=["fused", "two_launches"])
def test_paged_step_matches_oracle(mqa, shape, page_size, fused):
    case = paged_case(shape, page_size, seed_id=900 + SHAPES.index(shape))
    kp_ref, vp_ref, out_ref, st, gst = oracle_paged_step(case)
    assert st == oracle.OK
    kp, vp, out = gpu_paged(case, mqa, fused=fused)
    torch.cuda.synchronize()
    assert mqa.get_device_status() == 0
    assert np.array_equal(P.bits(kp), kp_ref), "K pool differs from the oracle's paged append"
    assert np.array_equal(P.bits(vp), vp_ref), "V pool differs from the oracle's paged append"
    P.assert_close(out, out_ref, f"paged {shape} page_size={page_size}")


@pytest.mark.parametrize("ctas", [1, 2, 3, 7, 64, 148, 1000])
@pytest.mark.parametrize("shape,path", [((2, 16, 2, 128, 0, 700), 0), ((3, 8, 4, 64, 100, 400), 1)],
                         ids=["mma_sync", "cuda_cores"])
def test_paged_step_any_cta_split(mqa, shape, path, ctas):
    case = paged_case(shape, 16, seed_id=920)
    kp_ref, vp_ref, out_ref, _, _ = oracle_paged_step(case)
    mqa.debug_override(ctas, path)
    try:
        kp, vp, out = gpu_paged(case, mqa)
        assert mqa.get_device_status() == 0
    finally:
        mqa.debug_override(0, 0)
    assert np.array_equal(P.bits(kp), kp_ref) and np.array_equal(P.bits(vp), vp_ref)
    P.assert_close(out, out_ref, f"paged {shape} ctas={ctas}")


@pytest.mark.parametrize("page_size", [16, 64])
@pytest.mark.parametrize("shape", [(3, 32, 8, 128, 100, 2000), (2, 8, 8, 128, 100, 2000),
                                   (2, 64, 2, 128, 100, 900)], ids=["G4", "G1", "G32"])
def test_paged_equals_contiguous_bit_for_bit(mqa, shape, page_size):
    # the same rows reach the same shared-memory layout, so the arithmetic is the same
    case = paged_case(shape, page_size, seed_id=930)
    mqa.debug_override(37, 0)   # the same split for both calls
    try:
        _, _, o_paged = gpu_paged(case, mqa)
        _, _, o_flat = P.gpu_step(case, mqa)
        torch.cuda.synchronize()
        assert mqa.get_device_status() == 0
    finally:
        mqa.debug_override(0, 0)
    assert torch.equal(o_paged.view(torch.int16), o_flat.view(torch.int16))


@pytest.mark.parametrize("path", [1, 2])
@pytest.mark.parametrize("ctas", [0, 1, 5])
def test_paged_append_row_anywhere(mqa, path, ctas):
    # append rows: the last attended row; inside the attended range; past the length inside the
    # last loaded tile; past every loaded tile; out of range (skipped, latched); first row of a
    # tile
    # a sequence addresses max_pages * page_size = 19 * 16 = 304 rows (its cache holds 301)
    lens = [200, 300, 100, 70, 150, 129]
    pos = [199, 37, 110, 250, 304, 128]
    case = paged_case((6, 8, 2, 128, 60, 300), 16, seed_id=940, lens=lens, pos=pos)
    assert case["table"].shape[1] * 16 == 304
    kp_ref, vp_ref, out_ref, st, _ = oracle_paged_step(case)
    assert st == oracle.ERR_BOUNDS
    mqa.debug_override(ctas, path)
    try:
        kp, vp, out = gpu_paged(case, mqa)
        assert mqa.get_device_status() == BOUNDS
    finally:
        mqa.debug_override(0, 0)
    assert np.array_equal(P.bits(kp), kp_ref) and np.array_equal(P.bits(vp), vp_ref)
    P.assert_close(out, out_ref, f"paged append rows anywhere, path {path}, ctas {ctas}")


def test_paged_shared_prefix_pages(mqa):
    # sequences 1 and 2 read sequence 0's first three pages (a common prefix) and have pages of
    # their own after them; nothing is appended to a shared page
    ps = 16
    case = paged_case((3, 16, 2, 128, 150, 150), ps, seed_id=950, spare_pages=5)
    table = case["table"].clone()
    shared = table[0, :3].clone()
    for bi in (1, 2):
        table[bi, :3] = shared
    case["table"] = table
    kp_ref, vp_ref, out_ref, st, gst = oracle_paged_step(case)
    assert st == oracle.OK
    kp, vp, out = gpu_paged(case, mqa)
    assert mqa.get_device_status() == 0
    assert np.array_equal(P.bits(kp), kp_ref) and np.array_equal(P.bits(vp), vp_ref)
    P.assert_close(out, out_ref, "shared prefix pages")
    # the shared rows really are shared: sequences 1 and 2 saw sequence 0's prefix
    kc, _ = oracle.gather_pages(kp_ref, table.numpy(), ps)
    assert np.array_equal(kc[1, :, :3 * ps], kc[0, :, :3 * ps])


@pytest.mark.parametrize("fused", [True, False], ids=["fused", "two_launches"])
def test_paged_bad_page_reads_zeros_and_latches(mqa, fused):
    # sequence 1's second page and sequence 2's append page are out of range: the first reads as
    # zero rows (as the oracle's gather gives it), the second append is skipped; both latch
    ps = 32
    case = paged_case((3, 16, 2, 128, 100, 200), ps, seed_id=960)
    table = case["table"].clone()
    num_pages = case["k_pool"].shape[0]
    table[1, 1] = num_pages
    p2 = int(case["pos"][2])
    table[2, p2 // ps] = -7
    case["table"] = table
    kp_ref, vp_ref, out_ref, st, gst = oracle_paged_step(case)
    assert st == oracle.ERR_BOUNDS and gst == oracle.ERR_BOUNDS
    kp, vp, out = gpu_paged(case, mqa, fused=fused)
    assert mqa.get_device_status() == BOUNDS
    assert np.array_equal(P.bits(kp), kp_ref) and np.array_equal(P.bits(vp), vp_ref)
    P.assert_close(out, out_ref, "bad page indices")


def test_paged_table_entries_past_the_length_are_not_read(mqa):
    # entries past each sequence's last page hold out-of-range values: no error, same result
    case = paged_case((2, 16, 2, 128, 100, 300), 16, seed_id=970)
    table = case["table"].clone()
    table[table < 0] = 1 << 30
    case["table"] = table
    lens = case["lens"].numpy()
    kp_ref, vp_ref, _, st, _ = oracle_paged_step(case)
    assert st == oracle.OK
    # the oracle's gather reports those entries; attend over the gathered rows it does produce
    kc, _ = oracle.gather_pages(kp_ref, table.numpy(), 16)
    vc, _ = oracle.gather_pages(vp_ref, table.numpy(), 16)
    out_ref = oracle.decode_attention(P.bits(case["q"]), kc, vc, lens, case["scale"])
    kp, vp, out = gpu_paged(case, mqa)
    assert mqa.get_device_status() == 0
    assert np.array_equal(P.bits(kp), kp_ref) and np.array_equal(P.bits(vp), vp_ref)
    P.assert_close(out, out_ref, "table entries past the length")


def test_paged_invalid_length_writes_zeros(mqa):
    case = paged_case((4, 8, 2, 64, 10, 300), 16, seed_id=980)
    lens = case["lens"].clone()
    lens[1] = 0
    case["lens"] = lens
    kp_ref, vp_ref, out_ref, st, _ = oracle_paged_step(case)
    kp, vp, out = gpu_paged(case, mqa)
    assert mqa.get_device_status() == BOUNDS
    assert np.array_equal(P.bits(kp), kp_ref) and np.array_equal(P.bits(vp), vp_ref)
    assert np.all(P.bits(out)[1] == 0)
    keep = [0, 2, 3]
    P.assert_close(out[keep], out_ref[keep], "valid sequences next to an invalid one")


def test_paged_rejects_the_tcgen05_path(mqa):
    case = paged_case((1, 32, 1, 128, 100, 100), 16, seed_id=990)
    mqa.debug_override(0, 3)
    try:
        with pytest.raises(mqa.MqaError) as e:
            gpu_paged(case, mqa)
        assert e.value.status == 2
    finally:
        mqa.debug_override(0, 0)


@pytest.mark.parametrize("fused", [True, False], ids=["fused", "two_launches"])
def test_paged_layers_share_one_table(mqa, fused):
    # four layers, each with its own page pools, one page table shared by all of them, driven by
    # layers.decode_layers; every layer against the oracle's paged append + gather + attention
    from query_grouped_decode_kv_b300.layers import LayerState, StepInputs, decode_layers
    ps, n_layers = 16, 4
    dev = torch.device("cuda")
    w = inputs.custom("paged_layers", 3, 16, 2, 128, 50, 600, wid=1100)
    pos, lens = inputs.positions_and_lengths(w)
    cases, layers, xs = [], [], []
    table = None
    for li in range(n_layers):
        lw = inputs.custom("paged_layers", 3, 16, 2, 128, 50, 600, wid=1100 + li)
        k, v = inputs.cache(lw, 0, "cpu", tail="nan", lengths=pos)
        kp, vp, t = inputs.page_pool(k, v, lens, ps, seed=1199, spare_pages=2)
        assert table is None or torch.equal(t, table)   # same seed and lengths: the same table
        table = t
        q, kn, vn = inputs.step_inputs(lw, 0, "cpu")
        cases.append(dict(q=q, k_new=kn, v_new=vn, k_pool=kp, v_pool=vp, table=t, pos=pos,
                          lens=lens, page_size=ps, scale=w.scale))
        layers.append(LayerState(kp.to(dev), vp.to(dev), None))
        xs.append(StepInputs(q.to(dev), kn.to(dev), vn.to(dev)))
    table_d = table.to(dev)
    for lay in layers:
        lay.page_table = table_d
    outs = [torch.empty(w.b, w.h, w.d_h, dtype=torch.bfloat16, device=dev)
            for _ in range(n_layers)]
    decode_layers(layers, xs, pos.to(dev), lens.to(dev), outs, w.scale, fused=fused)
    torch.cuda.synchronize()
    assert mqa.get_device_status() == 0
    for li, (case, lay, o) in enumerate(zip(cases, layers, outs)):
        kp_ref, vp_ref, out_ref, st, _ = oracle_paged_step(case)
        assert st == oracle.OK
        assert np.array_equal(P.bits(lay.k_cache), kp_ref), f"layer {li} K pool"
        assert np.array_equal(P.bits(lay.v_cache), vp_ref), f"layer {li} V pool"
        P.assert_close(o, out_ref, f"paged layer {li}")


def test_paged_host_pipeline_matches_the_device_step(mqa):
    # the host-buffer pipeline drives paged layers through the same fused calls
    from query_grouped_decode_kv_b300.layers import (HostStepBuffers, HostStepPipeline,
                                                     LayerState, StepInputs, decode_layers)
    ps, n_layers = 32, 5
    dev = torch.device("cuda")
    w = inputs.custom("paged_host", 2, 32, 4, 128, 100, 700, wid=1200)
    pos, lens = inputs.positions_and_lengths(w)
    pos_d, lens_d = pos.to(dev), lens.to(dev)
    lay_a, lay_b, xs = [], [], []
    for li in range(n_layers):
        lw = inputs.custom("paged_host", 2, 32, 4, 128, 100, 700, wid=1200 + li)
        k, v = inputs.cache(lw, 0, dev, tail="nan", lengths=pos)
        kp, vp, t = inputs.page_pool(k, v, lens, ps, seed=1299)
        td = t.to(dev)
        lay_a.append(LayerState(kp.clone(), vp.clone(), td))
        lay_b.append(LayerState(kp, vp, td))
        xs.append(StepInputs(*inputs.step_inputs(lw, 0, dev)))
    outs = [torch.empty(w.b, w.h, w.d_h, dtype=torch.bfloat16, device=dev)
            for _ in range(n_layers)]
    decode_layers(lay_a, xs, pos_d, lens_d, outs, w.scale)
    buf = HostStepBuffers.allocate(n_layers, w.b, w.h, w.g, w.d_h, dev)
    for li, x in enumerate(xs):
        buf.q_host[li].copy_(x.q.cpu())
        buf.kn_host[li].copy_(x.k_new.cpu())
        buf.vn_host[li].copy_(x.v_new.cpu())
    HostStepPipeline(lay_b, buf, chunk=2).run(pos_d, lens_d, w.scale,
                                              torch.cuda.current_stream())
    torch.cuda.synchronize()
    assert mqa.get_device_status() == 0
    for li in range(n_layers):
        assert torch.equal(buf.out_host[li].view(torch.int16), outs[li].cpu().view(torch.int16))
        assert torch.equal(lay_b[li].k_cache.view(torch.int16), lay_a[li].k_cache.view(torch.int16))
        assert torch.equal(lay_b[li].v_cache.view(torch.int16), lay_a[li].v_cache.view(torch.int16))
