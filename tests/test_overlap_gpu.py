"""Launch overlap (programmatic dependent launch, mqa_set_launch_overlap) on the GPU.

With overlap on, a decode launch may start while the launch ahead of it on the stream is still
running. Over caches of up to 768 MiB it writes at once, into scratch the launch ahead does not
use, and holds the launch after it back until the launch ahead has finished; over larger caches
it reads at once but writes nothing (outputs, appended rows, partial states, arrival counters)
until that launch has finished. Results must be bit for bit those of the same launches without
overlap. These tests run sequences of launches both ways -- eager and
captured in a CUDA graph, on every inner-product path, over contiguous, paged and fp8 caches, with
one and several tokens, with layers revisited (their appends repeated) -- and compare every output
and every cache byte, then check outputs against the fp64 oracle. No launch follows one on the same
caches or output, which the overlap contract requires.
"""
from __future__ import annotations

import pytest
import torch

import oracle
from query_grouped_decode_kv_b300 import inputs
from tests import _parity as P

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mqa():
    import query_grouped_decode_kv_b300 as m
    m.debug_override(0, 0)
    yield m
    m.debug_override(0, 0)


def _layers(b, h, g, d_h, lo, hi, n, seed, dev, T=1):
    """n layers of one shape (distinct seeds, shared lengths) with caches holding NaN past the
    context; returns (pos, lens, [(q, k_new, v_new, k, v)])."""
    w = inputs.custom("ovl", b, h, g, d_h, lo, hi, wid=seed)
    if T > 1:
        import dataclasses
        w = dataclasses.replace(w, extra_rows=T - 1)
    pos, _ = inputs.positions_and_lengths(w)
    lens = (pos + T).to(torch.int32)
    out = []
    for li in range(n):
        lw = inputs.custom("ovl", b, h, g, d_h, lo, hi, wid=seed + 1 + li)
        if T > 1:
            import dataclasses
            lw = dataclasses.replace(lw, extra_rows=T - 1)
            q, kn, vn = inputs.multi_step_inputs(lw, T, 0, dev)
        else:
            q, kn, vn = inputs.step_inputs(lw, 0, dev)
        k, v = inputs.cache(lw, 0, dev, tail="nan", lengths=pos)
        out.append((q, kn, vn, k, v))
    return pos, lens, out


def _run(mqa, order, data, pos_d, lens_d, scale, stream, overlap, graph, step_fn):
    """Launch step_fn for the layer indices in `order` on `stream`; returns the outputs (one per
    launch) and the caches after the sequence. Caches are cloned so both runs start equal."""
    mqa.set_launch_overlap(overlap, stream)
    caches = [(k.clone(), v.clone()) for (_, _, _, k, v) in data]
    outs = [torch.empty_like(data[li][0]) for li in order]

    def body():
        for o, li in zip(outs, order):
            q, kn, vn, _, _ = data[li]
            k, v = caches[li]
            step_fn(li, q, kn, vn, k, v, pos_d, lens_d, o, scale, stream)

    torch.cuda.synchronize()
    if graph:
        # size the stream's workspace first on throw-away caches, then record and replay
        keep = [(k.clone(), v.clone()) for k, v in caches]
        with torch.cuda.stream(stream):
            body()
        stream.synchronize()
        for (k, v), (k0, v0) in zip(caches, keep):
            k.copy_(k0)
            v.copy_(v0)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            body()
        with torch.cuda.stream(stream):
            g.replay()
    else:
        with torch.cuda.stream(stream):
            body()
    stream.synchronize()
    assert mqa.get_device_status() == 0
    mqa.set_launch_overlap(False, stream)
    return outs, caches


def _fused(mqa):
    def f(li, q, kn, vn, k, v, pos, lens, o, scale, stream):
        if q.dim() == 4:
            mqa.decode_step_multi(q, kn, vn, k, v, pos, lens, out=o, scale=scale, stream=stream)
        else:
            mqa.decode_step(q, kn, vn, k, v, pos, lens, out=o, scale=scale, stream=stream)
    return f


def _same_bits(a_outs, a_caches, b_outs, b_caches):
    for x, y in zip(a_outs, b_outs):
        assert torch.equal(x.view(torch.int16), y.view(torch.int16))
    for (k0, v0), (k1, v1) in zip(a_caches, b_caches):
        assert torch.equal(k0.view(torch.int16), k1.view(torch.int16))
        assert torch.equal(v0.view(torch.int16), v1.view(torch.int16))


def _check_oracle(order, data, outs, pos, lens, scale, T=1, max_checks=3):
    """The first launches of each distinct layer against the oracle (append, then attention)."""
    seen = set()
    for o, li in zip(outs, order):
        if li in seen or len(seen) >= max_checks:
            continue
        seen.add(li)
        q, kn, vn, k, v = data[li]
        kb, vb = P.bits(k).copy(), P.bits(v).copy()
        if T > 1:
            assert oracle.kv_append_multi(P.bits(kn), P.bits(vn), kb, vb, pos.numpy()) == oracle.OK
            ref = oracle.decode_attention_multi(P.bits(q), kb, vb, lens.numpy(), scale)
        else:
            assert oracle.kv_append(P.bits(kn), P.bits(vn), kb, vb, pos.numpy()) == oracle.OK
            ref = oracle.decode_attention(P.bits(q), kb, vb, lens.numpy(), scale)
        P.assert_close(o, ref, f"overlapped layer {li}")


@pytest.mark.parametrize("graph", [False, True], ids=["eager", "graph"])
@pytest.mark.parametrize("shape", [
    (4, 16, 8, 128, 300, 3000),   # G = 2, CUDA cores (eight warps)
    (4, 32, 8, 128, 300, 3000),   # G = 4, mma.sync (four warps)
    (2, 16, 2, 64, 100, 2500),    # G = 8, mma.sync, d_h = 64
    (8, 64, 8, 128, 1000, 6000),  # G = 8, the 70B-class layer shape, shorter contexts
    (6, 32, 1, 128, 2000, 5000),  # G = 32, MQA (eight warps)
], ids=["G2", "G4", "G8_d64", "G8", "G32"])
def test_overlapped_fused_layers_equal_serial_ones_bit_for_bit(mqa, shape, graph):
    dev = torch.device("cuda")
    pos, lens, data = _layers(*shape, n=4, seed=700 + shape[1] + shape[2], dev=dev)
    # distinct layers back to back, then layers again (their appends repeated); no launch
    # follows one on the same caches, the condition for overlap
    order = [0, 1, 2, 3, 0, 3, 1]
    scale = data[0][0].shape[-1] ** -0.5
    s = torch.cuda.Stream()
    args = (order, data, pos.to(dev), lens.to(dev), scale, s)
    serial = _run(mqa, *args, overlap=False, graph=graph, step_fn=_fused(mqa))
    overl = _run(mqa, *args, overlap=True, graph=graph, step_fn=_fused(mqa))
    _same_bits(*serial, *overl)
    _check_oracle(order, data, overl[0], pos, lens, scale)


def test_overlapped_attention_calls_on_distinct_caches_equal_serial_ones(mqa):
    """Unfused attention launches back to back (no append between them) on distinct caches."""
    dev = torch.device("cuda")
    pos, lens, data = _layers(3, 16, 2, 128, 500, 4000, n=3, seed=760, dev=dev)

    def attend(li, q, kn, vn, k, v, pos_d, lens_d, o, scale, stream):
        mqa.decode_attention(q, k, v, lens_d, out=o, scale=scale, stream=stream)
    s = torch.cuda.Stream()
    args = ([0, 1, 2, 0, 2], data, pos.to(dev), lens.to(dev), 128 ** -0.5, s)
    serial = _run(mqa, *args, overlap=False, graph=False, step_fn=attend)
    overl = _run(mqa, *args, overlap=True, graph=True, step_fn=attend)
    _same_bits(*serial, *overl)


@pytest.mark.parametrize("T", [2, 4])
def test_overlapped_multi_token_layers_equal_serial_ones(mqa, T):
    dev = torch.device("cuda")
    pos, lens, data = _layers(3, 32, 4, 128, 200, 2500, n=3, seed=780 + T, dev=dev, T=T)
    order = [0, 1, 2, 0, 2]
    s = torch.cuda.Stream()
    args = (order, data, pos.to(dev), lens.to(dev), 128 ** -0.5, s)
    serial = _run(mqa, *args, overlap=False, graph=False, step_fn=_fused(mqa))
    overl = _run(mqa, *args, overlap=True, graph=True, step_fn=_fused(mqa))
    _same_bits(*serial, *overl)
    _check_oracle(order, data, overl[0], pos, lens, 128 ** -0.5, T=T)


def test_overlapped_paged_and_fp8_layers_equal_serial_ones(mqa):
    dev = torch.device("cuda")
    pos, lens, data = _layers(4, 64, 8, 128, 300, 3000, n=3, seed=790, dev=dev)
    s = torch.cuda.Stream()
    order = [0, 1, 2, 1]
    # paged: every layer's rows in 16-row pages under one shared table
    rows = lens.clone()
    pools, table = [], None
    for li, (q, kn, vn, k, v) in enumerate(data):
        kp, vp, tbl = inputs.page_pool(k, v, rows, 16, seed=791)
        table = tbl.to(dev)
        pools.append((q, kn, vn, kp, vp))

    def paged(li, q, kn, vn, k, v, pos_d, lens_d, o, scale, stream):
        mqa.decode_step_paged(q, kn, vn, k, v, pos_d, table, lens_d, out=o, scale=scale,
                              stream=stream)
    args = (order, pools, pos.to(dev), lens.to(dev), 128 ** -0.5, s)
    serial = _run(mqa, *args, overlap=False, graph=False, step_fn=paged)
    overl = _run(mqa, *args, overlap=True, graph=True, step_fn=paged)
    _same_bits(*serial, *overl)
    # fp8: the same draws as E4M3 codes, one scale per tensor
    f8, scales = [], []
    for (q, kn, vn, k, v) in data:
        ks, vs = inputs.amax_scale(k), inputs.amax_scale(v)
        f8.append((q, kn, vn, inputs.fp8_codes(k, ks), inputs.fp8_codes(v, vs)))
        scales.append((ks, vs))

    def fp8_step(li, q, kn, vn, k, v, pos_d, lens_d, o, scale, stream):
        mqa.decode_step_fp8(q, kn, vn, k, v, pos_d, lens_d, *scales[li], out=o, scale=scale,
                            stream=stream)
    args = (order, f8, pos.to(dev), lens.to(dev), 128 ** -0.5, s)
    serial = _run(mqa, *args, overlap=False, graph=False, step_fn=fp8_step)
    overl = _run(mqa, *args, overlap=True, graph=True, step_fn=fp8_step)
    for x, y in zip(serial[0], overl[0]):
        assert torch.equal(x.view(torch.int16), y.view(torch.int16))
    for (k0, v0), (k1, v1) in zip(serial[1], overl[1]):
        assert torch.equal(k0, k1) and torch.equal(v0, v1)


def test_overlap_setting_is_per_stream_and_validated(mqa):
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    mqa.set_launch_overlap(True, s1)
    mqa.set_launch_overlap(False, s2)
    mqa.set_launch_overlap(False, s1)
    lib = mqa.raw()
    assert lib.mqa_set_launch_overlap(s1.cuda_stream, 2) == 1   # MQA_ERR_INVALID_ARG
    assert lib.mqa_set_launch_overlap(s1.cuda_stream, -1) == 1


@pytest.mark.parametrize("graph", [False, True], ids=["eager", "graph"])
@pytest.mark.parametrize("shape", [
    (4, 16, 8, 128, 300, 3000),   # G = 2, CUDA cores
    (4, 64, 8, 128, 300, 3000),   # G = 8, mma.sync
], ids=["G2", "G8"])
def test_overlapped_layers_over_large_caches_equal_serial_ones(mqa, shape, graph):
    """Caches of more than 768 MiB (here about 870 MB per layer, most of it rows past the
    contexts): overlapped launches then read early but wait for the launch ahead before their
    first write. Same bits as without overlap, and the oracle's result."""
    import dataclasses
    dev = torch.device("cuda")
    b, h, g, d_h, lo, hi = shape
    extra = 50_000
    assert 2 * b * g * (hi + 1 + extra) * d_h * 2 > 768 * 2 ** 20
    w = dataclasses.replace(inputs.custom("big", b, h, g, d_h, lo, hi, wid=820 + h),
                            extra_rows=extra)
    pos, lens = inputs.positions_and_lengths(w)
    data = []
    for li in range(3):
        lw = dataclasses.replace(inputs.custom("big", b, h, g, d_h, lo, hi, wid=821 + h + li),
                                 extra_rows=extra)
        q, kn, vn = inputs.step_inputs(lw, 0, dev)
        k, v = inputs.cache(lw, 0, dev, tail="nan", lengths=pos)
        data.append((q, kn, vn, k, v))
    order = [0, 1, 2, 0, 2]
    scale = d_h ** -0.5
    s = torch.cuda.Stream()
    args = (order, data, pos.to(dev), lens.to(dev), scale, s)
    serial = _run(mqa, *args, overlap=False, graph=graph, step_fn=_fused(mqa))
    overl = _run(mqa, *args, overlap=True, graph=graph, step_fn=_fused(mqa))
    _same_bits(*serial, *overl)
    _check_oracle(order, data, overl[0], pos, lens, scale, max_checks=1)


def test_overlapped_paged_fp8_and_paged_multi_layers_equal_serial_ones(mqa):
    """Pages combined with fp8 codes, and with several new tokens, under overlap: the two paged
    producer warps of every launch write their tiles' new rows early or after the wait."""
    dev = torch.device("cuda")
    s = torch.cuda.Stream()
    order = [0, 1, 2, 0, 2]
    # fp8 codes in 16-row pages
    pos, lens, data = _layers(4, 32, 4, 128, 300, 3000, n=3, seed=800, dev=dev)
    f8, scales, table = [], [], None
    for (q, kn, vn, k, v) in data:
        ks, vs = inputs.amax_scale(k), inputs.amax_scale(v)
        kp, vp, tbl = inputs.page_pool(inputs.fp8_codes(k, ks), inputs.fp8_codes(v, vs), lens, 16,
                                       seed=801)
        table = tbl.to(dev)
        f8.append((q, kn, vn, kp, vp))
        scales.append((ks, vs))

    def paged_fp8(li, q, kn, vn, k, v, pos_d, lens_d, o, scale, stream):
        mqa.decode_step_paged_fp8(q, kn, vn, k, v, pos_d, table, lens_d, *scales[li], out=o,
                                  scale=scale, stream=stream)
    args = (order, f8, pos.to(dev), lens.to(dev), 128 ** -0.5, s)
    serial = _run(mqa, *args, overlap=False, graph=False, step_fn=paged_fp8)
    overl = _run(mqa, *args, overlap=True, graph=True, step_fn=paged_fp8)
    for x, y in zip(serial[0], overl[0]):
        assert torch.equal(x.view(torch.int16), y.view(torch.int16))
    for (k0, v0), (k1, v1) in zip(serial[1], overl[1]):
        assert torch.equal(k0, k1) and torch.equal(v0, v1)
    # four tokens per sequence in 8-row pages
    T = 4
    pos, lens, data = _layers(3, 32, 4, 128, 200, 2500, n=3, seed=810, dev=dev, T=T)
    paged = []
    for (q, kn, vn, k, v) in data:
        kp, vp, tbl = inputs.page_pool(k, v, lens, 8, seed=811)
        table = tbl.to(dev)
        paged.append((q, kn, vn, kp, vp))

    def paged_multi(li, q, kn, vn, k, v, pos_d, lens_d, o, scale, stream):
        mqa.decode_step_paged_multi(q, kn, vn, k, v, pos_d, table, lens_d, out=o, scale=scale,
                                    stream=stream)
    args = (order, paged, pos.to(dev), lens.to(dev), 128 ** -0.5, s)
    serial = _run(mqa, *args, overlap=False, graph=False, step_fn=paged_multi)
    overl = _run(mqa, *args, overlap=True, graph=True, step_fn=paged_multi)
    _same_bits(*serial, *overl)


def test_a_launch_never_runs_beside_the_one_two_back(mqa):
    """Three fused steps over large caches (the wait-before-writing mode): A (layer 0, a long
    context, one CTA), B (layer 1, one CTA) and C (layer 0 again, the next token, four CTAs).
    A appends row p of layer 0 near its end; C attends over row p, and its last CTA reaches it
    early. The overlap contract only covers adjacent launches (A and C are two apart), so C must
    not start before A has finished: the launch-order warp of B releases C only after B's own wait
    on A. Same bits as without overlap. (On B300 a build that let B release C at its start passed
    this test as well: the hardware did not start C early. The release after the wait makes the
    order hold by construction.)"""
    import dataclasses
    dev = torch.device("cuda")
    b, h, g, d_h = 1, 64, 8, 128
    ctx = 150_000
    extra = 60_000  # caches of 2 * 8 * 210,002 * 128 * 2 B = 860 MB per layer: above 768 MiB
    w0 = dataclasses.replace(inputs.custom("far", b, h, g, d_h, ctx, ctx, wid=830), extra_rows=extra)
    w1 = dataclasses.replace(inputs.custom("far", b, h, g, d_h, 10, 10, wid=831), extra_rows=extra)
    assert 2 * b * g * w0.n_max * d_h * 2 > 768 * 2 ** 20
    pos0, lens0 = inputs.positions_and_lengths(w0)
    pos1, lens1 = inputs.positions_and_lengths(w1)
    k0, v0 = inputs.cache(w0, 0, dev, tail="nan")
    k1, v1 = inputs.cache(w1, 0, dev, tail="nan")
    qa, kna, vna = inputs.step_inputs(w0, 0, dev)
    qb, knb, vnb = inputs.step_inputs(w1, 0, dev)
    qc, knc, vnc = inputs.step_inputs(w0, 1, dev)
    pos_c, lens_c = (pos0 + 1).to(dev), (lens0 + 1).to(dev)
    scale = d_h ** -0.5

    def run(overlap):
        ks = [(k0.clone(), v0.clone()), (k1.clone(), v1.clone())]
        outs = [torch.empty_like(qa), torch.empty_like(qb), torch.empty_like(qc)]
        s = torch.cuda.Stream()
        mqa.set_launch_overlap(overlap, s)
        torch.cuda.synchronize()
        try:
            with torch.cuda.stream(s):
                mqa.debug_override(1, 0)
                mqa.decode_step(qa, kna, vna, *ks[0], pos0.to(dev), lens0.to(dev), out=outs[0],
                                scale=scale, stream=s)
                mqa.decode_step(qb, knb, vnb, *ks[1], pos1.to(dev), lens1.to(dev), out=outs[1],
                                scale=scale, stream=s)
                mqa.debug_override(4, 0)
                mqa.decode_step(qc, knc, vnc, *ks[0], pos_c, lens_c, out=outs[2], scale=scale,
                                stream=s)
            s.synchronize()
        finally:
            mqa.debug_override(0, 0)
            mqa.set_launch_overlap(False, s)
        assert mqa.get_device_status() == 0
        return outs, ks

    serial = run(False)
    overl = run(True)
    assert torch.isfinite(overl[0][2].float()).all(), "C read a row A had not written yet"
    _same_bits(*serial, *overl)
