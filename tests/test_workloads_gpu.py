"""GPU parity at the full sizes of the five decode workloads, in the launch configuration the
benchmark times. The oracle checks every output of the four one-layer workloads (every sequence
and head) and a sample of sequences of three layers of the 80-layer step; the append is checked
bit for bit on the checked rows and, on the device, for "nothing else changed".
"""
from __future__ import annotations

import numpy as np
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
    return m


def _bits_changed(a: torch.Tensor, b: torch.Tensor) -> torch.Tensor:
    """[b, g, n] mask of rows whose bit patterns differ."""
    return (a.view(torch.int16) != b.view(torch.int16)).any(dim=-1)


def _check_layer(mqa, w, q, kn, vn, k, v, pos, lens, sample, tag):
    """Append + attention on device; oracle on the sampled sequences."""
    dev = k.device
    k_host = P.bits(k[sample]).copy()
    v_host = P.bits(v[sample]).copy()
    k0, v0 = k.clone(), v.clone()
    mqa.kv_append(kn, vn, k, v, pos.to(dev))
    out = mqa.decode_attention(q, k, v, lens.to(dev), scale=w.scale)
    torch.cuda.synchronize()
    assert mqa.get_device_status() == 0
    # only the appended rows changed
    changed = _bits_changed(k, k0) | _bits_changed(v, v0)
    expect = torch.zeros_like(changed)
    for bi in range(w.b):
        expect[bi, :, int(pos[bi])] = True
    assert bool((changed & ~expect).sum() == 0), f"{tag}: append touched other rows"
    del k0, v0
    # oracle on the sample
    st = oracle.kv_append(P.bits(kn[sample]), P.bits(vn[sample]), k_host, v_host,
                          pos[sample].numpy())
    assert st == oracle.OK
    assert np.array_equal(P.bits(k[sample]), k_host), f"{tag}: K append not bit-exact"
    assert np.array_equal(P.bits(v[sample]), v_host), f"{tag}: V append not bit-exact"
    ref = oracle.decode_attention(P.bits(q[sample]), k_host, v_host, lens[sample].numpy(),
                                  w.scale)
    return P.assert_close(out[sample], ref, tag)


@pytest.mark.parametrize("name,sample", [
    ("mqa_tiny", None), ("gqa_8b", None), ("mqa_long", None), ("mha_ref", None),
])
def test_single_layer_workloads(mqa, name, sample):
    w = inputs.WORKLOADS[name]
    dev = torch.device("cuda")
    q, kn, vn = inputs.step_inputs(w, 0, dev)
    k, v = inputs.cache(w, 0, dev, tail="nan")
    pos, lens = inputs.positions_and_lengths(w)
    idx = list(range(w.b)) if sample is None else sample
    stats = _check_layer(mqa, w, q, kn, vn, k, v, pos, lens, idx, name)
    print(name, stats)


def test_80_layer_step_sampled(mqa):
    """The full 80-layer GQA step (about 86 GB of cache), run as the benchmark runs it; the oracle
    checks three layers on two sequences each."""
    from query_grouped_decode_kv_b300.layers import LayerState, StepInputs, decode_layers
    w = inputs.WORKLOADS["gqa_70b_80l"]
    dev = torch.device("cuda")
    pos, lens = inputs.positions_and_lengths(w)
    check_layers = {0: None, 41: None, 79: None}
    sample = [int(torch.argmax(lens)), int(torch.argmin(lens))]
    layers, xs, outs = [], [], []
    for li in range(w.layers):
        k, v = inputs.cache(w, li, dev, tail="nan")
        if li in check_layers:
            check_layers[li] = (P.bits(k[sample]).copy(), P.bits(v[sample]).copy())
        layers.append(LayerState(k, v))
        xs.append(StepInputs(*inputs.step_inputs(w, li, dev)))
        outs.append(torch.empty(w.b, w.h, w.d_h, dtype=torch.bfloat16, device=dev))
    decode_layers(layers, xs, pos.to(dev), lens.to(dev), outs, w.scale)
    torch.cuda.synchronize()
    assert mqa.get_device_status() == 0
    for li, (kh, vh) in check_layers.items():
        x = xs[li]
        assert oracle.kv_append(P.bits(x.k_new[sample]), P.bits(x.v_new[sample]), kh, vh,
                                pos[sample].numpy()) == oracle.OK
        assert np.array_equal(P.bits(layers[li].k_cache[sample]), kh)
        assert np.array_equal(P.bits(layers[li].v_cache[sample]), vh)
        ref = oracle.decode_attention(P.bits(x.q[sample]), kh, vh, lens[sample].numpy(), w.scale)
        print("layer", li, P.assert_close(outs[li][sample], ref, f"layer {li}"))


@pytest.mark.parametrize("graph", [False, True], ids=["eager", "graph"])
@pytest.mark.parametrize("chunk", [2, 3, 8], ids=["runs_2_3_2", "runs_3_1_3", "one_run"])
def test_host_driven_step_matches_the_device_step(mqa, chunk, graph):
    """layers.HostStepPipeline (inputs copied in and outputs out, overlapped in runs of layers)
    gives, bit for bit, the outputs and caches of the device-resident multi-layer step."""
    from query_grouped_decode_kv_b300.layers import (HostStepBuffers, HostStepPipeline,
                                                     LayerState, StepInputs, decode_layers)
    w = inputs.custom("host_step", 3, 16, 2, 128, 100, 900)
    n_layers = 7
    dev = torch.device("cuda")
    pos, lens = inputs.positions_and_lengths(w)
    pos_d, lens_d = pos.to(dev), lens.to(dev)
    xs, lay_a, lay_b = [], [], []
    for li in range(n_layers):
        lw = inputs.custom("host_step", 3, 16, 2, 128, 100, 900, wid=900 + li)
        k, v = inputs.cache(lw, 0, dev, tail="nan", lengths=pos)
        lay_a.append(LayerState(k.clone(), v.clone()))
        lay_b.append(LayerState(k, v))
        xs.append(StepInputs(*inputs.step_inputs(lw, 0, dev)))
    outs = [torch.empty(w.b, w.h, w.d_h, dtype=torch.bfloat16, device=dev) for _ in range(n_layers)]
    decode_layers(lay_a, xs, pos_d, lens_d, outs, w.scale)
    buf = HostStepBuffers.allocate(n_layers, w.b, w.h, w.g, w.d_h, dev)
    for li, x in enumerate(xs):
        buf.q_host[li].copy_(x.q.cpu())
        buf.kn_host[li].copy_(x.k_new.cpu())
        buf.vn_host[li].copy_(x.v_new.cpu())
    pipe = HostStepPipeline(lay_b, buf, chunk=chunk)
    if graph:
        # record the step on a side stream (the workspace of that stream is sized first by a run
        # on caches that are then discarded), replay it once on the real caches' copies
        side = torch.cuda.Stream()
        keep = [(l.k_cache.clone(), l.v_cache.clone()) for l in lay_b]
        with torch.cuda.stream(side):
            pipe.run(pos_d, lens_d, w.scale, side)
        side.synchronize()
        for l, (k0, v0) in zip(lay_b, keep):
            l.k_cache.copy_(k0)
            l.v_cache.copy_(v0)
        buf.out_host.zero_()
        torch.cuda.synchronize()
        g = pipe.capture(pos_d, lens_d, w.scale, side)
        with torch.cuda.stream(side):
            g.replay()
        side.synchronize()
    else:
        pipe.run(pos_d, lens_d, w.scale, torch.cuda.current_stream())
    torch.cuda.synchronize()
    assert mqa.get_device_status() == 0
    for li in range(n_layers):
        assert torch.equal(buf.out_host[li].view(torch.int16), outs[li].cpu().view(torch.int16))
        assert torch.equal(lay_b[li].k_cache.view(torch.int16), lay_a[li].k_cache.view(torch.int16))
        assert torch.equal(lay_b[li].v_cache.view(torch.int16), lay_a[li].v_cache.view(torch.int16))
