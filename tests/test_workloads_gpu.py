"""GPU parity at the full sizes of the five decode workloads, in the launch configuration the
benchmark times. The oracle checks every output of the small workloads and a sample of sequences
(all their heads) of the large ones; the append is checked bit for bit on the sampled rows and,
on the device, for "nothing else changed".
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
    ("mqa_tiny", None), ("gqa_8b", None), ("mqa_long", [0, 21, 63]), ("mha_ref", [0, 5]),
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
