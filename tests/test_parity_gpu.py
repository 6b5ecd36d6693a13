"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle on the same seeded inputs.

Small cases span several 64-row tiles with ragged tails, both head dimensions, every kernel
family (the automatic paths: CUDA cores for G = 1..2, mma.sync from G = 3 up to 64; forced:
CUDA cores G = 1..7, mma.sync G = 1..2, tcgen05 G = 1..64) and rows past each sequence's length
poisoned with NaN. Append is compared bit for bit over the whole cache.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

from tests import _parity as P

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mqa():
    import query_grouped_decode_kv_b300 as m
    m.debug_override(0, 0)
    yield m
    m.debug_override(0, 0)


SMALL = [
    # b, h, g, d_h, ctx_lo, ctx_hi
    (1, 8, 1, 64, 128, 128),      # the tiny MQA step: G = 8, one partial tile
    (3, 8, 2, 64, 0, 300),        # G = 4, lengths from 1
    (2, 4, 4, 128, 60, 70),       # MHA (G = 1) around the 64-row tile edge
    (2, 7, 1, 128, 1, 200),       # G = 7
    (2, 6, 2, 64, 5, 130),        # G = 3
    (2, 16, 2, 128, 100, 700),    # G = 8, tensor cores
    (2, 16, 1, 64, 100, 700),     # G = 16, d_h = 64
    (2, 32, 1, 128, 1, 1000),     # G = 32 (two warps per 16-head tile)
    (1, 64, 1, 128, 500, 900),    # G = 64
    (4, 32, 8, 128, 0, 513),      # GQA 8B-class heads, short ragged contexts
    (5, 2, 1, 64, 63, 65),        # G = 2, tile edges
]


@pytest.mark.parametrize("shape", SMALL, ids=lambda s: "b{}h{}g{}d{}_{}-{}".format(*s))
def test_append_and_attention_match_oracle(mqa, shape):
    case = P.make_case(*shape, seed_id=100 + SMALL.index(shape))
    k_ref, v_ref, out_ref = P.oracle_step(case)
    k, v, out = P.gpu_step(case, mqa)
    torch.cuda.synchronize()
    assert mqa.get_device_status() == 0
    assert np.array_equal(P.bits(k), k_ref), "K append is not bit-exact"
    assert np.array_equal(P.bits(v), v_ref), "V append is not bit-exact"
    P.assert_close(out, out_ref, str(shape))


@pytest.mark.parametrize("shape", [s for s in SMALL if s[1] // s[2] < 8],
                         ids=lambda s: "b{}h{}g{}d{}_{}-{}".format(*s))
def test_cuda_core_path_matches_oracle(mqa, shape):
    # the CUDA-core consumer, forced (it is also the automatic choice for these groups)
    case = P.make_case(*shape, seed_id=100 + SMALL.index(shape))
    _, _, out_ref = P.oracle_step(case)
    mqa.debug_override(0, 1)
    try:
        _, _, out = P.gpu_step(case, mqa)
        assert mqa.get_device_status() == 0
    finally:
        mqa.debug_override(0, 0)
    P.assert_close(out, out_ref, f"CUDA cores {shape}")


@pytest.mark.parametrize("ctas", [1, 2, 3, 7, 64, 148, 1000])
@pytest.mark.parametrize("shape,path", [((2, 16, 2, 128, 0, 700), 0), ((3, 8, 4, 64, 100, 400), 1),
                                        ((2, 64, 2, 128, 0, 700), 3), ((2, 16, 2, 128, 0, 700), 3)],
                         ids=["mma_sync", "cuda_cores", "tcgen05", "tcgen05_G8"])
def test_any_cta_split_gives_the_same_result(mqa, shape, path, ctas):
    case = P.make_case(*shape, seed_id=200)
    _, _, out_ref = P.oracle_step(case)
    mqa.debug_override(ctas, path)
    try:
        _, _, out = P.gpu_step(case, mqa)
        assert mqa.get_device_status() == 0
    finally:
        mqa.debug_override(0, 0)
    P.assert_close(out, out_ref, f"{shape} ctas={ctas}")


@pytest.mark.parametrize("path", [2, 3], ids=["mma_sync", "tcgen05"])
@pytest.mark.parametrize("shape", [(2, 4, 1, 128, 10, 300), (3, 2, 2, 64, 0, 200),
                                   (2, 7, 1, 64, 60, 140)])
def test_tensor_core_paths_also_serve_small_groups(mqa, shape, path):
    case = P.make_case(*shape, seed_id=300)
    _, _, out_ref = P.oracle_step(case)
    mqa.debug_override(0, path)
    try:
        _, _, out = P.gpu_step(case, mqa)
        assert mqa.get_device_status() == 0
    finally:
        mqa.debug_override(0, 0)
    P.assert_close(out, out_ref, f"{shape} forced path {path}")


TC_SHAPES = [
    # b, h, g, d_h, ctx_lo, ctx_hi: G = 8 .. 64 on both tensor-core paths
    (2, 16, 2, 128, 1, 900),     # G = 8
    (2, 24, 2, 64, 100, 700),    # G = 12
    (2, 32, 2, 128, 50, 1000),   # G = 16
    (3, 24, 1, 128, 1, 400),     # G = 24
    (2, 32, 1, 64, 500, 1300),   # G = 32, d_h = 64
    (2, 96, 2, 128, 60, 300),    # G = 48
    (2, 64, 1, 128, 0, 2100),    # G = 64
]


@pytest.mark.parametrize("path", [2, 3], ids=["mma_sync", "tcgen05"])
@pytest.mark.parametrize("shape", TC_SHAPES, ids=lambda s: "b{}h{}g{}d{}_{}-{}".format(*s))
def test_both_tensor_core_paths_at_every_group_size(mqa, shape, path):
    case = P.make_case(*shape, seed_id=310 + TC_SHAPES.index(shape))
    _, _, out_ref = P.oracle_step(case)
    mqa.debug_override(0, path)
    try:
        _, _, out = P.gpu_step(case, mqa)
        assert mqa.get_device_status() == 0
    finally:
        mqa.debug_override(0, 0)
    P.assert_close(out, out_ref, f"{shape} path {path}")


@pytest.mark.parametrize("path", [1, 2, 3])
def test_unit_values_give_exactly_one(mqa, path):
    b, h, g, d_h = 2, 8, 2, 128
    case = P.make_case(b, h, g, d_h, 50, 600, seed_id=400)
    case["v"] = torch.ones_like(case["v"])
    case["v_new"] = torch.ones_like(case["v_new"])
    mqa.debug_override(0, path)
    try:
        _, _, out = P.gpu_step(case, mqa)
    finally:
        mqa.debug_override(0, 0)
    assert np.all(P.bits(out) == 0x3F80)


@pytest.mark.parametrize("path", [1, 2, 3])
def test_length_one_returns_the_appended_value(mqa, path):
    case = P.make_case(3, 8, 2, 64, 0, 0, seed_id=401)
    mqa.debug_override(0, path)
    try:
        _, _, out = P.gpu_step(case, mqa)
    finally:
        mqa.debug_override(0, 0)
    G = 4
    expect = P.bits(case["v_new"]).repeat(G, axis=1)       # head i reads KV head i // G
    assert np.array_equal(P.bits(out), expect)


@pytest.mark.parametrize("path", [1, 2, 3])
def test_identical_queries_in_a_group_give_identical_outputs(mqa, path):
    case = P.make_case(2, 8, 2, 128, 100, 900, seed_id=402)
    q = case["q"].clone()
    q[:, 1] = q[:, 0]
    q[:, 7] = q[:, 5]
    case["q"] = q
    mqa.debug_override(0, path)
    try:
        _, _, out = P.gpu_step(case, mqa)
    finally:
        mqa.debug_override(0, 0)
    ob = P.bits(out)
    assert np.array_equal(ob[:, 1], ob[:, 0]) and np.array_equal(ob[:, 7], ob[:, 5])


@pytest.mark.parametrize("shape", [(2, 16, 2, 128, 200, 900), (2, 64, 2, 128, 200, 900)],
                         ids=["G8", "G32"])
def test_peaked_attention_large_scale(mqa, shape):
    # scale 1.0 instead of 1/sqrt(d_h): logits spread over about +-40, softmax nearly one-hot; on
    # the tcgen05 path the running reference is raised (and O rescaled) many times
    case = P.make_case(*shape, seed_id=403)
    case["scale"] = 1.0
    _, _, out_ref = P.oracle_step(case)
    _, _, out = P.gpu_step(case, mqa)
    P.assert_close(out, out_ref, "scale 1.0")


@pytest.mark.parametrize("d_h", [64, 128])
@pytest.mark.parametrize("G", [1, 2, 3, 4, 5, 6, 7])
def test_cuda_core_path_at_every_group_size(mqa, G, d_h):
    # every CUDA-core instance: lengths from 1 (a warp's 16 keys partly valid, odd counts, the
    # last pair or quad of keys cut short) to several tiles, NaN past each length
    case = P.make_case(3, 2 * G, 2, d_h, 1, 300, seed_id=700 + 10 * G + d_h // 64, tail="nan")
    _, _, out_ref = P.oracle_step(case)
    mqa.debug_override(0, 1)   # automatic only up to G = 2
    try:
        _, _, out = P.gpu_step(case, mqa)
        assert mqa.get_device_status() == 0
    finally:
        mqa.debug_override(0, 0)
    P.assert_close(out, out_ref, f"CUDA cores G={G} d_h={d_h}")


def test_growing_logits_force_rescales_on_cuda_cores(mqa):
    # as below, on the CUDA-core consumer (G = 6): the running maximum rises tile after tile
    case = P.make_case(2, 6, 1, 128, 600, 1500, seed_id=405, tail="nan")
    k = case["k"].float()
    ramp = torch.linspace(0.2, 3.0, k.shape[2]).view(1, 1, -1, 1)
    case["k"] = (k * ramp).to(torch.bfloat16)
    case["scale"] = 0.25
    _, _, out_ref = P.oracle_step(case)
    mqa.debug_override(0, 1)
    try:
        _, _, out = P.gpu_step(case, mqa)
        assert mqa.get_device_status() == 0
    finally:
        mqa.debug_override(0, 0)
    P.assert_close(out, out_ref, "growing logits, CUDA cores")


def test_growing_logits_force_rescales(mqa):
    # keys scaled up along the sequence, so the row maximum keeps rising tile after tile
    case = P.make_case(2, 32, 1, 128, 600, 1500, seed_id=404, tail="nan")
    k = case["k"].float()
    ramp = torch.linspace(0.2, 3.0, k.shape[2]).view(1, 1, -1, 1)
    case["k"] = (k * ramp).to(torch.bfloat16)
    case["scale"] = 0.25
    _, _, out_ref = P.oracle_step(case)
    for path in (2, 3):
        mqa.debug_override(0, path)
        try:
            _, _, out = P.gpu_step(case, mqa)
            assert mqa.get_device_status() == 0
        finally:
            mqa.debug_override(0, 0)
        P.assert_close(out, out_ref, f"growing logits, path {path}")


def test_out_of_range_lengths_latch_an_error_and_write_zeros(mqa):
    case = P.make_case(4, 8, 2, 64, 10, 300, seed_id=404)
    k_ref, v_ref, out_ref = P.oracle_step(case)
    dev = torch.device("cuda")
    k, v = case["k"].to(dev), case["v"].to(dev)
    mqa.kv_append(case["k_new"].to(dev), case["v_new"].to(dev), k, v, case["pos"].to(dev))
    lens = case["lens"].clone()
    lens[1] = 0
    lens[2] = case["w"].n_max + 1
    out = torch.full_like(case["q"], 7.0).to(dev)
    mqa.decode_attention(case["q"].to(dev), k, v, lens.to(dev), out=out, scale=case["scale"])
    assert mqa.get_device_status() == 4
    assert mqa.get_device_status() == 0            # reading clears it
    ob = P.bits(out)
    assert np.all(ob[1] == 0) and np.all(ob[2] == 0)
    keep = [0, 3]
    P.assert_close(out[keep], out_ref[keep], "valid sequences next to invalid ones")


def test_out_of_range_position_latches_an_error_and_writes_nothing(mqa):
    case = P.make_case(2, 4, 2, 128, 10, 20, seed_id=405)
    dev = torch.device("cuda")
    k, v = case["k"].to(dev), case["v"].to(dev)
    k0, v0 = P.bits(k), P.bits(v)
    pos = torch.tensor([case["w"].n_max, -1], dtype=torch.int32, device=dev)
    mqa.kv_append(case["k_new"].to(dev), case["v_new"].to(dev), k, v, pos)
    assert mqa.get_device_status() == 4
    assert np.array_equal(P.bits(k), k0) and np.array_equal(P.bits(v), v0)


def test_head_shards_match_the_whole(mqa):
    # tensor parallelism over KV heads: each shard holds g/2 KV heads and their h/2 query heads;
    # no exchange is needed, the shards' outputs concatenate to the whole
    case = P.make_case(3, 16, 4, 128, 100, 800, seed_id=406)
    _, _, out_ref = P.oracle_step(case)
    dev = torch.device("cuda")
    k, v = case["k"].to(dev), case["v"].to(dev)
    mqa.kv_append(case["k_new"].to(dev), case["v_new"].to(dev), k, v, case["pos"].to(dev))
    lens, q = case["lens"].to(dev), case["q"].to(dev)
    parts = []
    for s in range(2):
        qs = q[:, 8 * s:8 * (s + 1)].contiguous()
        ks, vs = k[:, 2 * s:2 * (s + 1)].contiguous(), v[:, 2 * s:2 * (s + 1)].contiguous()
        parts.append(mqa.decode_attention(qs, ks, vs, lens, scale=case["scale"]))
    P.assert_close(torch.cat(parts, dim=1), out_ref, "head shards")


def test_two_streams_do_not_share_a_workspace(mqa):
    cases = [P.make_case(2, 16, 2, 128, 300, 900, seed_id=407 + i) for i in range(2)]
    refs = [P.oracle_step(c)[2] for c in cases]
    streams = [torch.cuda.Stream() for _ in cases]
    outs = []
    for c, s in zip(cases, streams):
        with torch.cuda.stream(s):
            outs.append(P.gpu_step(c, mqa, stream=s)[2])
    torch.cuda.synchronize()
    for o, r in zip(outs, refs):
        P.assert_close(o, r, "concurrent streams")


@pytest.mark.parametrize("ctas", [0, 1, 7])
@pytest.mark.parametrize("d_h", [64, 128])
@pytest.mark.parametrize("G", [1, 2, 3, 5, 7, 8])
def test_transposed_consumer_at_every_small_group(mqa, G, d_h, ctas):
    """Up to 8 heads per KV head, the mma.sync path runs the transposed products (heads on the
    MMA's 8 columns, padding columns past G): every G on both head sizes, with the default CTA
    count, one CTA walking every segment, and 7 CTAs splitting segments at tile boundaries."""
    case = P.make_case(3, 2 * G, 2, d_h, 1, 700, seed_id=500 + 10 * G + d_h // 64)
    _, _, out_ref = P.oracle_step(case)
    mqa.debug_override(ctas, 2)
    try:
        _, _, out = P.gpu_step(case, mqa)
        assert mqa.get_device_status() == 0
    finally:
        mqa.debug_override(0, 0)
    P.assert_close(out, out_ref, f"G={G} d_h={d_h} ctas={ctas}")
