"""GPU parity of the fp8 E4M3 cache calls (mqa_kv_append_fp8, mqa_decode_attention_fp8,
mqa_decode_step_fp8) against the fp64 oracle on the same seeded inputs.

The oracle's side: the quantized append (oracle.kv_append_fp8: e4m3(fp32(x) / scale), nearest,
ties to even, saturating) and the fp64 attention over the dequantized caches
(oracle.decode_attention_fp8: code * scale). The caches' earlier rows are seeded normal draws
quantized with torch's float8_e4m3fn conversion (a library routine), rows at or past each length
hold NaN codes, and the scales map each tensor's largest magnitude to 448. Caches are compared
byte for byte; outputs within the contract's tolerances.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from query_grouped_decode_kv_b300 import inputs
from tests import _parity as P

pytestmark = pytest.mark.gpu

BOUNDS, UNSUPPORTED = 4, 2


@pytest.fixture(scope="module")
def mqa():
    import query_grouped_decode_kv_b300 as m
    m.debug_override(0, 0)
    yield m
    m.debug_override(0, 0)


def fp8_case(shape, seed_id, lens=None, pos=None, kv_std=1.0):
    case = P.make_case(*shape, seed_id=seed_id, kv_std=kv_std)
    if lens is not None:
        case["lens"] = torch.tensor(lens, dtype=torch.int32)
        case["pos"] = torch.tensor(pos, dtype=torch.int32)
        case["k"], case["v"] = inputs.cache(case["w"], 0, "cpu", tail="nan", lengths=case["lens"])
    ks = inputs.amax_scale(torch.cat([case["k"].flatten(), case["k_new"].flatten()]))
    vs = inputs.amax_scale(torch.cat([case["v"].flatten(), case["v_new"].flatten()]))
    case.update(k_scale=ks, v_scale=vs, k8=inputs.fp8_codes(case["k"], ks),
                v8=inputs.fp8_codes(case["v"], vs))
    return case


def oracle_fp8_step(case):
    kc, vc = case["k8"].numpy().copy(), case["v8"].numpy().copy()
    st = oracle.kv_append_fp8(P.bits(case["k_new"]), P.bits(case["v_new"]), kc, vc,
                              case["pos"].numpy(), case["k_scale"], case["v_scale"])
    out, ast = oracle.decode_attention_fp8(P.bits(case["q"]), kc, vc, case["lens"].numpy(),
                                           case["k_scale"], case["v_scale"], case["scale"],
                                           return_status=True)
    return kc, vc, out, st, ast


def gpu_fp8(case, mqa, fused=True, stream=None):
    dev = torch.device("cuda")
    q = case["q"].to(dev)
    kn, vn = case["k_new"].to(dev), case["v_new"].to(dev)
    kc, vc = case["k8"].to(dev), case["v8"].to(dev)
    pos, lens = case["pos"].to(dev), case["lens"].to(dev)
    ks, vs = case["k_scale"], case["v_scale"]
    if fused:
        out = mqa.decode_step_fp8(q, kn, vn, kc, vc, pos, lens, ks, vs, scale=case["scale"],
                                  stream=stream)
    else:
        mqa.kv_append_fp8(kn, vn, kc, vc, pos, ks, vs, stream=stream)
        out = mqa.decode_attention_fp8(q, kc, vc, lens, ks, vs, scale=case["scale"],
                                       stream=stream)
    return kc, vc, out


SHAPES = [
    # b, h, g, d_h, ctx_lo, ctx_hi
    (1, 8, 1, 128, 128, 128),     # G = 8, mma.sync (four consumer warps)
    (3, 8, 2, 128, 0, 300),       # G = 4
    (3, 4, 2, 128, 0, 300),       # G = 2 (mma.sync: fp8 caches take it at every G)
    (2, 7, 1, 128, 60, 200),      # G = 7
    (2, 4, 4, 128, 60, 70),       # G = 1 (MHA) around the tile edge
    (2, 32, 2, 128, 100, 700),    # G = 16
    (2, 32, 1, 128, 1, 1000),     # G = 32, eight consumer warps
    (2, 64, 1, 128, 1, 600),      # G = 64
    (4, 64, 8, 128, 0, 513),      # G = 8, the 70B-class grouping, short ragged contexts
]


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "b{}h{}g{}d{}_{}-{}".format(*s))
@pytest.mark.parametrize("fused", [True, False], ids=["fused", "two_launches"])
def test_fp8_step_matches_oracle(mqa, shape, fused):
    case = fp8_case(shape, seed_id=1300 + SHAPES.index(shape))
    k_ref, v_ref, out_ref, st, ast = oracle_fp8_step(case)
    assert st == oracle.OK and ast == oracle.OK
    kc, vc, out = gpu_fp8(case, mqa, fused=fused)
    torch.cuda.synchronize()
    assert mqa.get_device_status() == 0
    assert np.array_equal(kc.cpu().numpy(), k_ref), "K codes differ from the oracle's append"
    assert np.array_equal(vc.cpu().numpy(), v_ref), "V codes differ from the oracle's append"
    P.assert_close(out, out_ref, f"fp8 {shape}")


@pytest.mark.parametrize("ctas", [1, 2, 3, 7, 64, 148, 1000])
@pytest.mark.parametrize("shape,path", [((2, 16, 2, 128, 0, 700), 0), ((3, 8, 4, 128, 100, 400), 1),
                                        ((3, 8, 4, 128, 100, 400), 0), ((2, 64, 2, 128, 0, 700), 0)],
                         ids=["mma_sync", "cuda_cores", "mma_sync_G2", "mma_sync_G32"])
def test_fp8_any_cta_split(mqa, shape, path, ctas):
    case = fp8_case(shape, seed_id=1320)
    k_ref, v_ref, out_ref, _, _ = oracle_fp8_step(case)
    mqa.debug_override(ctas, path)
    try:
        kc, vc, out = gpu_fp8(case, mqa)
        assert mqa.get_device_status() == 0
    finally:
        mqa.debug_override(0, 0)
    assert np.array_equal(kc.cpu().numpy(), k_ref) and np.array_equal(vc.cpu().numpy(), v_ref)
    P.assert_close(out, out_ref, f"fp8 {shape} ctas={ctas}")


@pytest.mark.parametrize("path", [1, 2])
@pytest.mark.parametrize("ctas", [0, 1, 5])
def test_fp8_append_row_anywhere(mqa, path, ctas):
    # the last attended row; inside the attended range; past the length inside the last loaded
    # tile; past every loaded tile; out of range (skipped, latched); the first row of a tile
    lens = [200, 300, 100, 70, 150, 129]
    case = fp8_case((6, 8, 2, 128, 60, 300), 1330, lens=lens,
                    pos=[199, 37, 110, 250, 301, 128])
    k_ref, v_ref, out_ref, st, ast = oracle_fp8_step(case)
    assert st == oracle.ERR_BOUNDS and ast == oracle.OK
    mqa.debug_override(ctas, path)
    try:
        kc, vc, out = gpu_fp8(case, mqa)
        assert mqa.get_device_status() == BOUNDS
    finally:
        mqa.debug_override(0, 0)
    assert np.array_equal(kc.cpu().numpy(), k_ref) and np.array_equal(vc.cpu().numpy(), v_ref)
    P.assert_close(out, out_ref, f"fp8 append rows anywhere, path {path}, ctas {ctas}")


def test_fp8_append_saturates_and_rounds_like_the_oracle(mqa):
    # new rows far beyond the scale's range (saturate at +-448), tiny values (subnormal codes and
    # rounding to zero) and exact ties of the E4M3 grid
    case = fp8_case((2, 16, 2, 128, 50, 90), 1340)
    # power-of-two scales keep x / scale exact, so 17 and 3 * 2^-10 are exact ties of the grid
    case["k_scale"], case["v_scale"] = 2.0 ** -4, 2.0 ** -3
    case["k8"] = inputs.fp8_codes(case["k"], case["k_scale"])
    case["v8"] = inputs.fp8_codes(case["v"], case["v_scale"])
    g = case["k_new"].shape[1]
    vals = torch.tensor([1e4, -1e4, 449.0, 3 * 2.0 ** -10, 2.0 ** -10, 17.0, 18.0, 0.0],
                        dtype=torch.float32)
    pattern = vals.repeat(2 * g * 128 // vals.numel() + 1)[: 2 * g * 128].view(2, g, 128)
    case["k_new"] = (pattern * case["k_scale"]).to(torch.bfloat16)
    case["v_new"] = (-pattern * case["v_scale"]).to(torch.bfloat16)
    k_ref, v_ref, out_ref, _, _ = oracle_fp8_step(case)
    kc, vc, out = gpu_fp8(case, mqa, fused=False)
    assert mqa.get_device_status() == 0
    assert np.array_equal(kc.cpu().numpy(), k_ref) and np.array_equal(vc.cpu().numpy(), v_ref)
    kc2, vc2, _ = gpu_fp8(case, mqa, fused=True)
    assert np.array_equal(kc2.cpu().numpy(), k_ref) and np.array_equal(vc2.cpu().numpy(), v_ref)


def test_fp8_scales_are_applied(mqa):
    # scaling both tensors' scales by powers of two scales the logits and the outputs exactly
    case = fp8_case((2, 16, 1, 128, 300, 300), 1350)
    dev = torch.device("cuda")
    # no append here: attend over the context rows only (the append row still holds NaN codes)
    ctx = case["lens"] - 1
    q, lens = case["q"].to(dev), ctx.to(dev)
    kc, vc = case["k8"].to(dev), case["v8"].to(dev)
    ks, vs = case["k_scale"], case["v_scale"]
    a = mqa.decode_attention_fp8(q, kc, vc, lens, ks, vs, scale=case["scale"])
    b = mqa.decode_attention_fp8(q, kc, vc, lens, ks * 2, vs * 4, scale=case["scale"] / 2)
    torch.cuda.synchronize()
    assert mqa.get_device_status() == 0
    assert torch.isfinite(a.float()).all()
    assert torch.equal(b.float(), (a.float() * 4))
    ref = oracle.decode_attention_fp8(P.bits(case["q"]), case["k8"].numpy(), case["v8"].numpy(),
                                      ctx.numpy(), ks, vs, case["scale"])
    P.assert_close(a, ref, "fp8 scales")


def test_fp8_rejects_the_tcgen05_path(mqa):
    case = fp8_case((1, 32, 1, 128, 100, 100), 1360)
    mqa.debug_override(0, 3)
    try:
        with pytest.raises(mqa.MqaError) as e:
            gpu_fp8(case, mqa)
        assert e.value.status == UNSUPPORTED
    finally:
        mqa.debug_override(0, 0)


def test_fp8_caches_may_be_float8_tensors(mqa):
    case = fp8_case((2, 16, 2, 128, 100, 400), 1370)
    _, _, out_ref, _, _ = oracle_fp8_step(case)
    dev = torch.device("cuda")
    kc = case["k8"].to(dev).view(torch.float8_e4m3fn)
    vc = case["v8"].to(dev).view(torch.float8_e4m3fn)
    out = mqa.decode_step_fp8(case["q"].to(dev), case["k_new"].to(dev), case["v_new"].to(dev),
                              kc, vc, case["pos"].to(dev), case["lens"].to(dev),
                              case["k_scale"], case["v_scale"], scale=case["scale"])
    assert mqa.get_device_status() == 0
    P.assert_close(out, out_ref, "float8 tensors")


def test_fp8_invalid_length_writes_zeros(mqa):
    case = fp8_case((4, 16, 2, 128, 10, 300), 1380)
    lens = case["lens"].clone()
    lens[2] = 0
    case["lens"] = lens
    k_ref, v_ref, out_ref, _, _ = oracle_fp8_step(case)
    kc, vc, out = gpu_fp8(case, mqa)
    assert mqa.get_device_status() == BOUNDS
    assert np.array_equal(kc.cpu().numpy(), k_ref) and np.array_equal(vc.cpu().numpy(), v_ref)
    assert np.all(P.bits(out)[2] == 0)
    keep = [0, 1, 3]
    P.assert_close(out[keep], out_ref[keep], "valid sequences next to an invalid one")


def test_fp8_layers_through_the_multi_layer_driver(mqa):
    # three fp8 layers (each with its own scales) through layers.decode_layers, fused and not
    from query_grouped_decode_kv_b300.layers import LayerState, StepInputs, decode_layers
    dev = torch.device("cuda")
    for fused in (True, False):
        c0 = fp8_case((3, 32, 4, 128, 50, 600), 1400)
        cases = [c0] + [fp8_case((3, 32, 4, 128, 50, 600), 1400 + li, lens=c0["lens"].tolist(),
                                 pos=c0["pos"].tolist()) for li in (1, 2)]
        lays = [LayerState(c["k8"].to(dev), c["v8"].to(dev), fp8_scales=(c["k_scale"], c["v_scale"]))
                for c in cases]
        xs = [StepInputs(c["q"].to(dev), c["k_new"].to(dev), c["v_new"].to(dev)) for c in cases]
        outs = [torch.empty_like(x.q) for x in xs]
        pos, lens = cases[0]["pos"].to(dev), cases[0]["lens"].to(dev)
        assert all(torch.equal(c["lens"], cases[0]["lens"]) for c in cases)
        decode_layers(lays, xs, pos, lens, outs, cases[0]["scale"], fused=fused)
        torch.cuda.synchronize()
        assert mqa.get_device_status() == 0
        for c, lay, o in zip(cases, lays, outs):
            k_ref, v_ref, out_ref, _, _ = oracle_fp8_step(c)
            assert np.array_equal(lay.k_cache.cpu().numpy(), k_ref)
            assert np.array_equal(lay.v_cache.cpu().numpy(), v_ref)
            P.assert_close(o, out_ref, f"fp8 layers fused={fused}")
