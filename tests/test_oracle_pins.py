"""Pins for the CPU oracle: each test fixes an oracle function to something other than itself --
numbers printed on the pages, closed forms, invariants of the definition, special cases that reduce
to a library routine, and brute force on tiny inputs. A plausible slip in the oracle (a dropped
scale, a wrong sign, a transposed operand, a strided instead of contiguous head->group map, an
off-by-one length, a missing normalisation) fails at least one of these.

CPU only (no GPU marker).
"""
from __future__ import annotations

import json
import math
import os

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# --------------------------------------------------------------------------------------------
# KV-cache size formula: the pages' printed figures
# --------------------------------------------------------------------------------------------
def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


@pytest.mark.parametrize("case", _golden("kv_cache_bytes.json")["cases"], ids=lambda c: c["id"])
def test_kv_bytes_matches_page_figures(case):
    got = oracle.kv_cache_bytes(**case["args"])
    assert got == math.prod(case["printed_factors"])
    if case.get("printed_value_is_wrong"):
        # the page's decimal point slipped by one place: the product is ten times the print
        assert got == pytest.approx(10 * case["printed_value"], rel=0.01)
        assert got != pytest.approx(case["printed_value"], rel=0.5)
    else:
        assert got == pytest.approx(case["printed_value"], rel=case["printed_rel_tol"])


@pytest.mark.parametrize("ratio", _golden("kv_cache_bytes.json")["ratios"], ids=lambda r: r["id"])
def test_kv_bytes_group_ratio(ratio):
    full = oracle.kv_cache_bytes(1, ratio["h"], 4096, 128, 2)
    grouped = oracle.kv_cache_bytes(1, ratio["g"], 4096, 128, 2)
    if "mha_over_gqa" in ratio:
        assert full / grouped == ratio["mha_over_gqa"]
    else:
        assert 100.0 * grouped / full == pytest.approx(ratio["percent_of_mha"],
                                                       abs=ratio["printed_abs_tol"])


def test_kv_bytes_80_layer_workload_allocation():
    # 80 layers, g=8, 32769 rows (32768 context + the appended token), d_h=128, bf16, 8 sequences:
    # the 70B-class decode workload holds about 86 GB of cache.
    per_seq = oracle.kv_cache_bytes(80, 8, 32769, 128, 2)
    assert 8 * per_seq == 85_901_967_360


# --------------------------------------------------------------------------------------------
# bfloat16 conversions: against IEEE float32 reinterpretation and torch's rounding
# --------------------------------------------------------------------------------------------
def test_bf16_widening_all_patterns():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ours = oracle.bf16_to_f64(bits)
    # library route: a bf16 pattern is the upper half of an IEEE binary32
    with np.errstate(invalid="ignore"):
        ref = (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])


def test_bf16_rounding_ties_and_edges():
    one_ulp = 2.0 ** -7
    cases = [
        (1.0, 0x3F80),
        (1.0 + one_ulp / 2, 0x3F80),           # tie -> even (down)
        (1.0 + 3 * one_ulp / 2, 0x3F82),       # tie -> even (up)
        (1.0 + one_ulp / 2 + 2.0 ** -30, 0x3F81),  # just above the tie
        (-2.0, 0xC000),
        (0.0, 0x0000),
        (-0.0, 0x8000),
        (2.0 ** -133, 0x0001),                 # smallest subnormal
        (2.0 ** -134, 0x0000),                 # tie between 0 and the smallest subnormal -> even
        (3 * 2.0 ** -134, 0x0002),             # tie between 1 and 2 subnormal units -> even
        ((2 - 2.0 ** -7) * 2.0 ** 127, 0x7F7F),   # largest finite
        ((2 - 2.0 ** -8) * 2.0 ** 127, 0x7F80),   # tie at the top rounds to infinity
        (math.inf, 0x7F80),
        (-math.inf, 0xFF80),
    ]
    got = oracle.f64_to_bf16([x for x, _ in cases])
    assert [int(x) for x in got] == [bits for _, bits in cases]
    assert int(oracle.f64_to_bf16([math.nan])[0]) & 0x7F80 == 0x7F80


def test_bf16_rounding_matches_torch_on_float32_values():
    rng = np.random.default_rng(5)
    x = np.concatenate([rng.standard_normal(4000) * 10.0 ** rng.integers(-30, 30, 4000),
                        rng.standard_normal(1000)]).astype(np.float32)
    ours = oracle.f64_to_bf16(x.astype(np.float64))
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)


# --------------------------------------------------------------------------------------------
# KV append
# --------------------------------------------------------------------------------------------
def test_append_writes_exactly_one_row_per_kv_head():
    rng = np.random.default_rng(1)
    b, g, n_max, d_h = 3, 2, 9, 64
    kc = rng.integers(0, 65536, (b, g, n_max, d_h), dtype=np.uint16)
    vc = rng.integers(0, 65536, (b, g, n_max, d_h), dtype=np.uint16)
    kn = rng.integers(0, 65536, (b, g, d_h), dtype=np.uint16)
    vn = rng.integers(0, 65536, (b, g, d_h), dtype=np.uint16)
    pos = np.array([0, 8, 4], dtype=np.int32)
    k0, v0 = kc.copy(), vc.copy()
    assert oracle.kv_append(kn, vn, kc, vc, pos) == oracle.OK
    for bi in range(b):
        assert np.array_equal(kc[bi, :, pos[bi]], kn[bi])
        assert np.array_equal(vc[bi, :, pos[bi]], vn[bi])
    mask = np.ones((b, g, n_max), dtype=bool)
    for bi in range(b):
        mask[bi, :, pos[bi]] = False
    assert np.array_equal(kc[mask], k0[mask]) and np.array_equal(vc[mask], v0[mask])


def test_append_rejects_out_of_range_positions_without_writing():
    rng = np.random.default_rng(2)
    b, g, n_max, d_h = 2, 1, 4, 64
    kc = rng.integers(0, 65536, (b, g, n_max, d_h), dtype=np.uint16)
    vc = kc.copy()
    kn = rng.integers(0, 65536, (b, g, d_h), dtype=np.uint16)
    k0 = kc.copy()
    st = oracle.kv_append(kn, kn, kc, vc, np.array([4, -1], dtype=np.int32))
    assert st == oracle.ERR_BOUNDS
    assert np.array_equal(kc, k0)


# --------------------------------------------------------------------------------------------
# Attention: closed forms
# --------------------------------------------------------------------------------------------
def _f64_case(b, h, g, d_h, n_max, seed=0):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((b, h, d_h))
    k = rng.standard_normal((b, g, n_max, d_h))
    v = rng.standard_normal((b, g, n_max, d_h))
    return q, k, v


def test_closed_form_two_keys():
    # q = (1, 0); keys (0, 0) and (ln 3, 0), scale 1 -> weights 1/4, 3/4;
    # values (1, 0) and (0, 1) -> output (1/4, 3/4).
    q = np.array([[[1.0, 0.0]]])
    k = np.array([[[[0.0, 0.0], [math.log(3.0), 0.0]]]])
    v = np.array([[[[1.0, 0.0], [0.0, 1.0]]]])
    out = oracle.decode_attention(q, k, v, np.array([2], np.int32), scale=1.0)
    assert out[0, 0] == pytest.approx([0.25, 0.75], abs=1e-15)
    # the scale multiplies the logit: scale 2 -> weights 1/10, 9/10
    out2 = oracle.decode_attention(q, k, v, np.array([2], np.int32), scale=2.0)
    assert out2[0, 0] == pytest.approx([0.1, 0.9], abs=1e-15)
    # a negative query flips the preference: weights 3/4, 1/4
    out3 = oracle.decode_attention(-q, k, v, np.array([2], np.int32), scale=1.0)
    assert out3[0, 0] == pytest.approx([0.75, 0.25], abs=1e-15)


def test_closed_form_with_huge_logits():
    # logits 1000 and 1000 + ln 3: exp() of either overflows a double, the softmax does not --
    # weights are still 1/4 and 3/4
    q = np.array([[[1.0, 0.0]]])
    k = np.array([[[[1000.0, 0.0], [1000.0 + math.log(3.0), 0.0]]]])
    v = np.array([[[[1.0, 0.0], [0.0, 1.0]]]])
    out = oracle.decode_attention(q, k, v, np.array([2], np.int32), scale=1.0)
    assert out[0, 0] == pytest.approx([0.25, 0.75], abs=1e-12)


def test_closed_form_head_to_group_map_is_contiguous():
    # h=4, g=2: heads 0,1 read KV head 0 and heads 2,3 read KV head 1 (j = i // (h/g)).
    # KV head 0 values are all (1, 0); KV head 1 values are all (0, 1).
    b, h, g, d_h, n = 1, 4, 2, 2, 3
    q = np.random.default_rng(3).standard_normal((b, h, d_h))
    k = np.random.default_rng(4).standard_normal((b, g, n, d_h))
    v = np.zeros((b, g, n, d_h))
    v[0, 0, :, 0] = 1.0
    v[0, 1, :, 1] = 1.0
    out = oracle.decode_attention(q, k, v, np.array([n], np.int32), scale=0.7)
    expect = np.array([[1, 0], [1, 0], [0, 1], [0, 1]], dtype=float)
    assert np.allclose(out[0], expect, atol=1e-15)


def test_weights_sum_to_one():
    q, k, _ = _f64_case(2, 8, 2, 64, 37, seed=7)
    v = np.ones_like(k)
    out = oracle.decode_attention(q, k, v, np.array([37, 5], np.int32), scale=0.3)
    assert np.allclose(out, 1.0, atol=1e-14)


def test_identical_keys_give_mean_of_values():
    q, _, v = _f64_case(1, 4, 1, 64, 20, seed=8)
    k = np.broadcast_to(np.random.default_rng(9).standard_normal(64), (1, 1, 20, 64)).copy()
    L = 13
    out = oracle.decode_attention(q, k, v, np.array([L], np.int32), scale=0.125)
    assert np.allclose(out[0], v[0, 0, :L].mean(axis=0), atol=1e-14)


def test_zero_scale_gives_mean_of_values():
    q, k, v = _f64_case(2, 4, 2, 64, 11, seed=10)
    out = oracle.decode_attention(q, k, v, np.array([11, 3], np.int32), scale=0.0)
    for bi, L in enumerate((11, 3)):
        for i in range(4):
            assert np.allclose(out[bi, i], v[bi, i // 2, :L].mean(axis=0), atol=1e-14)


def test_one_dominant_key_selects_its_value():
    q, k, v = _f64_case(1, 2, 1, 64, 16, seed=11)
    t_star = 9
    k[0, 0, t_star] = 40.0 * q[0, 0] / np.linalg.norm(q[0, 0])  # logit ~ 40|q| above the rest
    out = oracle.decode_attention(q, k, v, np.array([16], np.int32), scale=1.0)
    assert np.allclose(out[0, 0], v[0, 0, t_star], atol=1e-9)


def test_single_row_returns_that_value_exactly():
    rng = np.random.default_rng(12)
    b, h, g, d_h, n_max = 2, 8, 2, 128, 4
    q = rng.integers(0, 65536, (b, h, d_h), dtype=np.uint16) & 0xBFFF  # finite values
    k = rng.integers(0, 65536, (b, g, n_max, d_h), dtype=np.uint16) & 0xBFFF
    v = rng.integers(0, 65536, (b, g, n_max, d_h), dtype=np.uint16) & 0xBFFF
    out = oracle.decode_attention(q, k, v, np.array([1, 1], np.int32), scale=0.088)
    for bi in range(b):
        for i in range(h):
            assert np.array_equal(out[bi, i], oracle.bf16_to_f64(v[bi, i // 4, 0]))


def test_rows_beyond_length_are_never_read():
    q, k, v = _f64_case(2, 4, 1, 64, 12, seed=13)
    lens = np.array([7, 12], np.int32)
    ref = oracle.decode_attention(q, k, v, lens, scale=0.2)
    k2, v2 = k.copy(), v.copy()
    k2[0, :, 7:] = np.nan
    v2[0, :, 7:] = np.inf
    out = oracle.decode_attention(q, k2, v2, lens, scale=0.2)
    assert np.array_equal(out, ref)


def test_shifting_every_key_by_one_vector_changes_nothing():
    # q.(K_t + c) = q.K_t + q.c: a per-row constant added to every logit cancels in softmax
    q, k, v = _f64_case(1, 4, 2, 64, 25, seed=14)
    c = np.random.default_rng(15).standard_normal(64) * 3.0
    a = oracle.decode_attention(q, k, v, np.array([25], np.int32), scale=0.5)
    bshift = oracle.decode_attention(q, k + c, v, np.array([25], np.int32), scale=0.5)
    assert np.allclose(a, bshift, atol=1e-12)


def test_length_out_of_range_is_an_error_with_zero_output():
    q, k, v = _f64_case(2, 2, 1, 64, 5, seed=16)
    out, st = oracle.decode_attention(q, k, v, np.array([0, 6], np.int32), scale=1.0,
                                      return_status=True)
    assert st == oracle.ERR_BOUNDS
    assert np.all(out == 0.0)


def test_uneven_grouping_is_rejected():
    q, k, v = _f64_case(1, 6, 4, 64, 3)
    with pytest.raises(ValueError):
        oracle.decode_attention(q, k, v, np.array([3], np.int32), scale=1.0)


# --------------------------------------------------------------------------------------------
# Attention: reductions to MHA / MQA, and library routines
# --------------------------------------------------------------------------------------------
def test_g_equals_h_is_independent_single_head_attention():
    b, h, d_h, n = 2, 4, 64, 10
    q, k, v = _f64_case(b, h, h, d_h, n, seed=17)
    lens = np.array([10, 6], np.int32)
    full = oracle.decode_attention(q, k, v, lens, scale=0.125)
    for i in range(h):
        single = oracle.decode_attention(q[:, i:i + 1], k[:, i:i + 1], v[:, i:i + 1], lens,
                                         scale=0.125)
        assert np.array_equal(full[:, i:i + 1], single)


def test_g_equals_one_shares_kv_across_every_head():
    b, h, d_h, n = 1, 8, 64, 10
    q, k, v = _f64_case(b, h, 1, d_h, n, seed=18)
    q[:, 5] = q[:, 2]                                 # two heads ask the same question
    out = oracle.decode_attention(q, k, v, np.array([n], np.int32), scale=0.125)
    assert np.array_equal(out[0, 5], out[0, 2])
    for i in range(h):
        single = oracle.decode_attention(q[:, i:i + 1], k, v, np.array([n], np.int32),
                                         scale=0.125)
        assert np.array_equal(out[:, i:i + 1], single)


@pytest.mark.parametrize("h,g,d_h", [(8, 1, 64), (8, 2, 64), (8, 8, 128), (4, 2, 128),
                                     (6, 3, 64)])
def test_matches_torch_sdpa_with_grouped_kv(h, g, d_h):
    # library route: torch's scaled_dot_product_attention in float64 with enable_gqa, whose
    # KV-head expansion is repeat_interleave over contiguous head groups (the ybb.press page's
    # reference module, §八)
    b, n_max = 2, 17
    q, k, v = _f64_case(b, h, g, d_h, n_max, seed=h * 100 + g * 10 + d_h)
    lens = np.array([17, 9], np.int32)
    scale = 1.0 / math.sqrt(d_h)
    out = oracle.decode_attention(q, k, v, lens, scale=scale)
    for bi in range(b):
        L = int(lens[bi])
        qt = torch.from_numpy(q[bi][:, None, :])          # [h, 1, d]
        kt = torch.from_numpy(k[bi][:, :L])               # [g, L, d]
        vt = torch.from_numpy(v[bi][:, :L])
        ref = torch.nn.functional.scaled_dot_product_attention(
            qt[None], kt[None], vt[None], scale=scale, enable_gqa=True)[0, :, 0]
        assert np.allclose(out[bi], ref.numpy(), atol=1e-12, rtol=0)


def test_matches_repeat_interleave_einsum_formulation():
    # the ybb.press page's §八 module expands the g KV heads to h with repeat_interleave, then
    # takes einsum logits, softmax and an einsum with the values; restated here in float64
    b, h, g, d_h, n = 1, 8, 2, 64, 13
    q, k, v = _f64_case(b, h, g, d_h, n, seed=19)
    scale = 1.0 / math.sqrt(d_h)
    out = oracle.decode_attention(q, k, v, np.array([n], np.int32), scale=scale)
    qt = torch.from_numpy(q)[:, None]                    # [B, T=1, h, d]
    krep = torch.from_numpy(k[0]).repeat_interleave(h // g, dim=0)   # [h, L, d]
    vrep = torch.from_numpy(v[0]).repeat_interleave(h // g, dim=0)
    scores = torch.einsum("bthd,hld->bhtl", qt, krep) * scale
    attn = torch.softmax(scores, dim=-1)
    ref = torch.einsum("bhtl,hld->bthd", attn, vrep)[:, 0]
    assert np.allclose(out, ref.numpy(), atol=1e-12, rtol=0)


def test_bf16_inputs_are_widened_exactly():
    rng = np.random.default_rng(20)
    b, h, g, d_h, n = 1, 4, 2, 64, 9
    q = oracle.f64_to_bf16(rng.standard_normal((b, h, d_h)))
    k = oracle.f64_to_bf16(rng.standard_normal((b, g, n, d_h)))
    v = oracle.f64_to_bf16(rng.standard_normal((b, g, n, d_h)))
    lens = np.array([n], np.int32)
    a = oracle.decode_attention(q, k, v, lens, scale=0.125)
    wide = [(x.astype(np.uint32) << 16).view(np.float32).astype(np.float64) for x in (q, k, v)]
    bref = oracle.decode_attention(*wide, lens, scale=0.125)
    assert np.array_equal(a, bref)


def test_brute_force_tiny_shapes_against_python_loops():
    # pure-Python loops, straight from the definition, on very small shapes
    for (b, h, g, d_h, n_max, seed) in [(1, 2, 1, 64, 3, 21), (2, 4, 2, 64, 5, 22),
                                        (2, 2, 2, 128, 4, 23)]:
        q, k, v = _f64_case(b, h, g, d_h, n_max, seed=seed)
        lens = np.array([n_max - bi for bi in range(b)], np.int32)
        out = oracle.decode_attention(q, k, v, lens, scale=0.3)
        for bi in range(b):
            for i in range(h):
                j = i // (h // g)
                L = int(lens[bi])
                logits = [0.3 * sum(q[bi, i, d] * k[bi, j, t, d] for d in range(d_h))
                          for t in range(L)]
                z = sum(math.exp(x) for x in logits)
                for d in range(0, d_h, 17):
                    o = sum(math.exp(logits[t]) / z * v[bi, j, t, d] for t in range(L))
                    assert out[bi, i, d] == pytest.approx(o, abs=1e-12)


# --------------------------------------------------------------------------------------------
# Split-sequence partials and the log-sum-exp merge
# --------------------------------------------------------------------------------------------
def test_merge_of_partials_equals_whole_range():
    b, h, g, d_h, n = 2, 8, 2, 64, 40
    q, k, v = _f64_case(b, h, g, d_h, n, seed=24)
    scale = 0.125
    full = oracle.decode_attention(q, k, v, np.array([n, n], np.int32), scale=scale)
    for cuts in ([0, 40], [0, 1, 40], [0, 13, 14, 27, 40], [0, 0, 20, 20, 40]):
        parts = [oracle.attention_partial(q, k, v, scale, lo, hi)
                 for lo, hi in zip(cuts[:-1], cuts[1:])]
        m = np.stack([p[0] for p in parts]); l = np.stack([p[1] for p in parts])
        o = np.stack([p[2] for p in parts])
        for bi in range(b):
            for i in range(h):
                merged = oracle.lse_merge(m[:, bi, i], l[:, bi, i], o[:, bi, i])
                assert np.allclose(merged, full[bi, i], atol=1e-13)


def test_merge_closed_form_with_huge_logits():
    # partial maxima 1000 and 1000 + ln 3 with unit sums: combination weights 1/3 and 1
    m = np.array([1000.0, 1000.0 + math.log(3.0)])
    l = np.array([1.0, 1.0])
    o = np.array([[1.0, 0.0], [0.0, 1.0]])
    assert oracle.lse_merge(m, l, o) == pytest.approx([0.25, 0.75], abs=1e-12)


def test_single_partial_normalises_and_empty_partials_carry_no_weight():
    q, k, v = _f64_case(1, 1, 1, 64, 6, seed=25)
    m, l, o = oracle.attention_partial(q, k, v, 0.5, 0, 6)
    me, le, oe = oracle.attention_partial(q, k, v, 0.5, 3, 3)
    assert me[0, 0] == -math.inf and le[0, 0] == 0.0 and not oe.any()
    one = oracle.lse_merge(m[0], l[0], o[0])
    assert np.allclose(one, o[0, 0] / l[0, 0], atol=1e-15)
    two = oracle.lse_merge(np.concatenate([m[0], me[0]]), np.concatenate([l[0], le[0]]),
                           np.concatenate([o[0], oe[0]]))
    assert np.array_equal(one, two)


# ------------------------------------------------------------------------------------------------
# Paged cache (nanhubrain.csdn.net MQA article §3.3, vLLM's 16-token blocks; ybb.press §十 item 12)
# ------------------------------------------------------------------------------------------------
def _paged_layout(b=2, g=2, max_pages=5, page_size=4, d_h=8, spare=3, seed=7):
    """A contiguous cache C [b, g, max_pages * page_size, d_h] and the same rows cut into pages
    by numpy reshapes alone, scattered over a pool with spare pages by a random permutation."""
    rng = np.random.default_rng(seed)
    n = max_pages * page_size
    C = rng.integers(0, 1 << 16, size=(b, g, n, d_h), dtype=np.uint16)
    blocks = C.reshape(b, g, max_pages, page_size, d_h).transpose(0, 2, 1, 3, 4)
    blocks = blocks.reshape(b * max_pages, g, page_size, d_h)
    num_pages = b * max_pages + spare
    slot = rng.permutation(num_pages)[:b * max_pages]
    pool = rng.integers(0, 1 << 16, size=(num_pages, g, page_size, d_h), dtype=np.uint16)
    pool[slot] = blocks
    table = slot.reshape(b, max_pages).astype(np.int32)
    return C, pool, table


@pytest.mark.parametrize("page_size", [1, 4, 16])
def test_paged_gather_undoes_an_independent_paging(page_size):
    C, pool, table = _paged_layout(page_size=page_size)
    got, st = oracle.gather_pages(pool, table, page_size)
    assert st == oracle.OK
    assert np.array_equal(got, C)


def test_paged_gather_reports_a_page_index_out_of_range():
    C, pool, table = _paged_layout()
    table = table.copy()
    table[1, 2] = pool.shape[0]          # one past the pool
    got, st = oracle.gather_pages(pool, table, 4)
    assert st == oracle.ERR_BOUNDS
    assert np.all(got[1, :, 8:12] == 0)  # the rows of that page
    assert np.array_equal(got[0], C[0]) and np.array_equal(got[1, :, :8], C[1, :, :8])


def test_paged_append_matches_the_contiguous_append():
    C, kpool, table = _paged_layout(seed=8)
    _, vpool, _ = _paged_layout(seed=8)
    rng = np.random.default_rng(9)
    kn = rng.integers(0, 1 << 16, size=(2, 2, 8), dtype=np.uint16)
    vn = rng.integers(0, 1 << 16, size=(2, 2, 8), dtype=np.uint16)
    pos = np.array([13, 6], dtype=np.int32)
    kc, _ = oracle.gather_pages(kpool, table, 4)
    vc, _ = oracle.gather_pages(vpool, table, 4)
    assert oracle.kv_append(kn, vn, kc, vc, pos) == oracle.OK
    kp, vp = kpool.copy(), vpool.copy()
    assert oracle.kv_append_paged(kn, vn, kp, vp, pos, table) == oracle.OK
    assert np.array_equal(oracle.gather_pages(kp, table, 4)[0], kc)
    assert np.array_equal(oracle.gather_pages(vp, table, 4)[0], vc)
    # pages no sequence maps stay as they were
    unused = sorted(set(range(kpool.shape[0])) - set(table.ravel().tolist()))
    assert np.array_equal(kp[unused], kpool[unused])


def test_paged_append_rejects_a_bad_position_or_page_without_writing():
    _, kpool, table = _paged_layout(seed=10)
    vpool = kpool.copy()
    kn = np.ones((2, 2, 8), dtype=np.uint16)
    t2 = table.copy()
    t2[0, 3] = -1
    for pos, tb in ((np.array([20, 0], dtype=np.int32), table),    # past max_pages * page_size
                    (np.array([13, -1], dtype=np.int32), table),   # negative
                    (np.array([13, 99], dtype=np.int32), t2)):     # page index -1, then bad pos
        kp, vp = kpool.copy(), vpool.copy()
        st = oracle.kv_append_paged(kn, kn, kp, vp, pos, tb)
        assert st == oracle.ERR_BOUNDS
    kp, vp = kpool.copy(), vpool.copy()
    assert oracle.kv_append_paged(kn, kn, kp, vp, np.array([13, 20], dtype=np.int32),
                                  t2) == oracle.ERR_BOUNDS
    assert np.array_equal(kp, kpool) and np.array_equal(vp, vpool)


def _paged_u8_layout(b=2, g=2, max_pages=5, page_size=4, d_h=8, spare=3, seed=7):
    """_paged_layout for one-byte codes: a contiguous C and the same rows cut into pages by
    numpy reshapes alone, scattered over a pool by a random permutation."""
    rng = np.random.default_rng(seed)
    n = max_pages * page_size
    C = rng.integers(0, 256, size=(b, g, n, d_h), dtype=np.uint8)
    blocks = C.reshape(b, g, max_pages, page_size, d_h).transpose(0, 2, 1, 3, 4)
    blocks = blocks.reshape(b * max_pages, g, page_size, d_h)
    num_pages = b * max_pages + spare
    slot = rng.permutation(num_pages)[:b * max_pages]
    pool = rng.integers(0, 256, size=(num_pages, g, page_size, d_h), dtype=np.uint8)
    pool[slot] = blocks
    return C, pool, slot.reshape(b, max_pages).astype(np.int32)


@pytest.mark.parametrize("page_size", [1, 4, 16])
def test_code_gather_undoes_an_independent_paging(page_size):
    C, pool, table = _paged_u8_layout(page_size=page_size)
    got, st = oracle.gather_pages_u8(pool, table, page_size)
    assert st == oracle.OK and np.array_equal(got, C)
    t2 = table.copy()
    t2[0, 1] = -3                        # a page index out of range: code 0 there
    got, st = oracle.gather_pages_u8(pool, t2, page_size)
    assert st == oracle.ERR_BOUNDS
    assert np.all(got[0, :, page_size:2 * page_size] == 0)
    assert np.array_equal(got[1], C[1])


def test_paged_append_of_several_tokens_matches_the_contiguous_one():
    # T = 3 tokens from rows 6 and 11 of 4-row pages: the rows cross a page boundary
    C, kpool, table = _paged_layout(seed=20)
    _, vpool, _ = _paged_layout(seed=21)
    rng = np.random.default_rng(22)
    T = 3
    kn = rng.integers(0, 1 << 16, size=(2, T, 2, 8), dtype=np.uint16)
    vn = rng.integers(0, 1 << 16, size=(2, T, 2, 8), dtype=np.uint16)
    pos = np.array([6, 11], dtype=np.int32)
    kc, _ = oracle.gather_pages(kpool, table, 4)
    vc, _ = oracle.gather_pages(vpool, table, 4)
    assert oracle.kv_append_multi(kn, vn, kc, vc, pos) == oracle.OK
    kp, vp = kpool.copy(), vpool.copy()
    assert oracle.kv_append_paged_multi(kn, vn, kp, vp, pos, table) == oracle.OK
    assert np.array_equal(oracle.gather_pages(kp, table, 4)[0], kc)
    assert np.array_equal(oracle.gather_pages(vp, table, 4)[0], vc)
    unused = sorted(set(range(kpool.shape[0])) - set(table.ravel().tolist()))
    assert np.array_equal(kp[unused], kpool[unused])
    # T = 1 is the one-token paged append
    kp1, vp1, kp2, vp2 = kpool.copy(), vpool.copy(), kpool.copy(), vpool.copy()
    assert oracle.kv_append_paged_multi(kn[:, :1], vn[:, :1], kp1, vp1, pos, table) == oracle.OK
    assert oracle.kv_append_paged(kn[:, 0], vn[:, 0], kp2, vp2, pos, table) == oracle.OK
    assert np.array_equal(kp1, kp2) and np.array_equal(vp1, vp2)


def test_paged_append_of_several_tokens_skips_bad_rows_and_sequences():
    _, kpool, table = _paged_layout(seed=23)
    vpool = kpool.copy()
    kn = np.full((2, 3, 2, 8), 7, dtype=np.uint16)
    # sequence 1's rows 18 .. 20 run past max_pages * page_size = 20: skipped whole
    kp, vp = kpool.copy(), vpool.copy()
    st = oracle.kv_append_paged_multi(kn, kn, kp, vp, np.array([0, 18], dtype=np.int32), table)
    assert st == oracle.ERR_BOUNDS
    sel = table[1]
    assert np.array_equal(kp[sel], kpool[sel])
    assert np.all(kp[table[0, 0], :, 0:3] == 7)
    # a bad page under row 4 (page 1) of sequence 0, rows 2 .. 4: rows 2, 3 written, row 4 not
    t2 = table.copy()
    t2[0, 1] = -1
    kp, vp = kpool.copy(), vpool.copy()
    st = oracle.kv_append_paged_multi(kn, kn, kp, vp, np.array([2, 0], dtype=np.int32), t2)
    assert st == oracle.ERR_BOUNDS
    assert np.all(kp[t2[0, 0], :, 2:4] == 7)
    assert np.array_equal(kp[table[0, 1]], kpool[table[0, 1]])


def test_paged_fp8_append_matches_the_contiguous_fp8_append():
    rng = np.random.default_rng(24)
    b, g, d_h, ps, mp = 2, 2, 16, 4, 5
    num_pages = b * mp + 3
    kpool = rng.integers(0, 256, size=(num_pages, g, ps, d_h), dtype=np.uint8)
    vpool = rng.integers(0, 256, size=(num_pages, g, ps, d_h), dtype=np.uint8)
    table = rng.permutation(num_pages)[:b * mp].reshape(b, mp).astype(np.int32)
    kn = oracle.f64_to_bf16(rng.standard_normal((b, g, d_h)) * 3)
    vn = oracle.f64_to_bf16(rng.standard_normal((b, g, d_h)))
    pos = np.array([13, 6], dtype=np.int32)
    ks, vs = 0.02, 0.005
    kc, _ = oracle.gather_pages_u8(kpool, table, ps)
    vc, _ = oracle.gather_pages_u8(vpool, table, ps)
    assert oracle.kv_append_fp8(kn, vn, kc, vc, pos, ks, vs) == oracle.OK
    kp, vp = kpool.copy(), vpool.copy()
    assert oracle.kv_append_paged_fp8(kn, vn, kp, vp, pos, table, ks, vs) == oracle.OK
    assert np.array_equal(oracle.gather_pages_u8(kp, table, ps)[0], kc)
    assert np.array_equal(oracle.gather_pages_u8(vp, table, ps)[0], vc)
    # a bad page or position writes nothing
    t2 = table.copy()
    t2[0, 3] = num_pages
    kp, vp = kpool.copy(), vpool.copy()
    assert oracle.kv_append_paged_fp8(kn, vn, kp, vp, np.array([13, 20], dtype=np.int32), t2,
                                      ks, vs) == oracle.ERR_BOUNDS
    assert np.array_equal(kp, kpool) and np.array_equal(vp, vpool)


def test_paged_attention_brute_force_through_the_table():
    """Attention computed with pure-Python loops that fetch every row through the page table
    equals the oracle's attention over the gathered cache."""
    b, h, g, d_h, ps, mp = 2, 4, 2, 8, 4, 4
    rng = np.random.default_rng(11)
    num_pages = b * mp + 2
    kpool = oracle.f64_to_bf16(rng.standard_normal((num_pages, g, ps, d_h)))
    vpool = oracle.f64_to_bf16(rng.standard_normal((num_pages, g, ps, d_h)))
    q = oracle.f64_to_bf16(rng.standard_normal((b, h, d_h)))
    table = rng.permutation(num_pages)[:b * mp].reshape(b, mp).astype(np.int32)
    lens = np.array([13, 6], dtype=np.int32)
    scale = 0.37
    kc, _ = oracle.gather_pages(kpool, table, ps)
    vc, _ = oracle.gather_pages(vpool, table, ps)
    got = oracle.decode_attention(q, kc, vc, lens, scale)
    qf, kf, vf = oracle.bf16_to_f64(q), oracle.bf16_to_f64(kpool), oracle.bf16_to_f64(vpool)
    for bi in range(b):
        for i in range(h):
            j = i // (h // g)
            rows = [(int(table[bi, t // ps]), t % ps) for t in range(int(lens[bi]))]
            s = [scale * sum(qf[bi, i, d] * kf[p, j, r, d] for d in range(d_h)) for p, r in rows]
            m = max(s)
            w = [math.exp(x - m) for x in s]
            tot = sum(w)
            for d in range(d_h):
                ref = sum(wt * vf[p, j, r, d] for wt, (p, r) in zip(w, rows)) / tot
                assert abs(got[bi, i, d] - ref) <= 1e-12 * max(1.0, abs(ref))


# --------------------------------------------------------------------------------------------
# fp8 E4M3 and the quantized cache
# --------------------------------------------------------------------------------------------
def _torch_e4m3_decode(codes: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(codes, dtype=np.uint8)).view(torch.float8_e4m3fn)
    return t.float().numpy().astype(np.float64)


def test_e4m3_decode_matches_torch_on_every_code():
    codes = np.arange(256, dtype=np.uint8)
    ours, ref = oracle.e4m3_to_f64(codes), _torch_e4m3_decode(codes)
    assert np.array_equal(np.isnan(ours), np.isnan(ref))
    assert np.array_equal(ours[~np.isnan(ours)], ref[~np.isnan(ref)])
    # the format's landmarks: largest finite, smallest normal, smallest subnormal, one
    assert ours[0x7E] == 448.0 and ours[0x08] == 2.0 ** -6 and ours[0x01] == 2.0 ** -9
    assert ours[0x38] == 1.0 and ours[0xB8] == -1.0 and np.isnan(ours[0x7F])


def test_e4m3_encode_matches_torch_on_every_bf16_value_in_range():
    """Every finite bfloat16 value of magnitude <= 448 rounds to the code torch's
    float8_e4m3fn conversion gives (nearest, ties to even)."""
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    x = oracle.bf16_to_f64(bits)
    keep = np.isfinite(x) & (np.abs(x) <= 448.0)
    xs = x[keep]
    ref = torch.from_numpy(xs.astype(np.float32)).to(torch.float8_e4m3fn).view(torch.uint8)
    assert np.array_equal(oracle.f64_to_e4m3(xs), ref.numpy())


def test_e4m3_encode_is_the_nearest_code_ties_to_even():
    """Brute force over the 127 non-negative finite codes, on random values and on every
    midpoint between neighbouring codes."""
    codes = np.arange(0x7F, dtype=np.uint8)
    vals = oracle.e4m3_to_f64(codes)                      # increasing
    rng = np.random.default_rng(3)
    xs = np.concatenate([rng.uniform(0, 448, 500), np.exp(rng.uniform(-12, 6, 500)),
                         (vals[:-1] + vals[1:]) / 2])
    for x in xs:
        d = np.abs(vals - x)
        best = np.flatnonzero(d == d.min())
        want = best[0] if len(best) == 1 else [c for c in best if c % 2 == 0][0]
        assert oracle.f64_to_e4m3(np.array([x]))[0] == want, x
        assert oracle.f64_to_e4m3(np.array([-x]))[0] == (want | 0x80 if x > 0 else 0x80), x


def test_e4m3_encode_saturates_beyond_the_largest_finite_value():
    got = oracle.f64_to_e4m3(np.array([448.0, 448.5, 464.0, 1e4, np.inf, -1e4, -np.inf]))
    assert list(got) == [0x7E, 0x7E, 0x7E, 0x7E, 0x7E, 0xFE, 0xFE]


def test_fp8_append_quantizes_with_the_scale_in_binary32():
    """The codes written are e4m3(float32(x) / float32(scale)): closed forms, and the
    round trip code * scale stays within half a step of x."""
    b, g, n_max, d_h = 2, 2, 5, 8
    rng = np.random.default_rng(5)
    kn = oracle.f64_to_bf16(rng.standard_normal((b, g, d_h)) * 3.0)
    vn = oracle.f64_to_bf16(rng.standard_normal((b, g, d_h)) * 0.01)
    kc = np.zeros((b, g, n_max, d_h), dtype=np.uint8)
    vc = np.zeros_like(kc)
    pos = np.array([4, 0], dtype=np.int32)
    ks, vs = 0.05, 1.0 / 4096
    assert oracle.kv_append_fp8(kn, vn, kc, vc, pos, ks, vs) == oracle.OK
    kx, vx = oracle.bf16_to_f64(kn), oracle.bf16_to_f64(vn)
    for bi in range(b):
        for j in range(g):
            for d in range(d_h):
                for x, cache, sc in ((kx, kc, ks), (vx, vc, vs)):
                    y = np.float32(np.float32(x[bi, j, d]) / np.float32(sc))
                    code = cache[bi, j, pos[bi], d]
                    assert code == _torch_e4m3_to_code(float(y))
                    back = oracle.e4m3_to_f64(np.array([code]))[0] * np.float32(sc)
                    step = 2.0 ** (math.floor(math.log2(max(abs(y), 2.0 ** -6))) - 3) * sc
                    assert abs(back - x[bi, j, d]) <= step / 2 + 1e-12
    # every other byte is untouched
    mask = np.ones_like(kc, dtype=bool)
    for bi in range(b):
        mask[bi, :, pos[bi]] = False
    assert not kc[mask].any() and not vc[mask].any()
    # closed forms: 1.0 / 0.5 = 2 -> 0x40; 1.0 / 3.0 rounds to 11/32 -> 0x2B
    one = oracle.f64_to_bf16(np.ones((1, 1, 1)))
    for sc, want in ((0.5, 0x40), (3.0, 0x2B), (1.0 / 1024, 0x7E)):
        c1 = np.zeros((1, 1, 1, 1), dtype=np.uint8)
        c2 = np.zeros_like(c1)
        assert oracle.kv_append_fp8(one, one, c1, c2, np.array([0], np.int32), sc, sc) == 0
        assert c1[0, 0, 0, 0] == want and c2[0, 0, 0, 0] == want


def _torch_e4m3_to_code(y: float) -> int:
    if abs(y) > 448.0:
        return 0x7E | (0x80 if y < 0 else 0)
    return int(torch.tensor([y], dtype=torch.float32).to(torch.float8_e4m3fn).view(torch.uint8))


def test_fp8_append_rejects_a_bad_position_without_writing():
    kn = oracle.f64_to_bf16(np.ones((2, 1, 4)))
    kc = np.zeros((2, 1, 3, 4), dtype=np.uint8)
    vc = np.zeros_like(kc)
    st = oracle.kv_append_fp8(kn, kn, kc, vc, np.array([3, -1], np.int32), 1.0, 1.0)
    assert st == oracle.ERR_BOUNDS and not kc.any() and not vc.any()


def test_fp8_attention_brute_force_on_decoded_codes():
    """Attention over fp8 caches equals pure-Python attention over torch's decoding of the codes
    times the scales."""
    b, h, g, d_h, n_max = 2, 4, 2, 8, 6
    rng = np.random.default_rng(17)
    kc = rng.integers(0, 256, (b, g, n_max, d_h), dtype=np.uint8)
    vc = rng.integers(0, 256, (b, g, n_max, d_h), dtype=np.uint8)
    for c in (kc, vc):                                     # no NaN codes
        c[(c & 0x7F) == 0x7F] = 0x3C
    q = oracle.f64_to_bf16(rng.standard_normal((b, h, d_h)))
    lens = np.array([6, 3], dtype=np.int32)
    ks, vs, scale = 0.01, 0.25, 0.3
    got = oracle.decode_attention_fp8(q, kc, vc, lens, ks, vs, scale)
    kf, vf = _torch_e4m3_decode(kc) * ks, _torch_e4m3_decode(vc) * vs
    qf = oracle.bf16_to_f64(q)
    for bi in range(b):
        for i in range(h):
            j = i // (h // g)
            s = [scale * sum(qf[bi, i, d] * kf[bi, j, t, d] for d in range(d_h))
                 for t in range(int(lens[bi]))]
            m = max(s)
            w = [math.exp(x - m) for x in s]
            for d in range(d_h):
                ref = sum(w[t] * vf[bi, j, t, d] for t in range(len(w))) / sum(w)
                assert abs(got[bi, i, d] - ref) <= 1e-12 * max(1.0, abs(ref))


def test_fp8_scales_fold_into_the_logit_scale_and_the_output():
    """k_scale multiplies every logit and v_scale every output: doubling k_scale equals doubling
    the logit scale, and doubling v_scale doubles the output exactly."""
    b, h, g, d_h, n_max = 1, 4, 1, 16, 9
    rng = np.random.default_rng(23)
    kc = oracle.f64_to_e4m3(rng.standard_normal((b, g, n_max, d_h)) * 30)
    vc = oracle.f64_to_e4m3(rng.standard_normal((b, g, n_max, d_h)) * 30)
    q = oracle.f64_to_bf16(rng.standard_normal((b, h, d_h)))
    lens = np.array([9], dtype=np.int32)
    a = oracle.decode_attention_fp8(q, kc, vc, lens, 0.02, 0.5, 0.25)
    assert np.allclose(oracle.decode_attention_fp8(q, kc, vc, lens, 0.04, 0.5, 0.25),
                       oracle.decode_attention_fp8(q, kc, vc, lens, 0.02, 0.5, 0.5), rtol=1e-13)
    assert np.array_equal(oracle.decode_attention_fp8(q, kc, vc, lens, 0.02, 1.0, 0.25), 2 * a)


# --------------------------------------------------------------------------------------------
# T new tokens per sequence, causal
# --------------------------------------------------------------------------------------------
def _multi_case(b, T, h, g, d_h, n_max, seed):
    rng = np.random.default_rng(seed)
    q = oracle.f64_to_bf16(rng.standard_normal((b, T, h, d_h)))
    k = oracle.f64_to_bf16(rng.standard_normal((b, g, n_max, d_h)))
    v = oracle.f64_to_bf16(rng.standard_normal((b, g, n_max, d_h)))
    return q, k, v


def test_multi_token_attention_with_one_token_is_decode_attention():
    q, k, v = _multi_case(2, 1, 8, 2, 16, 40, seed=31)
    lens = np.array([40, 17], dtype=np.int32)
    got = oracle.decode_attention_multi(q, k, v, lens, 0.25)
    assert np.array_equal(got[:, 0], oracle.decode_attention(q[:, 0], k, v, lens, 0.25))


def test_multi_token_attention_token_t_is_a_decode_step_at_its_own_length():
    """Token t of T sees exactly the rows a single-token step at length L - T + 1 + t sees."""
    T = 5
    q, k, v = _multi_case(3, T, 8, 4, 16, 50, seed=37)
    lens = np.array([50, 5, 23], dtype=np.int32)
    got = oracle.decode_attention_multi(q, k, v, lens, 0.3)
    for t in range(T):
        ref = oracle.decode_attention(np.ascontiguousarray(q[:, t]), k, v, lens - (T - 1 - t), 0.3)
        assert np.array_equal(got[:, t], ref)


def test_multi_token_attention_matches_the_pages_module_with_a_causal_mask():
    """The ybb.press §八 module (repeat_interleave K/V to h heads, einsum scores / sqrt(d_h),
    softmax, einsum with V) in float64 torch, with the causal mask of §十 item 10 added: query
    token t at row start + t may not see rows after it."""
    b, T, h, g, d_h, start = 1, 4, 8, 2, 16, 9
    q, k, v = _multi_case(b, T, h, g, d_h, start + T, seed=41)
    L = start + T
    qf = torch.from_numpy(oracle.bf16_to_f64(q))                     # (B, T, h, d_h)
    kc = torch.from_numpy(oracle.bf16_to_f64(k))[0, :, :L]           # (g, L, d_h)
    vc = torch.from_numpy(oracle.bf16_to_f64(v))[0, :, :L]
    krep = kc.repeat_interleave(h // g, dim=0)                       # (h, L, d_h)
    vrep = vc.repeat_interleave(h // g, dim=0)
    scores = torch.einsum("bthd,hld->bhtl", qf, krep) / (d_h ** 0.5)
    rows = torch.arange(L).view(1, L)
    causal = rows > (start + torch.arange(T)).view(T, 1)             # (T, L): future rows
    scores = scores.masked_fill(causal.view(1, 1, T, L), float("-inf"))
    attn = torch.softmax(scores, dim=-1)
    ref = torch.einsum("bhtl,hld->bthd", attn, vrep).numpy()
    got = oracle.decode_attention_multi(q, k, v, np.array([L], np.int32), 1 / math.sqrt(d_h))
    assert np.allclose(got, ref, rtol=1e-12, atol=1e-12)


def test_multi_token_attention_rejects_lengths_shorter_than_the_tokens():
    q, k, v = _multi_case(2, 3, 4, 1, 8, 10, seed=43)
    out, st = oracle.decode_attention_multi(q, k, v, np.array([2, 10], np.int32), 0.5,
                                            return_status=True)
    assert st == oracle.ERR_BOUNDS and np.all(out[0] == 0) and np.all(np.isfinite(out[1]))


def test_multi_token_append_is_t_single_appends():
    b, T, g, d_h, n_max = 2, 3, 2, 8, 9
    rng = np.random.default_rng(47)
    kn = oracle.f64_to_bf16(rng.standard_normal((b, T, g, d_h)))
    vn = oracle.f64_to_bf16(rng.standard_normal((b, T, g, d_h)))
    k0 = oracle.f64_to_bf16(rng.standard_normal((b, g, n_max, d_h)))
    v0 = oracle.f64_to_bf16(rng.standard_normal((b, g, n_max, d_h)))
    pos = np.array([6, 0], dtype=np.int32)
    k1, v1 = k0.copy(), v0.copy()
    assert oracle.kv_append_multi(kn, vn, k1, v1, pos) == oracle.OK
    k2, v2 = k0.copy(), v0.copy()
    for t in range(T):
        assert oracle.kv_append(np.ascontiguousarray(kn[:, t]), np.ascontiguousarray(vn[:, t]),
                                k2, v2, pos + t) == oracle.OK
    assert np.array_equal(k1, k2) and np.array_equal(v1, v2)
    # rows past the cache: that sequence is skipped, nothing written
    k3, v3 = k0.copy(), v0.copy()
    assert oracle.kv_append_multi(kn, vn, k3, v3, np.array([7, 0], np.int32)) == oracle.ERR_BOUNDS
    assert np.array_equal(k3[0], k0[0]) and np.array_equal(k3[1], k2[1])
