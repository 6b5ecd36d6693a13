"""Prefill-sized T on the GPU: the tcgen05 kernel that serves several new tokens per sequence when
their rows per KV head (T * h / g) exceed one 64-row tile of heads.

Every case compares with the fp64 oracle (``oracle_decode_attention_multi``, the ybb.press §八
module with the §十 item 10 causal mask): whole outputs where the oracle finishes in seconds, and
for the largest T every row of a sample of tokens, each checked as a one-token attention over its
own causal length. Caches hold NaN past every sequence's rows, lengths are ragged, and the rows of
a KV head are cut into 128-row blocks with a ragged last block. The fused step (append, then
attend) is checked bit for bit on the caches.
"""
from __future__ import annotations

import dataclasses

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
    yield m
    m.debug_override(0, 0)


def _case(b, h, g, d_h, lo, hi, T, seed):
    """Caches with `ctx` rows, NaN past them, room for T more; q [b, T, h, d_h]; lengths ctx+T."""
    w = dataclasses.replace(inputs.custom(f"pf{seed}", b, h, g, d_h, lo, hi, wid=seed),
                            extra_rows=T - 1)
    pos, _ = inputs.positions_and_lengths(w)
    lens = (pos + T).to(torch.int32)
    q, kn, vn = inputs.multi_step_inputs(w, T, 0, "cpu")
    k, v = inputs.cache(w, 0, "cpu", tail="nan", lengths=pos)
    return dict(w=w, pos=pos, lens=lens, q=q, kn=kn, vn=vn, k=k, v=v, T=T,
                scale=1.0 / d_h ** 0.5)


def _oracle_appended(c):
    kb, vb = P.bits(c["k"]).copy(), P.bits(c["v"]).copy()
    assert oracle.kv_append_multi(P.bits(c["kn"]), P.bits(c["vn"]), kb, vb,
                                  c["pos"].numpy()) == oracle.OK
    return kb, vb


def _gpu_attend(mqa, c, fused=True):
    dev = torch.device("cuda")
    k, v = c["k"].to(dev), c["v"].to(dev)
    q, kn, vn = c["q"].to(dev), c["kn"].to(dev), c["vn"].to(dev)
    pos, lens = c["pos"].to(dev), c["lens"].to(dev)
    if fused:
        out = mqa.decode_step_multi(q, kn, vn, k, v, pos, lens, scale=c["scale"])
    else:
        mqa.kv_append_multi(kn, vn, k, v, pos)
        out = mqa.decode_attention_multi(q, k, v, lens, scale=c["scale"])
    torch.cuda.synchronize()
    assert mqa.get_device_status() == 0
    return k, v, out


@pytest.mark.parametrize("fused", [True, False], ids=["fused", "two_calls"])
@pytest.mark.parametrize("shape", [
    # b, h, g, d_h, ctx_lo, ctx_hi, T
    (2, 16, 2, 128, 100, 700, 64),     # G = 8, T = 64: 512 rows per KV head (4 blocks)
    (2, 64, 2, 128, 50, 300, 64),      # G = 32, T = 64: 2048 rows (16 blocks)
    (3, 24, 3, 128, 10, 900, 45),      # G = 8, T = 45: 360 rows, a ragged last block
    (2, 16, 2, 64, 200, 600, 40),      # d_h = 64
    (2, 16, 2, 128, 300, 800, 512),    # G = 8, T = 512
    (1, 64, 2, 128, 100, 100, 512),    # G = 32, T = 512: 16384 rows per KV head
], ids=["G8_T64", "G32_T64", "G8_T45", "d64_T40", "G8_T512", "G32_T512"])
def test_prefill_matches_the_oracle(mqa, shape, fused):
    b, h, g, d_h, lo, hi, T = shape
    c = _case(b, h, g, d_h, lo, hi, T, seed=1200 + T + h)
    kb, vb = _oracle_appended(c)
    ref = oracle.decode_attention_multi(P.bits(c["q"]), kb, vb, c["lens"].numpy(), c["scale"])
    k, v, out = _gpu_attend(mqa, c, fused)
    assert np.array_equal(P.bits(k), kb) and np.array_equal(P.bits(v), vb)
    print(shape, P.assert_close(out, ref, f"prefill {shape}"))


@pytest.mark.parametrize("h,g", [(16, 2), (32, 1)], ids=["G8", "G32"])
def test_prefill_2048_tokens_on_sampled_tokens(mqa, h, g):
    """T = 2048: every row (all heads) of 48 sampled tokens, each against the one-token oracle at
    its own causal length L - T + 1 + t."""
    T = 2048
    c = _case(1, h, g, 128, 300, 300, T, seed=1300 + h)
    kb, vb = _oracle_appended(c)
    _, _, out = _gpu_attend(mqa, c, fused=True)
    rng = np.random.default_rng(5)
    toks = np.unique(np.concatenate([[0, 1, 63, 64, 127, 128, T - 1],
                                     rng.integers(0, T, 41)]))
    L = int(c["lens"][0])
    qb = P.bits(c["q"])
    for t in toks:
        lim = np.array([L - T + 1 + int(t)], dtype=np.int32)
        ref = oracle.decode_attention(np.ascontiguousarray(qb[:, t]), kb, vb, lim, c["scale"])
        P.assert_close(out[:, int(t)], ref, f"T=2048 token {t}")


def test_prefill_with_forced_path_agrees_with_the_decode_path_at_small_t(mqa):
    """T * h / g <= 64 runs on the mma.sync decode kernel; forcing the tcgen05 path sends the same
    call to the prefill kernel. Both must match the oracle."""
    c = _case(3, 16, 2, 128, 100, 1500, 4, seed=1400)   # 32 rows per KV head
    kb, vb = _oracle_appended(c)
    ref = oracle.decode_attention_multi(P.bits(c["q"]), kb, vb, c["lens"].numpy(), c["scale"])
    _, _, out_mma = _gpu_attend(mqa, c)
    mqa.debug_override(0, 3)
    try:
        _, _, out_pf = _gpu_attend(mqa, c)
    finally:
        mqa.debug_override(0, 0)
    P.assert_close(out_mma, ref, "decode path")
    P.assert_close(out_pf, ref, "prefill kernel")


@pytest.mark.parametrize("ctas", [1, 3, 7])
def test_prefill_result_does_not_depend_on_the_cta_count(mqa, ctas):
    """A CTA walks units u, u + P, ...: forcing few CTAs gives each several units of different
    sequences and KV heads, back to back, with the same result bit for bit."""
    c = _case(2, 32, 4, 128, 200, 900, 24, seed=1500)   # 192 rows per KV head: 2 blocks
    _, _, ref = _gpu_attend(mqa, c)
    mqa.debug_override(ctas, 0)
    try:
        _, _, out = _gpu_attend(mqa, c)
    finally:
        mqa.debug_override(0, 0)
    assert torch.equal(out.view(torch.int16), ref.view(torch.int16))


def test_prefill_zeroes_a_sequence_whose_length_is_below_t(mqa):
    c = _case(3, 16, 2, 128, 100, 400, 80, seed=1600)
    c["lens"][1] = 50                      # fewer rows than new tokens: invalid
    dev = torch.device("cuda")
    k, v = c["k"].to(dev), c["v"].to(dev)
    mqa.kv_append_multi(c["kn"].to(dev), c["vn"].to(dev), k, v, c["pos"].to(dev))
    out = torch.full(c["q"].shape, 7.0, dtype=torch.bfloat16, device=dev)
    mqa.decode_attention_multi(c["q"].to(dev), k, v, c["lens"].to(dev), out=out,
                               scale=c["scale"])
    assert mqa.get_device_status() == 4    # MQA_ERR_DEVICE_BOUNDS
    assert torch.all(out[1] == 0)
    kb, vb = _oracle_appended(c)
    lens = c["lens"].numpy().copy()
    for bi in (0, 2):
        ref = oracle.decode_attention_multi(P.bits(c["q"][bi:bi + 1]), kb[bi:bi + 1],
                                            vb[bi:bi + 1], lens[bi:bi + 1], c["scale"])
        P.assert_close(out[bi:bi + 1], ref, f"valid sequence {bi}")


@pytest.mark.parametrize("scale", [0.0, -0.07, 0.5], ids=["zero", "negative", "large"])
def test_prefill_any_finite_scale(mqa, scale):
    """The scale enters once per key (inside the exponential) and the row's largest scaled score
    is taken from the largest raw score, or the smallest for a negative scale; scale 0 gives the
    mean of the visible V rows."""
    c = _case(2, 16, 2, 128, 100, 600, 48, seed=1700)
    c["scale"] = scale
    kb, vb = _oracle_appended(c)
    ref = oracle.decode_attention_multi(P.bits(c["q"]), kb, vb, c["lens"].numpy(), scale)
    _, _, out = _gpu_attend(mqa, c, fused=True)
    P.assert_close(out, ref, f"prefill scale {scale}")
