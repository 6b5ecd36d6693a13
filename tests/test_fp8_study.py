"""How much fp8 E4M3 caches change the attention output, measured with the oracle (CPU).

The pages warn that quantizing K/V hurts more when many query heads share one K/V head: every
head of a group sees the same quantization error (the nanhubrain.csdn.net MQA article §4.3,
question 3; ybb.press page §十 item 7). This study quantizes the same
bf16 caches to E4M3 (one scale per tensor, largest magnitude -> 448, the oracle's rounding) and
compares the fp64 attention over the dequantized caches with the fp64 attention over the bf16
caches, for MHA (G = 1), GQA (G = 8) and MQA (G = 32) groupings of the same query heads.

Bound, from the format: E4M3 rounds each element to within 2^-4 of its magnitude (rms about
2^-4 / sqrt(3) = 0.036 for errors spread evenly over the step). V errors move the output by
sum_t p_t dv_t, K errors move each logit by about 0.036 sigma_q sigma_k and the output by the
softmax's first-order response sum_t p_t (ds_t - mean) (v_t - o); both are at most about
0.06 rms(V) in rms over the output elements. The study asserts that bound and that the per-head
error does not grow with the number of heads sharing a K/V head (sharing correlates the heads'
errors, it does not enlarge any one head's error).
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from query_grouped_decode_kv_b300 import inputs

B, H, D = 2, 32, 128


def _quantize(x: torch.Tensor):
    """codes (uint8) and scale of a bf16 tensor, by the oracle's rounding."""
    xf = x.float()
    scale = inputs.amax_scale(xf)
    y = (xf / torch.tensor(scale, dtype=torch.float32)).double().numpy()
    return oracle.f64_to_e4m3(y), scale


def _errors(g: int, ctx: int, kv_std: float, seed: int):
    w = inputs.custom(f"study_{g}_{ctx}", B, H, g, D, ctx, ctx, kv_std=kv_std, wid=seed)
    q, _, _ = inputs.step_inputs(w, 0, "cpu")
    k, v = inputs.cache(w, 0, "cpu")
    lens = np.full(B, ctx, dtype=np.int32)
    qb = q.view(torch.int16).numpy().view(np.uint16)
    kb = k.contiguous().view(torch.int16).numpy().view(np.uint16)
    vb = v.contiguous().view(torch.int16).numpy().view(np.uint16)
    ref = oracle.decode_attention(qb, kb, vb, lens, w.scale)
    kc, ks = _quantize(k)
    vc, vs = _quantize(v)
    got = oracle.decode_attention_fp8(qb, kc, vc, lens, ks, vs, w.scale)
    d = got - ref
    rms_v = float(np.sqrt(np.mean(oracle.bf16_to_f64(vb[:, :, :ctx]) ** 2)))
    per_head = np.sqrt(np.mean(d ** 2, axis=(0, 2)))           # [H]
    return {"max_abs": float(np.abs(d).max()), "rms": float(np.sqrt(np.mean(d ** 2))),
            "rms_over_rms_v": float(np.sqrt(np.mean(d ** 2)) / rms_v),
            "head_rms_mean": float(per_head.mean()), "rms_out": float(np.sqrt(np.mean(ref ** 2)))}


@pytest.mark.parametrize("ctx,kv_std", [(64, 1.0), (512, 1.0), (512, 0.5)])
def test_fp8_cache_error_is_within_the_format_bound_and_not_amplified_by_sharing(ctx, kv_std):
    rows = {g: _errors(g, ctx, kv_std, seed=1500 + ctx) for g in (32, 4, 1)}  # G = 1, 8, 32
    for g, e in rows.items():
        print(f"ctx={ctx} kv_std={kv_std} G={H // g}: max|d|={e['max_abs']:.2e} "
              f"rms={e['rms']:.2e} rms/rms(V)={e['rms_over_rms_v']:.4f} "
              f"rms(out)={e['rms_out']:.3f}")
        assert e["rms_over_rms_v"] <= 0.06
    # per-head error with 32 heads on one K/V head is not larger than with one head per K/V
    # head, beyond the spread between draws
    assert rows[1]["head_rms_mean"] <= 1.5 * rows[32]["head_rms_mean"]
