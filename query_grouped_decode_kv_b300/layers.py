"""A whole decode step over many layers: for every layer, append this token's K/V rows, then run
grouped attention -- all enqueued on one stream through the C ABI.

Host-side orchestration only (a loop over layers); the work is in ``libmqa.so``. By default each
layer is one fused launch (``mqa_decode_step``); ``fused=False`` issues the append and the
attention as two launches (``mqa_kv_append``, then ``mqa_decode_attention``).
"""
from __future__ import annotations

import dataclasses

import torch

from . import binding


@dataclasses.dataclass
class LayerState:
    k_cache: torch.Tensor   # [b, g, n_max, d_h] bf16
    v_cache: torch.Tensor


@dataclasses.dataclass
class StepInputs:
    q: torch.Tensor         # [b, h, d_h] bf16
    k_new: torch.Tensor     # [b, g, d_h] bf16
    v_new: torch.Tensor


def decode_layers(layers: list[LayerState], step_in: list[StepInputs], pos: torch.Tensor,
                  seq_lens: torch.Tensor, outs: list[torch.Tensor], scale: float,
                  stream=None, attn_events=None, fused: bool = True) -> None:
    """Enqueue append + attention for every layer. ``attn_events`` (optional) is a list of
    (start, end) CUDA event pairs, one per layer, recorded around each layer's attention launch
    (the fused launch when ``fused``)."""
    for li, (lay, x, o) in enumerate(zip(layers, step_in, outs)):
        if not fused:
            binding.kv_append(x.k_new, x.v_new, lay.k_cache, lay.v_cache, pos, stream=stream)
        if attn_events is not None:
            attn_events[li][0].record(stream)
        if fused:
            binding.decode_step(x.q, x.k_new, x.v_new, lay.k_cache, lay.v_cache, pos, seq_lens,
                                out=o, scale=scale, stream=stream)
        else:
            binding.decode_attention(x.q, lay.k_cache, lay.v_cache, seq_lens, out=o, scale=scale,
                                     stream=stream)
        if attn_events is not None:
            attn_events[li][1].record(stream)
