"""Seeded synthetic workloads for the decode step (shapes, lengths, tensors).

This module only draws random numbers and lays them out; it holds none of the attention
arithmetic. Both the CUDA path's tests/benchmark and the CPU oracle's callers use it, so that the
two sides see the same inputs.

Workloads (the decode-attention shapes the MQA/GQA pages discuss; "context" is the number of
tokens cached before this step's token is appended, so the attended length is ``context + 1``):

* ``mqa_tiny``     b=1,  h=8,  g=1,  d_h=64,  context 128, q/K/V ~ N(0,1)
* ``gqa_8b``       b=8,  h=32, g=8,  d_h=128, context ~ U{512..4096} per sequence
* ``mqa_long``     b=64, h=32, g=1,  d_h=128, context 8192
* ``mha_ref``      b=8,  h=32, g=32, d_h=128, context 8192
* ``gqa_70b_80l``  b=8,  h=64, g=8,  d_h=128, context ~ U{1024..32768}, 80 layers, caches ~ N(0, 0.5)
* ``gqa_70b_1l``   the first layer of ``gqa_70b_80l`` alone (same seeds and lengths)

Every tensor is bfloat16 rounded (nearest-even) from a float32 normal draw. Seeds are fixed per
(workload, layer, tensor) so any single layer can be regenerated on its own, on any device.
"""
from __future__ import annotations

import dataclasses
import math

import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    wid: int            # numeric id, used in seeds
    b: int
    h: int
    g: int
    d_h: int
    ctx_lo: int         # context length range before the append (inclusive)
    ctx_hi: int
    layers: int = 1
    kv_std: float = 1.0
    qkv_std: float = 1.0
    extra_rows: int = 0  # cache rows past ctx_hi + 1 (room for several new tokens)

    @property
    def group_size(self) -> int:
        return self.h // self.g

    @property
    def n_max(self) -> int:
        """Cache capacity in rows: the longest context plus the appended token (and extra_rows
        more)."""
        return self.ctx_hi + 1 + self.extra_rows

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d_h)


WORKLOADS = {
    w.name: w
    for w in (
        Workload("mqa_tiny", 1, b=1, h=8, g=1, d_h=64, ctx_lo=128, ctx_hi=128),
        Workload("gqa_8b", 2, b=8, h=32, g=8, d_h=128, ctx_lo=512, ctx_hi=4096),
        Workload("mqa_long", 3, b=64, h=32, g=1, d_h=128, ctx_lo=8192, ctx_hi=8192),
        Workload("mha_ref", 4, b=8, h=32, g=32, d_h=128, ctx_lo=8192, ctx_hi=8192),
        Workload("gqa_70b_80l", 5, b=8, h=64, g=8, d_h=128, ctx_lo=1024, ctx_hi=32768,
                 layers=80, kv_std=0.5),
        # one layer of the 80-layer workload (same kernel configuration; for profiling)
        Workload("gqa_70b_1l", 5, b=8, h=64, g=8, d_h=128, ctx_lo=1024, ctx_hi=32768,
                 layers=1, kv_std=0.5),
    )
}

# tensor kinds, part of the seed
_Q, _KNEW, _VNEW, _KCACHE, _VCACHE, _LENS = range(6)


def seed_for(w: Workload, layer: int, kind: int) -> int:
    return (1000 + w.wid) * 1_000_003 + layer * 16 + kind


def _gen(device, seed: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def normal_bf16(shape, std: float, seed: int, device="cpu") -> torch.Tensor:
    """float32 N(0, std^2) draw rounded to bfloat16."""
    x = torch.randn(shape, generator=_gen(device, seed), device=device, dtype=torch.float32)
    if std != 1.0:
        x.mul_(std)
    return x.to(torch.bfloat16)


def context_lengths(w: Workload) -> torch.Tensor:
    """Context length per sequence (int32, CPU), uniform on the inclusive range."""
    if w.ctx_lo == w.ctx_hi:
        return torch.full((w.b,), w.ctx_lo, dtype=torch.int32)
    g = _gen("cpu", seed_for(w, 0, _LENS))
    return torch.randint(w.ctx_lo, w.ctx_hi + 1, (w.b,), generator=g, dtype=torch.int32)


def step_inputs(w: Workload, layer: int = 0, device="cpu"):
    """This step's q [b,h,d_h] and new K/V rows [b,g,d_h] for one layer."""
    q = normal_bf16((w.b, w.h, w.d_h), w.qkv_std, seed_for(w, layer, _Q), device)
    k_new = normal_bf16((w.b, w.g, w.d_h), w.qkv_std, seed_for(w, layer, _KNEW), device)
    v_new = normal_bf16((w.b, w.g, w.d_h), w.qkv_std, seed_for(w, layer, _VNEW), device)
    return q, k_new, v_new


def cache(w: Workload, layer: int = 0, device="cpu", tail: str = "random",
          lengths: torch.Tensor | None = None):
    """K and V caches [b, g, n_max, d_h] for one layer, before this step's append.

    Rows below each sequence's context length hold N(0, kv_std^2) draws. ``tail`` sets the rows
    at and beyond the context length: ``"random"`` keeps the draws, ``"zero"`` writes zeros,
    ``"nan"`` writes NaN (rows the attention must never read).
    """
    shape = (w.b, w.g, w.n_max, w.d_h)
    k = normal_bf16(shape, w.kv_std, seed_for(w, layer, _KCACHE), device)
    v = normal_bf16(shape, w.kv_std, seed_for(w, layer, _VCACHE), device)
    if tail != "random":
        ctx = context_lengths(w) if lengths is None else lengths
        fill = 0.0 if tail == "zero" else float("nan")
        for bi in range(w.b):
            n = int(ctx[bi])
            k[bi, :, n:, :] = fill
            v[bi, :, n:, :] = fill
    return k, v


def positions_and_lengths(w: Workload):
    """(pos, seq_lens) int32 [b]: the append row and the attended length (context + 1)."""
    ctx = context_lengths(w)
    return ctx.clone(), (ctx + 1).to(torch.int32)


def custom(name: str, b: int, h: int, g: int, d_h: int, ctx_lo: int, ctx_hi: int,
           kv_std: float = 1.0, wid: int = 99) -> Workload:
    """A workload of arbitrary shape (used for small parity cases)."""
    return Workload(name, wid, b=b, h=h, g=g, d_h=d_h, ctx_lo=ctx_lo, ctx_hi=ctx_hi,
                    kv_std=kv_std)


def page_pool(k: torch.Tensor, v: torch.Tensor, rows: torch.Tensor, page_size: int, seed: int,
              spare_pages: int = 0, max_pages: int | None = None, fill: str = "nan"):
    """Lay contiguous caches [b, g, n_max, d_h] out as page pools and a page table.

    Sequence bi gets ceil(rows[bi] / page_size) pages, drawn without replacement from a seeded
    shuffle of all pages (``spare_pages`` more are left unused); its table row lists them in
    order and holds -1 past them (``max_pages`` entries, by default enough for n_max rows).
    Returns (k_pool, v_pool, table): pools [num_pages, g, page_size, d_h] on the caches' device,
    table [b, max_pages] int32 on the CPU. Pool rows no sequence maps (spare pages, and rows of a
    last page past n_max) hold ``fill``: NaN or zero (for pools of uint8 E4M3 codes, the NaN code
    0x7F or code 0).
    """
    b, g, n_max, d_h = k.shape
    need = [(int(r) + page_size - 1) // page_size for r in rows]
    if max_pages is None:
        max_pages = (n_max + page_size - 1) // page_size
    if max(need) > max_pages:
        raise ValueError("a sequence needs more pages than its table row holds")
    num_pages = sum(need) + spare_pages
    order = torch.randperm(num_pages, generator=_gen("cpu", seed)).to(torch.int32)
    table = torch.full((b, max_pages), -1, dtype=torch.int32)
    if k.dtype == torch.uint8:   # E4M3 codes: 0x7F is a NaN code
        value = 0 if fill == "zero" else 0x7F
    else:
        value = 0.0 if fill == "zero" else float("nan")
    k_pool = torch.full((num_pages, g, page_size, d_h), value, dtype=k.dtype, device=k.device)
    v_pool = torch.full_like(k_pool, value)
    used = 0
    for bi in range(b):
        n = need[bi]
        pages = order[used:used + n]
        used += n
        table[bi, :n] = pages
        r = min(n * page_size, n_max)
        for src, pool in ((k, k_pool), (v, v_pool)):
            rows_b = src[bi, :, :r]
            if r < n * page_size:   # the last page runs past n_max: keep the fill there
                rows_b = torch.cat([rows_b, torch.full((g, n * page_size - r, d_h), value,
                                                       dtype=src.dtype, device=src.device)], 1)
            pool[pages.to(src.device, torch.long)] = rows_b.reshape(g, n, page_size,
                                                                    d_h).transpose(0, 1)
    return k_pool, v_pool, table


def fp8_codes(x: torch.Tensor, scale: float) -> torch.Tensor:
    """E4M3 codes (uint8) of x / scale by torch's float8_e4m3fn conversion (a library routine;
    magnitudes are clamped to 448 first, NaN stays NaN): synthetic contents for fp8 caches."""
    y = (x.float() / scale).clamp(-448.0, 448.0)
    return y.to(torch.float8_e4m3fn).view(torch.uint8)


def amax_scale(x: torch.Tensor) -> float:
    """A per-tensor scale that maps the largest finite magnitude of x to 448."""
    a = x.float()
    a = a[torch.isfinite(a)].abs()
    m = float(a.max()) if a.numel() else 1.0
    return (m if m > 0 else 1.0) / 448.0


def multi_step_inputs(w: Workload, T: int, layer: int = 0, device="cpu"):
    """q [b, T, h, d_h] and new K/V rows [b, T, g, d_h] for T new tokens per sequence (token-
    major, like the single-token tensors with a token axis after the batch)."""
    seed = seed_for(w, layer, _Q) * 131 + T
    q = normal_bf16((w.b, T, w.h, w.d_h), w.qkv_std, seed, device)
    k_new = normal_bf16((w.b, T, w.g, w.d_h), w.qkv_std, seed + 1, device)
    v_new = normal_bf16((w.b, T, w.g, w.d_h), w.qkv_std, seed + 2, device)
    return q, k_new, v_new
