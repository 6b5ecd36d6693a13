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
    """One layer's caches: contiguous [b, g, n_max, d_h] bf16, or, with a page table, page pools
    [num_pages, g, page_size, d_h] whose pages ``page_table`` [b, max_pages] int32 lists per
    sequence (the layers of a model normally share one table). With ``fp8_scales`` = (k_scale,
    v_scale) the caches (contiguous or pools) hold fp8 E4M3 codes (uint8) of value code * scale."""
    k_cache: torch.Tensor
    v_cache: torch.Tensor
    page_table: torch.Tensor | None = None
    fp8_scales: tuple[float, float] | None = None

    def step(self, q, k_new, v_new, pos, seq_lens, out, scale, stream) -> None:
        """One fused append + attention on this layer (q of shape [b, T, h, d_h]: T new tokens
        per sequence, causal; one launch, or two for a prefill-sized T on contiguous caches)."""
        if q.dim() == 4:
            if self.fp8_scales is not None:
                raise ValueError("several tokens per step run on bf16 caches")
            if self.page_table is not None:
                binding.decode_step_paged_multi(q, k_new, v_new, self.k_cache, self.v_cache, pos,
                                                self.page_table, seq_lens, out=out, scale=scale,
                                                stream=stream)
            else:
                binding.decode_step_multi(q, k_new, v_new, self.k_cache, self.v_cache, pos,
                                          seq_lens, out=out, scale=scale, stream=stream)
        elif self.fp8_scales is not None and self.page_table is not None:
            ks, vs = self.fp8_scales
            binding.decode_step_paged_fp8(q, k_new, v_new, self.k_cache, self.v_cache, pos,
                                          self.page_table, seq_lens, ks, vs, out=out,
                                          scale=scale, stream=stream)
        elif self.fp8_scales is not None:
            ks, vs = self.fp8_scales
            binding.decode_step_fp8(q, k_new, v_new, self.k_cache, self.v_cache, pos, seq_lens,
                                    ks, vs, out=out, scale=scale, stream=stream)
        elif self.page_table is None:
            binding.decode_step(q, k_new, v_new, self.k_cache, self.v_cache, pos, seq_lens,
                                out=out, scale=scale, stream=stream)
        else:
            binding.decode_step_paged(q, k_new, v_new, self.k_cache, self.v_cache, pos,
                                      self.page_table, seq_lens, out=out, scale=scale,
                                      stream=stream)

    def append(self, k_new, v_new, pos, stream) -> None:
        if k_new.dim() == 4 and self.page_table is not None:
            binding.kv_append_paged_multi(k_new, v_new, self.k_cache, self.v_cache, pos,
                                          self.page_table, stream=stream)
        elif k_new.dim() == 4:
            binding.kv_append_multi(k_new, v_new, self.k_cache, self.v_cache, pos, stream=stream)
        elif self.fp8_scales is not None and self.page_table is not None:
            binding.kv_append_paged_fp8(k_new, v_new, self.k_cache, self.v_cache, pos,
                                        self.page_table, *self.fp8_scales, stream=stream)
        elif self.fp8_scales is not None:
            binding.kv_append_fp8(k_new, v_new, self.k_cache, self.v_cache, pos,
                                  *self.fp8_scales, stream=stream)
        elif self.page_table is None:
            binding.kv_append(k_new, v_new, self.k_cache, self.v_cache, pos, stream=stream)
        else:
            binding.kv_append_paged(k_new, v_new, self.k_cache, self.v_cache, pos,
                                    self.page_table, stream=stream)

    def attend(self, q, seq_lens, out, scale, stream) -> None:
        if q.dim() == 4 and self.page_table is not None:
            binding.decode_attention_paged_multi(q, self.k_cache, self.v_cache, self.page_table,
                                                 seq_lens, out=out, scale=scale, stream=stream)
        elif q.dim() == 4:
            binding.decode_attention_multi(q, self.k_cache, self.v_cache, seq_lens, out=out,
                                           scale=scale, stream=stream)
        elif self.fp8_scales is not None and self.page_table is not None:
            binding.decode_attention_paged_fp8(q, self.k_cache, self.v_cache, self.page_table,
                                               seq_lens, *self.fp8_scales, out=out, scale=scale,
                                               stream=stream)
        elif self.fp8_scales is not None:
            binding.decode_attention_fp8(q, self.k_cache, self.v_cache, seq_lens,
                                         *self.fp8_scales, out=out, scale=scale, stream=stream)
        elif self.page_table is None:
            binding.decode_attention(q, self.k_cache, self.v_cache, seq_lens, out=out,
                                     scale=scale, stream=stream)
        else:
            binding.decode_attention_paged(q, self.k_cache, self.v_cache, self.page_table,
                                           seq_lens, out=out, scale=scale, stream=stream)


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
            lay.append(x.k_new, x.v_new, pos, stream)
        if attn_events is not None:
            attn_events[li][0].record(stream)
        if fused:
            lay.step(x.q, x.k_new, x.v_new, pos, seq_lens, o, scale, stream)
        else:
            lay.attend(x.q, seq_lens, o, scale, stream)
        if attn_events is not None:
            attn_events[li][1].record(stream)


@dataclasses.dataclass
class HostStepBuffers:
    """A whole step's per-layer inputs and outputs, packed layer-major so that a run of layers is
    one contiguous block, plus the step's append positions and attended lengths (shared by all
    layers): pinned host copies and their device mirrors."""
    q_host: torch.Tensor      # [layers, b, h, d_h] bf16, pinned
    kn_host: torch.Tensor     # [layers, b, g, d_h]
    vn_host: torch.Tensor
    out_host: torch.Tensor    # [layers, b, h, d_h]
    q_dev: torch.Tensor
    kn_dev: torch.Tensor
    vn_dev: torch.Tensor
    out_dev: torch.Tensor
    pos_host: torch.Tensor    # [b] int32, pinned
    lens_host: torch.Tensor   # [b] int32, pinned
    pos_dev: torch.Tensor
    lens_dev: torch.Tensor

    @classmethod
    def allocate(cls, layers: int, b: int, h: int, g: int, d_h: int, device,
                 tokens: int = 1) -> "HostStepBuffers":
        """Buffers for one new token per sequence ([layers, b, h, d_h] ...) or, with tokens = T
        > 1, for T ([layers, b, T, h, d_h] ...)."""
        t = () if tokens == 1 else (tokens,)

        def host(*shape, dtype=torch.bfloat16):
            return torch.empty(shape, dtype=dtype).pin_memory()

        def dev(*shape, dtype=torch.bfloat16):
            return torch.empty(shape, dtype=dtype, device=device)
        return cls(host(layers, b, *t, h, d_h), host(layers, b, *t, g, d_h),
                   host(layers, b, *t, g, d_h), host(layers, b, *t, h, d_h),
                   dev(layers, b, *t, h, d_h), dev(layers, b, *t, g, d_h),
                   dev(layers, b, *t, g, d_h), dev(layers, b, *t, h, d_h),
                   host(b, dtype=torch.int32), host(b, dtype=torch.int32),
                   dev(b, dtype=torch.int32), dev(b, dtype=torch.int32))

    @property
    def h2d_bytes(self) -> int:
        return sum(t.numel() * t.element_size()
                   for t in (self.q_host, self.kn_host, self.vn_host, self.pos_host,
                             self.lens_host))

    @property
    def d2h_bytes(self) -> int:
        return self.out_host.numel() * self.out_host.element_size()


class HostStepPipeline:
    """Drives whole decode steps from pinned host inputs to pinned host outputs with the transfers
    overlapped with the kernels: the inputs of each run of layers are copied in on one stream,
    that run's fused launches wait only for them, and its outputs are copied out on another
    stream while the next run computes. A step of one run stays on the caller's stream.
    Streams and events are created once, so a step costs only the enqueues.

    The runs are the first `chunk` layers, the layers between, and the last `chunk` layers. Only
    the first run's inputs and the last run's outputs are exposed; the middle run's copies hide
    under the first and last runs' kernels. Every boundary between runs is an event wait and
    record on the launch stream, and there consecutive launches cannot overlap, so the runs are
    as few as that allows."""

    def __init__(self, layers: list[LayerState], buf: HostStepBuffers, chunk: int = 8):
        self.layers, self.buf = layers, buf
        n = len(layers)
        if n <= 2 * chunk:
            self.runs = [(c0, min(n, c0 + chunk)) for c0 in range(0, n, chunk)]
        else:
            self.runs = [(0, chunk), (chunk, n - chunk), (n - chunk, n)]
        if len(self.runs) > 1:
            dev = buf.q_dev.device
            self.h2d, self.d2h = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
            self.start = torch.cuda.Event()
            self.back = torch.cuda.Event()
            self.ready = [torch.cuda.Event() for _ in self.runs]
            self.done = [torch.cuda.Event() for _ in self.runs]

    def _copy_in(self, c0: int, c1: int, positions: bool = False) -> None:
        b = self.buf
        if positions:
            b.pos_dev.copy_(b.pos_host, non_blocking=True)
            b.lens_dev.copy_(b.lens_host, non_blocking=True)
        b.q_dev[c0:c1].copy_(b.q_host[c0:c1], non_blocking=True)
        b.kn_dev[c0:c1].copy_(b.kn_host[c0:c1], non_blocking=True)
        b.vn_dev[c0:c1].copy_(b.vn_host[c0:c1], non_blocking=True)

    def _compute(self, c0: int, c1: int, pos, seq_lens, scale: float, stream) -> None:
        b = self.buf
        for li in range(c0, c1):
            self.layers[li].step(b.q_dev[li], b.kn_dev[li], b.vn_dev[li], pos, seq_lens,
                                 b.out_dev[li], scale, stream)

    def run(self, pos: torch.Tensor | None, seq_lens: torch.Tensor | None, scale: float,
            stream: torch.cuda.Stream) -> None:
        """Enqueue one step after the work already on `stream`; `stream` waits for the last copy
        out before anything issued after this call. With `pos` and `seq_lens` None, the step's
        positions and lengths are copied in from the pinned host buffers too (with the first run
        of layers' inputs) and the device mirrors are used."""
        b = self.buf
        from_host = pos is None
        if from_host:
            pos, seq_lens = b.pos_dev, b.lens_dev
        if len(self.runs) == 1:
            c0, c1 = self.runs[0]
            with torch.cuda.stream(stream):
                self._copy_in(c0, c1, positions=from_host)
                self._compute(c0, c1, pos, seq_lens, scale, stream)
                b.out_host[c0:c1].copy_(b.out_dev[c0:c1], non_blocking=True)
            return
        self.start.record(stream)
        self.h2d.wait_event(self.start)
        with torch.cuda.stream(self.h2d):
            for ri, ((c0, c1), ev) in enumerate(zip(self.runs, self.ready)):
                self._copy_in(c0, c1, positions=from_host and ri == 0)
                ev.record(self.h2d)
        for (c0, c1), ready, done in zip(self.runs, self.ready, self.done):
            stream.wait_event(ready)
            self._compute(c0, c1, pos, seq_lens, scale, stream)
            done.record(stream)
            self.d2h.wait_event(done)
            with torch.cuda.stream(self.d2h):
                b.out_host[c0:c1].copy_(b.out_dev[c0:c1], non_blocking=True)
        self.back.record(self.d2h)
        stream.wait_event(self.back)

    def capture(self, pos: torch.Tensor, seq_lens: torch.Tensor, scale: float,
                stream: torch.cuda.Stream) -> torch.cuda.CUDAGraph:
        """Record one step (copies in, launches, copies out) as a CUDA graph on `stream`; each
        replay performs the whole step again, transfers included, for one host-side launch. The
        library's workspace for this stream must already be large enough (run one step first)."""
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            self.run(pos, seq_lens, scale, stream)
        return graph
