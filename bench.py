"""Benchmark: the MQA/GQA decode step (KV append + grouped attention) on B300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME] [--paged PAGE_SIZE] [--kv bf16|fp8] [--tokens T]

With no ``--workload`` the run measures all five decode workloads and prints one JSON line (rank
0) whose headline is the 80-layer GQA step of a 70B-class model (b=8 sequences, h=64 query
heads, g=8 KV heads, d_h=128, contexts uniform in [1024, 32768], about 86 GB of bf16 cache): one
step appends one token's K/V and runs attention in all 80 layers back to back, one fused launch
(``mqa_decode_step``) per layer. The four one-layer workloads (``mqa_tiny``, ``gqa_8b``,
``mqa_long``, ``mha_ref``) are measured the same way and reported under ``configs``.

How a workload is timed (``value``, ``configs[*].us_per_step``): K steps are recorded as one CUDA
graph through the public calls and replayed once between two events, after W eager warm-up
steps; consecutive launches may overlap (``mqa_set_launch_overlap`` on the benchmark's stream:
a launch's fill runs under the previous launch's drain). No step reads data that L2 could still
hold from an earlier step: a multi-layer step reads every layer once (57 GB), and a one-layer
workload rotates through as many distinct copies of its layer (other seeds, same shapes and
lengths) as make four times the L2 between two reads of the same copy. The tiny workload cannot
(one copy is 33 KB), so every one of its steps is preceded by an L2 flush (a 252 MB write) and
bracketed by its own events, the flush untimed. ``us_per_launch`` is the step time divided by the
launches in it, so launches x us_per_launch = us_per_step exactly; ``us_per_launch_isolated`` is
one launch alone (L2 flushed before it, no overlap), the fixed cost included.

``roofline`` is the headline kernel's HBM throughput on algorithmic bytes (K/V rows read, q
read, out written, new rows read and written) per launch divided by ``us_per_launch``, against the
measured copy bandwidth. ``e2e`` is the same step driven eagerly through the C ABI every step
(``layers.HostStepPipeline``: one ``mqa_decode_step`` call per layer from the host, no graph), with
the host->device copy of the step's inputs (q, k_new, v_new of every layer, pos, seq_lens) from
pinned memory and the device->host read of every layer's output inside the timed region of every
step. ``cpu_baseline`` times the fp64 CPU oracle on one whole layer of the workload and scales by
the layer count. The reference arm (``--impl reference``) times that oracle the same way, one
whole layer per step.

``--kv fp8`` (caches as fp8 E4M3 codes of the same draws, one scale per tensor), ``--tokens T``
(T new tokens per sequence, causal) and ``--paged PAGE_SIZE`` (caches in page pools, one seeded
random page table shared by all layers) measure the named workload (default: the 80-layer step)
in that variant alone.
"""
from __future__ import annotations

import argparse
import dataclasses
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

from query_grouped_decode_kv_b300 import inputs  # noqa: E402

METRIC = "decode-attention µs/step and KV-cache GB/s as % of B300 HBM peak"
UNIT = "us/step"
FALLBACK_HBM_GBS = 6400.0
HEADLINE = "gqa_70b_80l"
ALL_WORKLOADS = ["mqa_tiny", "gqa_8b", "mqa_long", "mha_ref", "gqa_70b_80l"]
# The sources each kernel family is built from: a stored DRAM capture of a family's kernel holds
# while they are unchanged.
KERNEL_SOURCES = {
    "decode": ["query_grouped_decode_kv_b300/csrc/decode_attention.cuh",
               "query_grouped_decode_kv_b300/csrc/kv_append.cuh",
               "query_grouped_decode_kv_b300/csrc/ptx.cuh",
               "query_grouped_decode_kv_b300/csrc/status.cuh",
               "query_grouped_decode_kv_b300/csrc/mqa_abi.cu",
               "include/mqa.h"],
}
KERNEL_SOURCES["prefill"] = KERNEL_SOURCES["decode"] + [
    "query_grouped_decode_kv_b300/csrc/decode_attention_tc.cuh",
    "query_grouped_decode_kv_b300/csrc/prefill_attention_tc.cuh"]
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "decode_attention_traffic.json")
L2_BYTES = 126 * 1024 * 1024
ROTATION_L2_MULTIPLE = 4   # bytes read between two reads of the same copy, in L2 sizes
MAX_COPIES = 8             # beyond this a workload is flushed instead of rotated
PAGE_TABLE_SEED = 4242


# ------------------------------------------------------------------------------------------------
# helpers
# ------------------------------------------------------------------------------------------------
def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def max_over_ranks(values, device):
    """Each value's maximum over the ranks of the default process group: the slowest rank sets
    the time of the whole job."""
    import torch.distributed as dist
    t = torch.tensor(list(values), device=device, dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(x) for x in t.tolist()]


def whole_job_us_per_step(ms_per_step: float, world: int) -> float:
    """Weak scaling: every rank runs a full step of its own, so `world` steps finish in the
    slowest rank's step time."""
    return ms_per_step * 1000.0 / world


def measured_peak_bf16():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["bf16_tflops"]), "measured"
    except Exception:
        return 1800.0, "fallback"


def is_prefill(w, T: int) -> bool:
    """Several tokens with more than 64 rows per KV head run on the tcgen05 prefill kernel."""
    return T > 1 and T * (w.h // w.g) > 64


def measured_peak_hbm():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def code_tokens(text: str) -> str:
    """C/C++/CUDA source without its comments, whitespace runs collapsed: what the compiler
    sees, so that a change to the comments keeps a stored capture valid. (String literals in
    these sources hold no comment markers.)"""
    import re
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    return " ".join(text.split())


def kernel_source_hash(family: str = "decode") -> str:
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES[family]:
        with open(os.path.join(ROOT, rel), encoding="utf-8") as f:
            h.update(code_tokens(f.read()).encode())
    return h.hexdigest()[:16]


def recorded_traffic(workload: str):
    """DRAM bytes per launch of the step's dominant kernel from a committed ncu summary, if it
    was taken on the current sources of that kernel's family; else None."""
    try:
        with open(TRAFFIC_FILE) as f:
            rec = json.load(f)
    except Exception:
        return None
    per = rec.get("per_workload", {}).get(workload)
    if per is None:
        return None
    family = per.get("family", "decode")
    if family not in KERNEL_SOURCES or per.get("source_hash") != kernel_source_hash(family):
        return None
    return per.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms while active."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = f"/tmp/mqa_clocks_{os.getpid()}.csv"

    def __enter__(self):
        try:
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"], stdout=self.fh,
                stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
        try:
            self.fh.close()
        except Exception:
            pass

    def summary(self):
        rows = []
        try:
            with open(self.path) as f:
                for ln in f:
                    parts = [p.strip() for p in ln.split(",")]
                    if len(parts) >= 9:
                        rows.append(parts)
        except Exception:
            pass
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"], "samples": 0}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(r[1]) for r in rows if num(r[1]) is not None]
        smax = [num(r[2]) for r in rows if num(r[2]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i] == "Active"})
        power = [num(r[3]) for r in rows if num(r[3]) is not None]
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None, "reasons": reasons,
                "samples": len(rows), "power_w_max": max(power) if power else None}


def step_shape(w, T: int = 1):
    """The workload as a step with T new tokens per sequence runs it: room for the T new rows
    in the cache, and the new rows' positions with the lengths attended (all T rows, by the
    last token)."""
    if T > 1:
        w = dataclasses.replace(w, extra_rows=T - 1)
    pos, _ = inputs.positions_and_lengths(w)
    return w, pos, (pos + T).to(torch.int32)


def kv_bytes(w, lens, eb: int = 2, T: int = 1) -> int:
    """Algorithmic bytes of one fused decode-step launch (one layer) with T new tokens per
    sequence: K and V rows read once for all tokens (2 * g * L_b * d_h * eb over the batch; eb = 2
    bf16, 1 fp8), q read and out written (b * T * h * d_h * 2 each), and the append's new rows
    read (2 * b * T * g * d_h * 2, bf16) and written (2 * b * T * g * d_h * eb)."""
    total_rows = int(lens.sum())
    return (2 * w.g * total_rows * w.d_h * eb + 2 * w.b * T * w.h * w.d_h * 2
            + 2 * w.b * T * w.g * w.d_h * 2 + 2 * w.b * T * w.g * w.d_h * eb)


def attention_flops(w, lens, T: int = 1) -> int:
    """4 h d_h FLOPs per (query row, visible key): token t of T sees L - T + 1 + t rows."""
    rows = sum(T * int(L) - T * (T - 1) // 2 for L in lens.tolist())
    return 4 * w.h * rows * w.d_h


def step_kv_bytes(w, eb: int = 2) -> int:
    _, lens = inputs.positions_and_lengths(w)
    return kv_bytes(w, lens, eb) * w.layers


def copies_for(w, eb: int = 2) -> int:
    """Distinct copies of a one-layer workload that consecutive steps rotate through: enough that
    ROTATION_L2_MULTIPLE L2 sizes of data are read between two reads of the same copy, and at
    least two, so that no launch follows one on the same caches and output (the condition under
    which consecutive launches may overlap). 1 for a multi-layer workload, whose own layers
    rotate. 0 when it would take more than MAX_COPIES (the workload is then flushed from L2
    before every step instead)."""
    if w.layers > 1:
        return 1
    n = max(2, math.ceil(ROTATION_L2_MULTIPLE * L2_BYTES / step_kv_bytes(w, eb)))
    return n if n <= MAX_COPIES else 0


def needs_l2_flush(w, eb: int = 2) -> bool:
    """Only a workload too small to rotate through distinct copies is flushed between steps."""
    return copies_for(w, eb) == 0


def workload_config(w, paged: int = 0, kv: str = "bf16", T: int = 1):
    eb = 1 if kv == "fp8" else 2
    n = copies_for(w, eb)
    return {"workload": w.name, "b": w.b, "h": w.h, "g": w.g, "d_h": w.d_h, "layers": w.layers,
            "context": [w.ctx_lo, w.ctx_hi], "n_max": w.n_max,
            "kv_dtype": ("fp8 e4m3, one scale per tensor (largest magnitude -> 448)"
                         if kv == "fp8" else "bf16"),
            "kv_layout": (f"paged, {paged}-row pages in a seeded random order" if paged
                          else "contiguous [b, g, n_max, d_h]"),
            "l2": ("L2 flushed before every step (252 MB write, untimed)" if n == 0 else
                   ("inputs larger than L2 (no flush; every layer read once per step)"
                    if w.layers > 1 else
                    f"inputs larger than L2: steps rotate through {n} copies of the layer "
                    f"({n * step_kv_bytes(w, eb) / 2**20:.0f} MiB)")),
            "tokens_per_step": T}


def traffic_key(w, paged: int = 0, kv: str = "bf16", T: int = 1) -> str:
    return (w.name + (f"_paged{paged}" if paged else "") + ("_fp8" if kv == "fp8" else "")
            + (f"_T{T}" if T > 1 else ""))


def path_name(w, kv: str = "bf16", T: int = 1) -> str:
    """The inner-product path the library picks for this workload (its automatic rule)."""
    G = w.h // w.g
    if is_prefill(w, T):
        return (f"tcgen05 tensor cores (prefill kernel), {T} tokens x {G} heads = {T * G} rows "
                "per KV head in 128-row tiles")
    if T > 1:
        return f"mma.sync tensor cores, {T} tokens x {G} heads = {T * G} rows per KV head"
    if G <= 2 and kv != "fp8":
        return f"CUDA cores (fp32 FMA), G={G}"
    return f"mma.sync tensor cores, G={G}" + (" (fp16 over widened fp8 codes)" if kv == "fp8"
                                              else " (bf16)")


# ------------------------------------------------------------------------------------------------
# the CPU oracle on whole layers (our arm's cpu_baseline and the reference arm)
# ------------------------------------------------------------------------------------------------
class OracleLayer:
    """Layer 0 of a workload on the host, ready for the fp64 oracle: q and the caches as bf16
    bit patterns, with this step's rows appended."""

    def __init__(self, w, T: int = 1):
        import numpy as np

        import oracle
        self.w, self.T = w, T
        w2, pos, lens = step_shape(w, T)
        q, kn, vn = (inputs.multi_step_inputs(w2, T, 0, "cpu") if T > 1
                     else inputs.step_inputs(w2, 0, "cpu"))
        k, v = inputs.cache(w2, 0, "cpu")

        def bits(t):
            return t.contiguous().view(torch.int16).numpy().view(np.uint16)
        self.q = bits(q)
        self.k, self.v = bits(k), bits(v)
        # the step's append, by the oracle itself (untimed)
        if T > 1:
            oracle.kv_append_multi(bits(kn), bits(vn), self.k, self.v, pos.numpy())
        else:
            oracle.kv_append(bits(kn), bits(vn), self.k, self.v, pos.numpy())
        self.lens = lens.numpy().astype(np.int32)
        self.scale = w2.scale
        self.threads = oracle.num_threads()

    # past this many attended (row, key) pairs a layer is timed on a sample of its tokens
    MAX_PAIRS = 80_000_000   # about 40 GFLOP of fp64 at d_h = 128: some 20 s on 16 cores

    def _sample(self):
        """Tokens timed for T > 1: all when the layer is small, else an even sample, each token
        run as the one-token attention it is (its own causal length)."""
        T = self.T
        pairs = self.w.h * sum(T * int(L) - T * (T - 1) // 2 for L in self.lens.tolist())
        if T == 1 or pairs <= self.MAX_PAIRS:
            return None
        n = max(1, min(T, int(T * self.MAX_PAIRS / pairs)))
        return sorted({int(round(i * (T - 1) / max(n - 1, 1))) for i in range(n)})

    def time_layer(self, threads: int | None = None) -> float:
        """Seconds of one whole-layer attention by the oracle (all sequences, all heads); with a
        token sample, the sample's time scaled by the attended rows of the whole layer.
        `threads`: the oracle's thread count (default: every host core)."""
        import numpy as np

        import oracle
        nthr = self.threads if threads is None else threads
        toks = self._sample()
        t0 = time.perf_counter()
        if self.T > 1 and toks is None:
            oracle.decode_attention_multi(self.q, self.k, self.v, self.lens, self.scale,
                                          threads=nthr)
            return time.perf_counter() - t0
        if self.T == 1:
            oracle.decode_attention(self.q, self.k, self.v, self.lens, self.scale,
                                    threads=nthr)
            return time.perf_counter() - t0
        T, rows_sampled = self.T, 0
        for t in toks:
            lim = (self.lens - T + 1 + t).astype(np.int32)
            oracle.decode_attention(np.ascontiguousarray(self.q[:, t]), self.k, self.v, lim,
                                    self.scale, threads=nthr)
            rows_sampled += int(lim.sum())
        spent = time.perf_counter() - t0
        rows_all = sum(T * int(L) - T * (T - 1) // 2 for L in self.lens.tolist())
        return spent * rows_all / rows_sampled

    def describe(self, seconds: float) -> str:
        w = self.w
        toks = self._sample()
        part = ("" if toks is None else
                f"; {len(toks)} of {self.T} tokens timed (each at its own causal length), scaled "
                "by attended rows to the whole layer")
        return (f"one whole layer measured ({w.b} sequences, lengths {self.lens.tolist()}, all "
                f"{w.h} heads" + (f", {self.T} tokens" if self.T > 1 else "") + part
                + f"): {seconds:.2f} s of oracle time, x {w.layers} identical layer(s)")


def run_reference(args, world, rank):
    if rank != 0:
        return 0
    w = inputs.WORKLOADS[args.workload or HEADLINE]
    T = args.tokens
    lay = OracleLayer(w, T)
    times = []
    for it in range(args.warmup + args.steps):
        s = lay.time_layer()
        if it >= args.warmup:
            times.append(s)
    us = statistics.median(times) * w.layers * 1e6
    line = {
        "impl": "reference", "metric": METRIC, "value": us, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": us / 1000.0,
        "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": workload_config(w, args.paged, args.kv, T),
        "cpu_baseline": {"value": us, "unit": UNIT, "cores": lay.threads, "kind": "oracle",
                         "sample": lay.describe(statistics.median(times))
                         + f"; median of {args.steps} timed layers"},
        "e2e": {"value": us, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------------------------------------------------------------
# our arm
# ------------------------------------------------------------------------------------------------
class Units:
    """The launches of a workload on the device: one (layer state, step inputs, output) per layer
    of a multi-layer workload, or per rotated copy of a one-layer workload. Step k launches
    `per_step` consecutive units starting at unit k * per_step (mod the unit count)."""

    def __init__(self, w, dev, T: int = 1, kv: str = "bf16", paged: int = 0):
        from query_grouped_decode_kv_b300.layers import LayerState, StepInputs
        self.w, self.T, self.kv, self.paged = w, T, kv, paged
        self.eb = 1 if kv == "fp8" else 2
        w2, pos, lens = step_shape(w, T)
        self.w2, self.pos, self.lens = w2, pos, lens
        self.pos_d, self.lens_d = pos.to(dev), lens.to(dev)
        self.flush_each_step = needs_l2_flush(w, self.eb)
        n_units = w.layers if w.layers > 1 else max(copies_for(w, self.eb), 1)
        self.per_step = w.layers
        self.layers, self.xs, self.outs = [], [], []
        table_d = None
        for li in range(n_units):
            k, v = inputs.cache(w2, li, dev, tail="random")
            if kv == "fp8":
                ks, vs = inputs.amax_scale(k), inputs.amax_scale(v)
                k, v = inputs.fp8_codes(k, ks), inputs.fp8_codes(v, vs)
                if paged:
                    k, v, table = inputs.page_pool(k, v, lens, paged, seed=PAGE_TABLE_SEED)
                    if table_d is None:
                        table_d = table.to(dev)
                self.layers.append(LayerState(k, v, table_d, fp8_scales=(ks, vs)))
            elif paged:
                k, v, table = inputs.page_pool(k, v, lens, paged, seed=PAGE_TABLE_SEED)
                if table_d is None:
                    table_d = table.to(dev)
                self.layers.append(LayerState(k, v, table_d))
            else:
                self.layers.append(LayerState(k, v))
            if T > 1:
                self.xs.append(StepInputs(*inputs.multi_step_inputs(w2, T, li, dev)))
                self.outs.append(torch.empty(w.b, T, w.h, w.d_h, dtype=torch.bfloat16,
                                             device=dev))
            else:
                self.xs.append(StepInputs(*inputs.step_inputs(w2, li, dev)))
                self.outs.append(torch.empty(w.b, w.h, w.d_h, dtype=torch.bfloat16, device=dev))
        self.bytes_per_launch = kv_bytes(w2, lens, self.eb, T)
        self.flops_per_launch = attention_flops(w2, lens, T)

    def launch(self, u: int, stream) -> None:
        x = self.xs[u]
        self.layers[u].step(x.q, x.k_new, x.v_new, self.pos_d, self.lens_d, self.outs[u],
                            self.w2.scale, stream)

    def step(self, k: int, stream) -> None:
        n = len(self.layers)
        for i in range(self.per_step):
            self.launch((k * self.per_step + i) % n, stream)


def timing_event():
    return torch.cuda.Event(enable_timing=True, external=True)


REPLAYS = 5  # timed replays after the one the step time is taken from, for the spread


def spread(samples) -> dict:
    """p10, median and p90 of a list of µs-per-step samples (nearest rank)."""
    xs = sorted(samples)
    pick = lambda q: xs[min(len(xs) - 1, max(0, int(round(q * (len(xs) - 1)))))]  # noqa: E731
    return {"n": len(xs), "p10": pick(0.1), "median": pick(0.5), "p90": pick(0.9)}


def time_steps(units: Units, stream, steps: int, flush, mqa, overlap: bool,
               one_launch: bool = False) -> tuple[float, int, dict]:
    """Mean µs per step over `steps` steps recorded as one CUDA graph and replayed once (after
    an untimed replay). With `flush`, every step is preceded by an L2 flush and bracketed by its
    own event nodes (the flush untimed); else the graph runs between two events. `one_launch`:
    every step is a single launch (unit k mod count). Returns (µs per step, launches per step,
    spread): the spread is over the single steps of that replay when each step has its own
    events, else over REPLAYS more timed replays of the whole graph."""
    mqa.set_launch_overlap(overlap, stream)
    n = len(units.layers)
    pairs = []
    n0 = mqa.kernel_launch_count()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for k in range(steps):
            if flush is not None:
                flush.fill_(1)
                pair = (timing_event(), timing_event())
                pair[0].record(stream)
            if one_launch:
                units.launch(k % n, stream)
            else:
                units.step(k, stream)
            if flush is not None:
                pair[1].record(stream)
                pairs.append(pair)
    per_step = (mqa.kernel_launch_count() - n0) // steps
    with torch.cuda.stream(stream):
        g.replay()
    torch.cuda.synchronize()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        t0.record(stream)
        g.replay()
        t1.record(stream)
    torch.cuda.synchronize()
    assert mqa.get_device_status() == 0, "device status latched an error in a timed region"
    if flush is not None:
        per = [a.elapsed_time(b) * 1000.0 for a, b in pairs]
        ms = sum(per) / 1000.0
        dist = spread(per)
    else:
        ms = t0.elapsed_time(t1)
        more = []
        for _ in range(REPLAYS):
            a, b = (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
            with torch.cuda.stream(stream):
                a.record(stream)
                g.replay()
                b.record(stream)
            torch.cuda.synchronize()
            more.append(a.elapsed_time(b) * 1000.0 / steps)
        assert mqa.get_device_status() == 0, "device status latched an error in a timed region"
        dist = spread(more)
    del g
    return ms * 1000.0 / steps, per_step, dist


def measure_workload(w, dev, stream, args, mqa, flush_buf, T=1, kv="bf16", paged=0):
    """One workload: warm-up, the overlapped step time and the isolated launch time. Returns
    (summary dict, Units)."""
    units = Units(w, dev, T, kv, paged)
    with torch.cuda.stream(stream):
        mqa.set_launch_overlap(True, stream)
        for k in range(args.warmup):
            units.step(k, stream)
    torch.cuda.synchronize()
    assert mqa.get_device_status() == 0, "device status latched an error during warm-up"
    flush = flush_buf if units.flush_each_step else None
    us_step, per_step, dist = time_steps(units, stream, args.steps, flush, mqa, overlap=True)
    us_iso, _, dist_iso = time_steps(units, stream, min(args.steps, 20), flush_buf, mqa,
                                     overlap=False, one_launch=True)
    mqa.set_launch_overlap(True, stream)
    peak, _ = measured_peak_hbm()
    us_launch = us_step / per_step
    gbs = units.bytes_per_launch / (us_launch * 1e-6) / 1e9
    summary = {
        "us_per_step": us_step, "launches_per_step": per_step, "us_per_launch": us_launch,
        "us_per_step_spread": dict(dist, over=("single steps of the timed replay" if flush is not None
                                               else f"{REPLAYS} more timed replays of the K steps")),
        "us_per_launch_isolated": us_iso,
        "us_per_launch_isolated_spread": dict(dist_iso, over="single isolated launches"),
        "algorithmic_bytes_per_launch": units.bytes_per_launch,
        "kv_gbs": gbs, "frac_of_hbm": gbs / peak,
        "kv_gbs_isolated": units.bytes_per_launch / (us_iso * 1e-6) / 1e9,
        # one attention launch per layer (the prefill step adds an append launch per layer)
        "tflops": units.flops_per_launch * w.layers / (us_step * 1e-6) / 1e12,
        "path": path_name(w, kv, T),
        "kernel": ("prefill_attention_tc_kernel (mqa_decode_step_multi: an append launch, "
                   "then this)" if is_prefill(w, T) else
                   "decode_attention_kernel (fused append + attention, mqa_decode_step"
                   + ("_fp8" if kv == "fp8" else "_paged" if paged else "_multi" if T > 1 else "")
                   + ")"),
        "l2": workload_config(w, paged, kv, T)["l2"],
        "overlap": "consecutive launches overlap (mqa_set_launch_overlap)"
                   + ("; the L2 flush between steps separates them" if flush is not None else ""),
    }
    return summary, units


def e2e_host_driven(units: Units, dev, stream, steps: int, warmup: int, mqa):
    """The step driven eagerly through the C ABI from pinned host buffers, every step: returns
    (µs per step, h2d bytes, d2h bytes)."""
    from query_grouped_decode_kv_b300.layers import HostStepBuffers, HostStepPipeline
    w = units.w
    n = units.per_step
    lay = units.layers[:n]
    buf = HostStepBuffers.allocate(n, w.b, w.h, w.g, w.d_h, dev, tokens=units.T)
    for li in range(n):
        x = units.xs[li]
        buf.q_host[li].copy_(x.q.cpu())
        buf.kn_host[li].copy_(x.k_new.cpu())
        buf.vn_host[li].copy_(x.v_new.cpu())
    buf.pos_host.copy_(units.pos)
    buf.lens_host.copy_(units.lens)
    pipeline = HostStepPipeline(lay, buf)
    mqa.set_launch_overlap(True, stream)
    with torch.cuda.stream(stream):
        for _ in range(warmup):
            pipeline.run(None, None, units.w2.scale, stream)
    torch.cuda.synchronize()
    events = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(steps)]
    with torch.cuda.stream(stream):
        for a, b in events:
            a.record(stream)
            pipeline.run(None, None, units.w2.scale, stream)
            b.record(stream)
    torch.cuda.synchronize()
    assert mqa.get_device_status() == 0, "device status latched an error in the e2e region"
    ms = sum(a.elapsed_time(b) for a, b in events)
    return ms * 1000.0 / steps, buf.h2d_bytes, buf.d2h_bytes


def read_bandwidth_reference(dev, gib: int = 4, reps: int = 5) -> dict:
    """Context for the roofline: what a plain library read stream reaches on this GPU (a torch
    sum over `gib` GiB of bf16, best of `reps`). The roofline's peak stays the measured copy
    bandwidth, whose bytes are half reads, half writes; a read-only stream such as the decode
    kernel's can go past it."""
    x = torch.ones(gib * 2**30 // 2, dtype=torch.bfloat16, device=dev)
    best = float("inf")
    for _ in range(reps + 1):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        x.sum(dtype=torch.float32)
        b.record()
        torch.cuda.synchronize()
        best = min(best, a.elapsed_time(b))
    del x
    torch.cuda.empty_cache()
    return {"gbs": gib * 2**30 / (best * 1e-3) / 1e9,
            "how": f"torch bf16 sum over {gib} GiB (reads only), best of {reps}"}


def run_ours(args, world, rank, local):
    import query_grouped_decode_kv_b300 as mqa

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    T, kv, paged = args.tokens, args.kv, args.paged
    headline = args.workload or HEADLINE
    variant = T > 1 or kv != "bf16" or paged
    others = [] if (args.workload or variant) else [n for n in ALL_WORKLOADS if n != headline]
    stream = torch.cuda.Stream(dev)
    flush_buf = torch.empty(2 * L2_BYTES, dtype=torch.uint8, device=dev)

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()

    configs = {}
    read_ref = read_bandwidth_reference(dev)
    n_launch0 = mqa.kernel_launch_count()
    with ClockSampler(local) as clocks:
        for name in others:
            barrier()
            summary, units = measure_workload(inputs.WORKLOADS[name], dev, stream, args, mqa,
                                              flush_buf)
            configs[name] = summary
            del units
            torch.cuda.empty_cache()
        barrier()
        summary, units = measure_workload(inputs.WORKLOADS[headline], dev, stream, args, mqa,
                                          flush_buf, T, kv, paged)
        configs[headline] = summary
        barrier()
    launches_timed = summary["launches_per_step"] * args.steps
    e2e_us, h2d, d2h = e2e_host_driven(units, dev, stream, args.steps, args.warmup, mqa)
    barrier()

    us_step, us_launch, e2e_step = summary["us_per_step"], summary["us_per_launch"], e2e_us
    if world > 1:
        us_step, us_launch, e2e_step = max_over_ranks([us_step, us_launch, e2e_step], dev)

    if rank == 0:
        w = units.w
        peak, peak_kind = measured_peak_hbm()
        nbytes = units.bytes_per_launch
        achieved = nbytes / (us_launch * 1e-6) / 1e9
        traffic = recorded_traffic(traffic_key(w, paged, kv, T))
        value_us = whole_job_us_per_step(us_step / 1000.0, world)
        common = {"kernel": summary["kernel"], "algorithmic_bytes_per_launch": nbytes,
                  "flops_per_launch": units.flops_per_launch, "us_per_launch": us_launch,
                  "us_per_launch_from": "step time / launches per step "
                                        "(launches x us_per_launch = ms_per_step)"}
        if is_prefill(w, T):
            # the prefill kernel's score and value products are dense: tensor-bound
            tpeak, tkind = measured_peak_bf16()
            tflops = units.flops_per_launch * w.layers / (us_step * 1e-6) / 1e12
            roofline = dict({"bound": "tensor", "achieved": tflops, "peak": tpeak,
                             "unit": "TFLOP/s", "frac": tflops / tpeak, "traffic": traffic,
                             "peak_kind": f"{tkind} cuBLAS bf16 (burst)",
                             "note": "attention FLOPs of a step over the whole step time "
                                     "(an append launch and an attention launch per layer)"},
                            **common)
        else:
            roofline = dict({"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                             "frac": achieved / peak, "traffic": traffic,
                             "peak_kind": f"{peak_kind} copy bandwidth (burst)",
                             "read_stream_reference": dict(read_ref,
                                                           frac=achieved / read_ref["gbs"])},
                            **common)
        lay = OracleLayer(w, T)
        cb_s = lay.time_layer()
        cb_us = cb_s * w.layers * 1e6
        line = {
            "metric": METRIC, "value": value_us, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": us_step / 1000.0,
            "higher_is_better": False, "scaling": "weak", "vs_baseline": None,
            "dtype": "f16" if kv == "fp8" else "bf16",
            "data": "synthetic", "config": workload_config(w, paged, kv, T),
            "kv_gbs": achieved, "kv_frac_of_peak": achieved / peak,
            "attention_us_per_layer": us_launch,
            "roofline": roofline,
            "configs": configs,
            "e2e": {"value": whole_job_us_per_step(e2e_step / 1000.0, world), "unit": UNIT,
                    "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                    "how": f"eager: {units.per_step} C-ABI call(s) per step from the host, "
                           "pinned-host copies in and out inside every step's timed region"},
            "gpu_launches": int(launches_timed),
            "gpu_launches_all_configs": int(mqa.kernel_launch_count() - n_launch0),
            "clocks": clocks.summary(),
            "cpu_baseline": {"value": cb_us, "unit": UNIT, "cores": lay.threads, "kind": "oracle",
                             "sample": lay.describe(cb_s)},
        }
        if others:
            # the two smallest workloads' oracle on one host thread (one whole layer each)
            line["cpu_baseline"]["single_thread_us_per_step"] = {
                name: OracleLayer(inputs.WORKLOADS[name]).time_layer(threads=1) * 1e6
                for name in ("mqa_tiny", "gqa_8b")}
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def line_problems(line: dict, rel: float = 1e-6) -> list[str]:
    """Consistency checks of a printed JSON line (ours): each workload's launches times its time
    per launch is its step time (so no launch takes longer than the step it is part of), the
    roofline's achieved figure is the algorithmic bytes (or FLOPs) per launch over that time and
    its fraction the achieved over the peak, and the end-to-end step is no faster than the
    device-resident one. Returns the problems found (empty when consistent)."""
    out = []

    def close(a, b):
        return abs(a - b) <= rel * max(abs(a), abs(b), 1e-30)

    for name, c in line.get("configs", {}).items():
        step, per, n = c["us_per_step"], c["us_per_launch"], c["launches_per_step"]
        if n * per > step * (1 + rel):
            out.append(f"{name}: {n} launches x {per} us > {step} us per step")
        if not close(n * per, step):
            out.append(f"{name}: launches x us_per_launch != us_per_step")
        if not close(c["kv_gbs"], c["algorithmic_bytes_per_launch"] / (per * 1e-6) / 1e9):
            out.append(f"{name}: kv_gbs is not bytes per launch over the time per launch")
        for key in ("us_per_step_spread", "us_per_launch_isolated_spread"):
            d = c.get(key)
            if d is not None and not d["p10"] <= d["median"] <= d["p90"]:
                out.append(f"{name}: {key} is not ordered")
    r = line["roofline"]
    head = line["configs"][line["config"]["workload"]]
    if not close(r["us_per_launch"], head["us_per_launch"]):
        out.append("roofline us_per_launch differs from the headline workload's")
    if not close(line["value"], head["us_per_step"] * 1.0 / max(line.get("n_gpus", 1), 1)):
        out.append("value is not the headline workload's step time (whole job)")
    per_unit = (r["algorithmic_bytes_per_launch"] / 1e9 if r["bound"] == "hbm"
                else r["flops_per_launch"] / 1e12)
    if r["bound"] == "hbm" and not close(r["achieved"], per_unit / (r["us_per_launch"] * 1e-6)):
        out.append("roofline achieved is not bytes per launch over us_per_launch")
    if not close(r["frac"], r["achieved"] / r["peak"]):
        out.append("roofline frac is not achieved / peak")
    if line["e2e"]["value"] < line["value"] * (1 - 1e-3):
        out.append("e2e step faster than the device-resident step")
    return out


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=None, choices=sorted(inputs.WORKLOADS),
                    help="measure this workload alone (default: all five, the 80-layer step "
                         "as the headline)")
    ap.add_argument("--paged", type=int, default=0, metavar="PAGE_SIZE",
                    help="keep the caches in page pools of this many rows (0: contiguous)")
    ap.add_argument("--kv", choices=["bf16", "fp8"], default="bf16",
                    help="cache element type: bf16, or fp8 E4M3 codes with per-tensor scales")
    ap.add_argument("--tokens", type=int, default=1, metavar="T",
                    help="new tokens per sequence per step (causal; T > 1: speculative decoding)")
    args = ap.parse_args(argv)
    if args.tokens < 1 or (args.tokens > 1 and args.kv == "fp8"):
        ap.error("--tokens T > 1 runs on bf16 caches")
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    world, rank, local = dist_env()
    if args.impl == "reference":
        return run_reference(args, world, rank)
    return run_ours(args, world, rank, local)


if __name__ == "__main__":
    sys.exit(main())
