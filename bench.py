"""Benchmark: the MQA/GQA decode step (KV append + grouped attention) on B300.

Default workload: the 80-layer GQA decode step of a 70B-class model (b=8 sequences, h=64 query
heads, g=8 KV heads, d_h=128, contexts uniform in [1024, 32768], about 86 GB of bf16 cache): one
step appends one token's K/V and runs attention in all 80 layers back to back, one fused launch
(mqa_decode_step) per layer.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME] [--paged PAGE_SIZE] [--kv bf16|fp8] [--tokens T]

Prints one JSON line (rank 0). ``value`` is microseconds per decode step measured on the device
with inputs resident in HBM (lower is better), from CUDA-graph replays of the whole step (every
layer's append and attention): K replays back to back between two events, or, for workloads small
enough to sit in L2, one graph per step that flushes L2 (a 252 MB write) and then times the step
between its own event nodes. ``e2e`` is the same step driven eagerly through the public Python
API from pinned host buffers (``layers.HostStepPipeline``, recorded once as a CUDA graph and
replayed per step), with the host->device copy of the step's inputs (q, k_new, v_new of every
layer) and the device->host read of its outputs inside the timed region of every step,
overlapped with the kernels in runs of eight layers. ``roofline``
reports the decode kernel's HBM throughput on algorithmic bytes (K/V rows read, q read, out
written, new rows read and written) against the measured copy bandwidth; its launch durations
come from a second timed pass of K steps whose graphs carry CUDA event nodes around every launch.
``cpu_baseline`` times the fp64 CPU oracle on a bounded sample of the same workload. The reference
arm (``--impl reference``) times that oracle as the reference.

``--kv fp8`` runs the same workload with every layer's caches held as fp8 E4M3 codes of the same
draws, one scale per tensor (the largest magnitude maps to 448), through ``mqa_decode_step_fp8``;
the algorithmic bytes count one byte per cached element.

``--tokens T`` runs every step with T new tokens per sequence (causal; speculative decoding):
each sequence appends T rows and attends with T query rows per head, through
``mqa_decode_step_multi``; the caches get T - 1 more rows, and every K/V byte is still read once
per step.

``--paged PAGE_SIZE`` runs the same workload with every layer's cache held in page pools (the rows
each sequence attends, laid out in pages of PAGE_SIZE rows in a seeded random order, one page table
shared by all layers) through the paged calls (``mqa_decode_step_paged``).

Every layer of the default workload reads about 0.7 GB of cache (above the 126 MB L2) and a step
reads about 57 GB, so no L2 flush is needed between its timed steps.
"""
from __future__ import annotations

import argparse
import hashlib
import json
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
KERNEL_SOURCES = ["query_grouped_decode_kv_b300/csrc/decode_attention.cuh",
                  "query_grouped_decode_kv_b300/csrc/decode_attention_tc.cuh",
                  "query_grouped_decode_kv_b300/csrc/kv_append.cuh",
                  "query_grouped_decode_kv_b300/csrc/ptx.cuh",
                  "query_grouped_decode_kv_b300/csrc/status.cuh",
                  "query_grouped_decode_kv_b300/csrc/mqa_abi.cu",
                  "include/mqa.h"]
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "decode_attention_traffic.json")


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


def measured_peak_hbm():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic(workload: str):
    """DRAM bytes per attention launch from a committed ncu summary, if it was taken on the
    current kernel sources; else None."""
    try:
        with open(TRAFFIC_FILE) as f:
            rec = json.load(f)
    except Exception:
        return None
    if rec.get("source_hash") != kernel_source_hash():
        return None
    per = rec.get("per_workload", {}).get(workload)
    return None if per is None else per.get("dram_bytes_per_launch")


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
        import dataclasses
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


# ------------------------------------------------------------------------------------------------
# the CPU oracle on a bounded sample (our arm's cpu_baseline and the reference arm)
# ------------------------------------------------------------------------------------------------
def oracle_sample_timing(w, target_s: float = 12.0, max_s: float = 40.0, T: int = 1):
    """Time the fp64 oracle on whole sequences of this workload's shape (one layer, T new tokens
    per sequence), adding sequences until about ``target_s`` seconds of CPU work; return
    (us_per_step, details)."""
    import numpy as np

    import oracle
    _, lens = inputs.positions_and_lengths(w)
    threads = oracle.num_threads()
    # sample sequences: one per length quantile, longest first, generated on the host
    order = sorted(range(w.b), key=lambda i: -int(lens[i]))
    spent, rows_done, seqs = 0.0, 0, []
    for bi in order:
        L = int(lens[bi])
        sw = inputs.custom("oracle_sample", 1, w.h, w.g, w.d_h, L - 1, L - 1, kv_std=w.kv_std,
                           wid=500 + bi)
        if T > 1:
            q, _, _ = inputs.multi_step_inputs(sw, T, 0, "cpu")
        else:
            q, _, _ = inputs.step_inputs(sw, 0, "cpu")
        k, v = inputs.cache(sw, 0, "cpu")
        qb = q.contiguous().view(torch.int16).numpy().view(np.uint16)
        kb = k.view(torch.int16).numpy().view(np.uint16)
        vb = v.view(torch.int16).numpy().view(np.uint16)
        lb = np.array([L], dtype=np.int32)
        t0 = time.perf_counter()
        if T > 1:
            oracle.decode_attention_multi(qb, kb, vb, lb, sw.scale, threads=threads)
        else:
            oracle.decode_attention(qb, kb, vb, lb, sw.scale, threads=threads)
        spent += time.perf_counter() - t0
        rows_done += L
        seqs.append(L)
        if spent >= target_s or spent >= max_s:
            break
    total_rows = int(lens.sum()) * w.layers
    us_per_step = spent / rows_done * total_rows * 1e6
    detail = (f"{len(seqs)} whole sequence(s) of one layer (lengths {seqs}, all {w.h} heads"
              + (f", {T} tokens" if T > 1 else "") + "), "
              f"{spent:.1f} s of oracle time, scaled by attended rows to {w.layers} layer(s) x "
              f"{w.b} sequences")
    return us_per_step, threads, detail, spent


def run_reference(args, world, rank):
    if rank != 0:
        return 0
    w = inputs.WORKLOADS[args.workload]
    times = []
    for it in range(args.warmup + args.steps):
        us, threads, detail, _ = oracle_sample_timing(w, target_s=2.0, max_s=10.0)
        if it >= args.warmup:
            times.append(us)
    us = statistics.median(times)
    line = {
        "impl": "reference", "metric": METRIC, "value": us, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": us / 1000.0,
        "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": workload_config(w, args.paged, args.kv),
        "cpu_baseline": {"value": us, "unit": UNIT, "cores": threads, "kind": "oracle",
                         "sample": detail},
        "e2e": {"value": us, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


L2_BYTES = 126 * 1024 * 1024


def step_kv_bytes(w, eb: int = 2) -> int:
    _, lens = inputs.positions_and_lengths(w)
    return kv_bytes(w, lens, eb) * w.layers


def needs_l2_flush(w, eb: int = 2) -> bool:
    """A step that reads less than twice the L2 could be served from it on the next step."""
    return step_kv_bytes(w, eb) < 2 * L2_BYTES


def workload_config(w, paged: int = 0, kv: str = "bf16"):
    eb = 1 if kv == "fp8" else 2
    return {"workload": w.name, "b": w.b, "h": w.h, "g": w.g, "d_h": w.d_h, "layers": w.layers,
            "context": [w.ctx_lo, w.ctx_hi], "n_max": w.n_max,
            "kv_dtype": ("fp8 e4m3, one scale per tensor (largest magnitude -> 448)"
                         if kv == "fp8" else "bf16"),
            "kv_layout": (f"paged, {paged}-row pages in a seeded random order" if paged
                          else "contiguous [b, g, n_max, d_h]"),
            "l2": ("L2 flushed between steps (256 MB write)" if needs_l2_flush(w, eb)
                   else "inputs larger than L2 (no flush)")}


PAGE_TABLE_SEED = 4242


def traffic_key(w, paged: int = 0, kv: str = "bf16", T: int = 1) -> str:
    return (w.name + (f"_paged{paged}" if paged else "") + ("_fp8" if kv == "fp8" else "")
            + (f"_T{T}" if T > 1 else ""))


# ------------------------------------------------------------------------------------------------
# our arm
# ------------------------------------------------------------------------------------------------
def run_ours(args, world, rank, local):
    import query_grouped_decode_kv_b300 as mqa
    from query_grouped_decode_kv_b300.layers import (HostStepBuffers, HostStepPipeline,
                                                     LayerState, StepInputs, decode_layers)

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    w = inputs.WORKLOADS[args.workload]
    T = args.tokens
    w, pos, lens = step_shape(w, T)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)

    pos_d, lens_d = pos.to(dev), lens.to(dev)
    layers, xs, outs = [], [], []
    table_d = None
    for li in range(w.layers):
        k, v = inputs.cache(w, li, dev, tail="random")
        if args.kv == "fp8":
            # codes of the same draws, one scale per tensor (largest magnitude -> 448)
            ks, vs = inputs.amax_scale(k), inputs.amax_scale(v)
            k, v = inputs.fp8_codes(k, ks), inputs.fp8_codes(v, vs)
            layers.append(LayerState(k, v, fp8_scales=(ks, vs)))
            xs.append(StepInputs(*inputs.step_inputs(w, li, dev)))
            outs.append(torch.empty(w.b, w.h, w.d_h, dtype=torch.bfloat16, device=dev))
            continue
        if args.paged:
            # the same rows in page pools; one page table (a seeded shuffle of the pages that the
            # attended rows need) shared by every layer
            k, v, table = inputs.page_pool(k, v, lens, args.paged, seed=PAGE_TABLE_SEED)
            if table_d is None:
                table_d = table.to(dev)
        layers.append(LayerState(k, v, table_d))
        if T > 1:
            xs.append(StepInputs(*inputs.multi_step_inputs(w, T, li, dev)))
            outs.append(torch.empty(w.b, T, w.h, w.d_h, dtype=torch.bfloat16, device=dev))
            continue
        xs.append(StepInputs(*inputs.step_inputs(w, li, dev)))
        outs.append(torch.empty(w.b, w.h, w.d_h, dtype=torch.bfloat16, device=dev))
    # small workloads fit in L2: flush it between steps by writing a buffer twice its size
    eb = 1 if args.kv == "fp8" else 2
    flush = (torch.empty(2 * L2_BYTES, dtype=torch.uint8, device=dev) if needs_l2_flush(w, eb)
             else None)
    stream = torch.cuda.Stream(dev)
    torch.cuda.synchronize()

    def step(events=None, step_events=None):
        if flush is not None:
            flush.fill_(1)
        if step_events is not None:
            step_events[0].record(stream)
        decode_layers(layers, xs, pos_d, lens_d, outs, w.scale, stream=stream, attn_events=events)
        if step_events is not None:
            step_events[1].record(stream)

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()

    def timing_event():
        return torch.cuda.Event(enable_timing=True, external=True)

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            step()
    torch.cuda.synchronize()
    assert mqa.get_device_status() == 0, "device status latched an error during warm-up"

    # ---- `value`: the step as CUDA-graph replays. Without an L2 flush, one graph replayed K
    # times back to back between two events. With a flush, one graph per step whose event nodes
    # bracket the step but not the flush before it, so the flush's time is not counted. ----
    n0 = mqa.kernel_launch_count()
    if flush is None:
        step_graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(step_graph, stream=stream):
            step()
        value_graphs, value_events = [step_graph] * args.steps, None
    else:
        value_graphs, value_events = [], []
        for _ in range(args.steps):
            pair = (timing_event(), timing_event())
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                step(step_events=pair)
            value_graphs.append(g)
            value_events.append(pair)
    launches_per_step = (mqa.kernel_launch_count() - n0) // (1 if flush is None else args.steps)
    # ---- per-launch attention durations: the same step with external event nodes around every
    # attention launch, one graph per timed step so each launch keeps its own events ----
    timed_graphs, ev = [], []
    for _ in range(args.steps):
        evs = [(timing_event(), timing_event()) for _ in range(w.layers)]
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            step(evs)
        timed_graphs.append(g)
        ev.append(evs)
    with torch.cuda.stream(stream):
        value_graphs[0].replay()
        timed_graphs[0].replay()
    torch.cuda.synchronize()

    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clocks:
        barrier()
        torch.cuda.synchronize()
        with torch.cuda.stream(stream):
            t_start.record(stream)
            for g in value_graphs:
                g.replay()
            t_end.record(stream)
        torch.cuda.synchronize()
        barrier()
        # second timed region: kernel durations (event nodes add a little time between launches,
        # so they stay out of the step time above)
        with torch.cuda.stream(stream):
            for g in timed_graphs:
                g.replay()
        torch.cuda.synchronize()
        barrier()
    launches = launches_per_step * args.steps
    assert mqa.get_device_status() == 0, "device status latched an error in the timed region"
    ms_total = (t_start.elapsed_time(t_end) if value_events is None
                else sum(a.elapsed_time(b) for a, b in value_events))
    attn_ms = [a.elapsed_time(b) for row in ev for (a, b) in row]
    attn_avg_s = sum(attn_ms) / len(attn_ms) / 1000.0

    # ---- end to end through host buffers: every step copies its inputs in from pinned host
    # memory and its outputs out, overlapped with the kernels (layers.HostStepPipeline) ----
    buf = HostStepBuffers.allocate(w.layers, w.b, w.h, w.g, w.d_h, dev, tokens=T)
    for li, x in enumerate(xs):
        buf.q_host[li].copy_(x.q.cpu())
        buf.kn_host[li].copy_(x.k_new.cpu())
        buf.vn_host[li].copy_(x.v_new.cpu())
    pipeline = HostStepPipeline(layers, buf)
    h2d, d2h = buf.h2d_bytes, buf.d2h_bytes

    def e2e_step(step_graph_e2e, pair=None):
        # an L2 flush (small workloads only) runs before the step's start event
        if flush is not None:
            flush.fill_(1)
        if pair is not None:
            pair[0].record(stream)
        step_graph_e2e.replay()
        if pair is not None:
            pair[1].record(stream)

    # the step through the public API once eagerly (it sizes the workspace), then as one graph
    with torch.cuda.stream(stream):
        pipeline.run(pos_d, lens_d, w.scale, stream)
    torch.cuda.synchronize()
    e2e_graph = pipeline.capture(pos_d, lens_d, w.scale, stream)
    with torch.cuda.stream(stream):
        for _ in range(2):
            e2e_step(e2e_graph)
    torch.cuda.synchronize()
    e2e_events = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                  for _ in range(args.steps)]
    barrier()
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        for pair in e2e_events:
            e2e_step(e2e_graph, pair)
    torch.cuda.synchronize()
    barrier()
    assert mqa.get_device_status() == 0, "device status latched an error in the e2e region"
    e2e_ms = sum(a.elapsed_time(b) for a, b in e2e_events)

    # ---- max over ranks ----
    ms_per_step = ms_total / args.steps
    e2e_per_step = e2e_ms / args.steps
    if world > 1:
        ms_per_step, e2e_per_step, attn_avg_s = max_over_ranks(
            [ms_per_step, e2e_per_step, attn_avg_s], dev)

    if rank == 0:
        peak, peak_kind = measured_peak_hbm()
        nbytes = kv_bytes(w, lens, eb, T)
        achieved = nbytes / attn_avg_s / 1e9
        traffic = recorded_traffic(traffic_key(w, args.paged, args.kv, T))
        value_us = whole_job_us_per_step(ms_per_step, world)
        cb_us, cb_threads, cb_detail, _ = oracle_sample_timing(w, T=T)
        line = {
            "metric": METRIC, "value": value_us, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
            "higher_is_better": False, "scaling": "weak", "vs_baseline": None,
            "dtype": "f16" if args.kv == "fp8" else "bf16",
            "data": "synthetic", "config": dict(workload_config(w, args.paged, args.kv),
                                                tokens_per_step=T),
            "kv_gbs": achieved, "kv_frac_of_peak": achieved / peak,
            "attention_us_per_layer": attn_avg_s * 1e6,
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                         "frac": achieved / peak, "traffic": traffic,
                         "peak_kind": f"{peak_kind} copy bandwidth",
                         "kernel": "decode_attention_kernel (one fused append + attention launch per layer)",
                         "algorithmic_bytes_per_launch": nbytes,
                         "flops_per_launch": attention_flops(w, lens, T)},
            "e2e": {"value": whole_job_us_per_step(e2e_per_step, world), "unit": UNIT,
                    "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
            "gpu_launches": int(launches),
            "clocks": clocks.summary(),
            "cpu_baseline": {"value": cb_us, "unit": UNIT, "cores": cb_threads, "kind": "oracle",
                             "sample": cb_detail},
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="gqa_70b_80l", choices=sorted(inputs.WORKLOADS))
    ap.add_argument("--paged", type=int, default=0, metavar="PAGE_SIZE",
                    help="keep the caches in page pools of this many rows (0: contiguous)")
    ap.add_argument("--kv", choices=["bf16", "fp8"], default="bf16",
                    help="cache element type: bf16, or fp8 E4M3 codes with per-tensor scales")
    ap.add_argument("--tokens", type=int, default=1, metavar="T",
                    help="new tokens per sequence per step (causal; T > 1: speculative decoding)")
    args = ap.parse_args(argv)
    if args.kv == "fp8" and args.paged:
        ap.error("--kv fp8 runs on contiguous caches")
    if args.tokens < 1 or (args.tokens > 1 and (args.kv == "fp8" or args.paged)):
        ap.error("--tokens T > 1 runs on contiguous bf16 caches")
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    world, rank, local = dist_env()
    if args.impl == "reference":
        return run_reference(args, world, rank)
    return run_ours(args, world, rank, local)


if __name__ == "__main__":
    sys.exit(main())
