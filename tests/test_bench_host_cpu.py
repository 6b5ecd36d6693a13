"""Host logic of bench.py on CPU.

Covers the clock record, the stored DRAM traffic and its tie to the kernel sources, the variant
keys, the L2-flush rule and the causal FLOP count. The benchmark's timing rules and its
`roofline` object rest on these.
"""
from __future__ import annotations

import json
import os
import re

import pytest
import torch

import bench
from query_grouped_decode_kv_b300 import inputs


def _sampler_reading(tmp_path, lines):
    s = bench.ClockSampler(0)
    s.path = str(tmp_path / "clocks.csv")
    (tmp_path / "clocks.csv").write_text("".join(ln + "\n" for ln in lines))
    return s


def test_clock_summary_takes_the_median_clock_and_the_active_reasons(tmp_path):
    # nvidia-smi --format=csv,noheader,nounits rows, in the sampler's field order
    rows = ["0, 2032, 2032, 600.5, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active",
            "0, 1980, 2032, 700.0, 0x0000000000000004, Not Active, Not Active, Not Active, Active",
            "0, 2032, 2032, 650.0, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active"]
    got = _sampler_reading(tmp_path, rows).summary()
    assert got["sm_mhz"] == 2032.0 and got["sm_max_mhz"] == 2032.0
    assert got["reasons"] == ["sw_power_cap"]
    assert got["samples"] == 3 and got["power_w_max"] == 700.0


def test_clock_summary_reports_hardware_and_thermal_slowdowns(tmp_path):
    rows = ["0, 1500, 2032, 900, 0x8, Active, Not Active, Active, Not Active",
            "0, 1490, 2032, 910, 0x8, Not Active, Active, Not Active, Not Active"]
    got = _sampler_reading(tmp_path, rows).summary()
    assert got["reasons"] == ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown"]
    assert got["sm_mhz"] == 1495.0


def test_clock_summary_without_samples_says_unavailable(tmp_path):
    got = _sampler_reading(tmp_path, []).summary()
    assert got["reasons"] == ["unavailable"] and got["samples"] == 0 and got["sm_mhz"] is None


def test_stored_traffic_is_used_only_on_the_sources_it_was_taken_on(tmp_path, monkeypatch):
    f = tmp_path / "traffic.json"
    rec = {"per_workload": {
        "w": {"dram_bytes_per_launch": 123, "family": "decode",
              "source_hash": bench.kernel_source_hash("decode")},
        "w_T512": {"dram_bytes_per_launch": 456, "family": "prefill",
                   "source_hash": bench.kernel_source_hash("prefill")}}}
    f.write_text(json.dumps(rec))
    monkeypatch.setattr(bench, "TRAFFIC_FILE", str(f))
    assert bench.recorded_traffic("w") == 123
    assert bench.recorded_traffic("w_T512") == 456
    assert bench.recorded_traffic("another") is None
    rec["per_workload"]["w"]["source_hash"] = "0" * 16    # taken on other kernel sources
    rec["per_workload"]["w_T512"]["family"] = "decode"    # hashed over the wrong family
    f.write_text(json.dumps(rec))
    assert bench.recorded_traffic("w") is None
    assert bench.recorded_traffic("w_T512") is None
    monkeypatch.setattr(bench, "TRAFFIC_FILE", str(tmp_path / "absent.json"))
    assert bench.recorded_traffic("w") is None


def test_the_prefill_family_covers_the_decode_sources():
    assert set(bench.KERNEL_SOURCES["decode"]) < set(bench.KERNEL_SOURCES["prefill"])
    for fam in bench.KERNEL_SOURCES.values():
        for rel in fam:
            assert os.path.exists(os.path.join(bench.ROOT, rel)), rel


_KEY = re.compile(r"^(?P<wl>[a-z0-9_]+?)(?:_paged(?P<p>\d+))?(?P<f8>_fp8)?(?:_T(?P<T>\d+))?$")


def test_committed_traffic_is_close_above_the_algorithmic_bytes():
    # every stored capture must read at least the bytes the launch needs and not much more;
    # a capture filed under the wrong variant or workload fails one side
    with open(bench.TRAFFIC_FILE) as fh:
        rec = json.load(fh)
    assert rec["per_workload"], "no stored captures"
    for key, entry in rec["per_workload"].items():
        m = _KEY.match(key)
        assert m and m.group("wl") in inputs.WORKLOADS, key
        T = int(m.group("T") or 1)
        w, _, lens = bench.step_shape(inputs.WORKLOADS[m.group("wl")], T)
        algorithmic = bench.kv_bytes(w, lens, 1 if m.group("f8") else 2, T)
        ratio = entry["dram_bytes_per_launch"] / algorithmic
        # a decode launch reads each K/V row once; the prefill kernel's 128-row blocks of one
        # segment read its K/V through L2, and the rows that miss come from DRAM again
        hi = 1.15 if entry.get("family") == "prefill" else 1.04
        assert 0.999 <= ratio <= hi, (key, ratio)
        assert entry["family"] in bench.KERNEL_SOURCES, key


def test_traffic_keys_name_the_variant():
    w = inputs.WORKLOADS["gqa_70b_80l"]
    assert bench.traffic_key(w) == "gqa_70b_80l"
    assert bench.traffic_key(w, paged=16) == "gqa_70b_80l_paged16"
    assert bench.traffic_key(w, paged=16, kv="fp8", T=4) == "gqa_70b_80l_paged16_fp8_T4"


def test_one_layer_workloads_rotate_through_copies_worth_four_l2_sizes():
    for name in ("gqa_8b", "mqa_long", "mha_ref"):
        w = inputs.WORKLOADS[name]
        n = bench.copies_for(w)
        assert 1 <= n <= bench.MAX_COPIES, name
        # n copies hold at least four L2 sizes between two reads of one copy; n - 1 would not,
        # unless n is the floor of two (no launch follows one on the same caches)
        assert n * bench.step_kv_bytes(w) >= bench.ROTATION_L2_MULTIPLE * bench.L2_BYTES
        assert n == 2 or (n - 1) * bench.step_kv_bytes(w) < \
            bench.ROTATION_L2_MULTIPLE * bench.L2_BYTES
        assert n >= 2
        assert not bench.needs_l2_flush(w)
    assert bench.copies_for(inputs.WORKLOADS["mqa_long"]) == 2
    assert bench.copies_for(inputs.WORKLOADS["mha_ref"]) == 2
    assert bench.copies_for(inputs.WORKLOADS["gqa_70b_80l"]) == 1   # its 80 layers rotate


def test_only_the_tiny_workload_is_flushed_between_steps():
    assert bench.needs_l2_flush(inputs.WORKLOADS["mqa_tiny"])
    assert "flushed" in bench.workload_config(inputs.WORKLOADS["mqa_tiny"])["l2"]
    for name in ("gqa_8b", "mqa_long", "mha_ref", "gqa_70b_80l"):
        assert not bench.needs_l2_flush(inputs.WORKLOADS[name]), name


def test_both_arms_describe_the_same_config():
    # the reference arm and ours print workload_config of the same arguments
    w = inputs.WORKLOADS["gqa_70b_80l"]
    cfg = bench.workload_config(w)
    assert cfg["tokens_per_step"] == 1 and cfg["workload"] == "gqa_70b_80l"
    assert bench.workload_config(w, T=4)["tokens_per_step"] == 4


def test_the_automatic_path_names_follow_the_group_size():
    assert bench.path_name(inputs.WORKLOADS["mha_ref"]).startswith("CUDA cores")
    assert bench.path_name(inputs.WORKLOADS["gqa_8b"]).startswith("mma.sync")   # G = 4
    assert bench.path_name(inputs.WORKLOADS["mqa_long"]).startswith("mma.sync")


@pytest.mark.parametrize("T", [1, 2, 4])
def test_attention_flops_count_each_tokens_visible_keys(T):
    w = inputs.WORKLOADS["mqa_long"]
    lens = torch.tensor([5, 9, 64], dtype=torch.int32)
    # token t of T (t = 0 oldest) sees the rows up to its own: L - (T - 1 - t) of them
    brute = sum(4 * w.h * w.d_h * (int(L) - (T - 1 - t)) for L in lens for t in range(T))
    assert bench.attention_flops(w, lens, T) == brute


@pytest.mark.parametrize("T", [1, 4])
def test_step_shape_attends_every_new_row(T):
    w0 = inputs.WORKLOADS["gqa_8b"]
    w, pos, lens = bench.step_shape(w0, T)
    assert w.n_max == w0.n_max + T - 1
    assert torch.equal(lens, pos + T) and lens.dtype == torch.int32
    assert int(lens.max()) <= w.n_max


RECORDED_LINE = bench.os.path.join(bench.ROOT, "profiles", "bench_default_line.json")


def test_the_recorded_default_line_is_self_consistent():
    """The JSON line of a default run on B300 (profiles/bench_default_line.json): every
    workload's launches x time per launch equals its step time, the roofline follows from the
    bytes and that time, and the end-to-end step is no faster than the device step."""
    with open(RECORDED_LINE) as fh:
        line = json.load(fh)
    assert bench.line_problems(line) == []
    head = line["configs"][line["config"]["workload"]]
    assert head["launches_per_step"] * line["roofline"]["us_per_launch"] <= \
        line["ms_per_step"] * 1000.0 * (1 + 1e-9)
    assert set(line["configs"]) == set(bench.ALL_WORKLOADS)


def test_the_line_checks_catch_a_launch_longer_than_its_step():
    with open(RECORDED_LINE) as fh:
        line = json.load(fh)
    bad = json.loads(json.dumps(line))
    head = bad["config"]["workload"]
    bad["configs"][head]["us_per_launch"] *= 1.04      # as an event-decorated launch time would
    assert any("launches" in p for p in bench.line_problems(bad))
    bad = json.loads(json.dumps(line))
    bad["roofline"]["frac"] *= 1.1
    assert any("frac" in p for p in bench.line_problems(bad))


def test_spread_is_nearest_rank_percentiles():
    d = bench.spread([5.0, 1.0, 4.0, 2.0, 3.0])
    assert d == {"n": 5, "p10": 1.0, "median": 3.0, "p90": 5.0}
    one = bench.spread([7.0])
    assert one["p10"] == one["median"] == one["p90"] == 7.0
    many = bench.spread(list(range(101)))
    assert (many["p10"], many["median"], many["p90"]) == (10, 50, 90)


def test_line_checker_flags_an_unordered_spread():
    line = json.loads(open(os.path.join(bench.ROOT, "profiles", "bench_default_line.json")).read())
    assert bench.line_problems(line) == []
    name = line["config"]["workload"]
    line["configs"][name]["us_per_step_spread"] = {"n": 5, "p10": 3.0, "median": 2.0, "p90": 4.0}
    assert any("not ordered" in p for p in bench.line_problems(line))


def test_the_source_hash_ignores_comments_and_whitespace():
    code = "int f(int x) {\n  return x + 1;  // one more\n}\n/* note\n   on two lines */\n"
    assert bench.code_tokens(code) == "int f(int x) { return x + 1; }"
    assert bench.code_tokens(code.replace("// one more", "// another note")) == \
        bench.code_tokens(code)
    assert bench.code_tokens(code.replace("x + 1", "x + 2")) != bench.code_tokens(code)
