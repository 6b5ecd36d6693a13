"""The oracle's pins must be able to fail: plant plausible mistakes in a temporary copy of the
oracle's C source (on the CPU), build it, and check that at least one pin rejects each mutant.
"""
from __future__ import annotations

import os
import subprocess

import pytest

import oracle
from oracle import build as oracle_build
from tests import test_oracle_pins as pins

# (name, text in the oracle source, replacement)
MUTANTS = [
    ("strided_group_map", "int j = i / group_size;", "int j = i % g;"),
    ("dropped_scale", "    s *= scale;\n", "\n"),
    ("sign_flip", "    s *= scale;\n", "    s *= -scale;\n"),
    ("transposed_key_index", "kv_off + (size_t)t * d_h + d, kind);\n    s *= scale;",
     "kv_off + (size_t)d * d_h + t, kind);\n    s *= scale;"),
    ("length_off_by_one", "attend_range(q, k_cache, v_cache, kind, bi, i, h, g, d_h, n_max, scale, 0, L,",
     "attend_range(q, k_cache, v_cache, kind, bi, i, h, g, d_h, n_max, scale, 0, L - 1,"),
    ("no_max_subtraction", "double w = exp(scores[t - t_begin] - m);",
     "double w = exp(scores[t - t_begin]);"),
    ("missing_normalisation", "o[d] = acc[d] / l;", "o[d] = acc[d];"),
    ("no_max_subtraction_in_merge", "double w = exp(m[s] - M);", "double w = exp(m[s]);"),
    ("kv_bytes_without_factor_two", "return 2u * num_layers", "return num_layers"),
    ("append_wrong_row", "(size_t)n_max + (size_t)p) * (size_t)d_h;",
     "(size_t)n_max + (size_t)(p > 0 ? p - 1 : p)) * (size_t)d_h;"),
    ("bf16_subnormal_exponent", "mag = ldexp((double)frac, -133);", "mag = ldexp((double)frac, -134);"),
    ("bf16_round_half_up", "(rem == 0.5 && fmod(r, 2.0) != 0.0)", "(rem == 0.5)"),
    ("paged_gather_wrong_page", "table[(size_t)bi * max_pages + t / page_size];",
     "table[(size_t)bi * max_pages + (t / page_size + 1) % max_pages];"),
    ("paged_gather_wrong_row", "(size_t)(t % page_size)) * (size_t)d_h;",
     "(size_t)((t + 1) % page_size)) * (size_t)d_h;"),
    ("paged_append_wrong_row", "(size_t)(p % page_size)) *",
     "(size_t)((p + 1) % page_size)) *"),
    ("e4m3_exponent_bias", "mag = ldexp((double)(8 + frac), expo - 7 - 3);",
     "mag = ldexp((double)(8 + frac), expo - 6 - 3);"),
    ("e4m3_ties_away_from_zero", "(rem == 0.5 && fmod(r, 2.0) == 1.0)", "(rem == 0.5)"),
    ("e4m3_subnormal_step", "int spacing_exp = (E < -6) ? -9 : (E - 3);",
     "int spacing_exp = (E < -7) ? -10 : (E - 3);"),
    ("e4m3_overflow_to_nan", "if (a >= 448.0) return sign | 0x7E;",
     "if (a >= 448.0) return sign | 0x7F;"),
    ("fp8_append_wrong_row", "(size_t)n_max + (size_t)p;\n", "(size_t)n_max + (size_t)(p ^ 1);\n"),
    ("multi_token_no_causal_offset", "const int visible = Lb - T + 1 + tq;",
     "const int visible = Lb;"),
    ("multi_token_causal_off_by_one", "const int visible = Lb - T + 1 + tq;",
     "const int visible = Lb - T + tq;"),
    ("multi_token_wrong_query_token", "const size_t row_off = (((size_t)bi * T + tq) * h + i)",
     "const size_t row_off = (((size_t)bi * T + (T - 1 - tq)) * h + i)"),
    ("multi_token_append_wrong_row", "(size_t)n_max + (size_t)(p0 + t);",
     "(size_t)n_max + (size_t)(p0 + T - 1 - t);"),
    ("fp8_append_without_scale", "(float)oracle_bf16_to_double(k_new[src + d]) / k_scale;",
     "(float)oracle_bf16_to_double(k_new[src + d]);"),
    ("code_gather_wrong_page", "table[(size_t)bi * max_pages + (t / page_size)];",
     "table[(size_t)bi * max_pages + (t / page_size + 1) % max_pages];"),
    ("code_gather_wrong_row", "const size_t in_page = (size_t)(t % page_size);",
     "const size_t in_page = (size_t)((t + 1) % page_size);"),
    ("paged_multi_append_no_token_offset", "const int p = p0 + t;", "const int p = p0;"),
    ("paged_multi_append_wrong_row", "const size_t row_in_page = (size_t)(p % page_size);",
     "const size_t row_in_page = (size_t)((p + 1) % page_size);"),
    ("paged_fp8_append_wrong_row", "const size_t prow = (size_t)(p % page_size);",
     "const size_t prow = (size_t)((p + 1) % page_size);"),
    ("paged_fp8_append_without_scale", "volatile float kq = kx / k_scale;",
     "volatile float kq = kx;"),
]

PIN_TESTS = [getattr(pins, n) for n in dir(pins) if n.startswith("test_")]


def _run_pins() -> int:
    """Run every pin once (parametrised pins with their cases); return the number that fail."""
    import inspect
    import json
    failures = 0
    golden = json.load(open(os.path.join(pins.GOLDEN, "kv_cache_bytes.json")))
    for fn in PIN_TESTS:
        params = inspect.signature(fn).parameters
        if "case" in params:
            calls = [dict(case=c) for c in golden["cases"]]
        elif "ratio" in params:
            calls = [dict(ratio=r) for r in golden["ratios"]]
        elif set(params) == {"h", "g", "d_h"}:
            calls = [dict(h=8, g=2, d_h=64), dict(h=6, g=3, d_h=64)]
        elif set(params) == {"page_size"}:
            calls = [dict(page_size=p) for p in (1, 4, 16)]
        else:
            calls = [{}]
        for kw in calls:
            try:
                fn(**kw)
            except Exception:
                failures += 1
    return failures


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_reject_mutant(name, old, new, tmp_path):
    src = open(oracle_build.SRC).read()
    assert src.count(old) == 1, f"mutation anchor for {name} not found exactly once"
    mutated = tmp_path / "mutant.c"
    mutated.write_text(src.replace(old, new))
    lib = tmp_path / "libmutant.so"
    subprocess.run(["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared", "-o", str(lib),
                    str(mutated), "-lm"], check=True)
    prev = oracle._swap_library(str(lib))
    try:
        failures = _run_pins()
    finally:
        oracle._restore_library(prev)
    assert failures > 0, f"no pin caught the planted mistake '{name}'"


def test_unmutated_oracle_passes_every_pin():
    assert _run_pins() == 0
