"""mqa_decode_attention_noalloc: grouped decode attention for callers that cannot allocate device
memory, such as a framework that has already reserved the GPU's memory for its own pool, or a
latency-critical loop that cannot afford cudaMalloc's implicit synchronisation. It keeps its split
partial states in a fixed array inside the library instead of a cudaMalloc'd workspace.

These tests call it through the C ABI (ctypes, raw pointers). They check its output against the
allocating entry point, mqa_decode_attention, and against the fp64 oracle, within the parity
tolerance used everywhere else, on two calls in a row: the second call starts from the array
contents the first call left behind. They also check that a problem too large for the array is
refused without writing anything, that a call that gave up with arrival counters left non-zero
does not spoil later calls of any size, and that consecutive calls allowed to overlap
(mqa_set_launch_overlap) give the same bits as calls that do not. The file name makes pytest
collect it last.
"""
from __future__ import annotations

import ctypes
import math

import numpy as np
import pytest
import torch

from tests import _parity as P

pytestmark = pytest.mark.gpu

NOALLOC_SCRATCH_BYTES = 8 * 1024 * 1024   # MQA_NOALLOC_SCRATCH_BYTES in include/mqa.h
NOALLOC_MAX_SEGMENTS = 16384              # MQA_NOALLOC_MAX_SEGMENTS: counters at the array's head
UNSUPPORTED = 2


@pytest.fixture(scope="module")
def api():
    import query_grouped_decode_kv_b300.binding as B
    B.debug_override(0, 0)
    lib = B.raw()
    vp, i32 = ctypes.c_void_p, ctypes.c_int
    lib.mqa_decode_attention_noalloc.restype = i32
    lib.mqa_decode_attention_noalloc.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, i32,
                                                 ctypes.c_float, vp]
    yield B, lib
    B.debug_override(0, 0)


def _call_noalloc(lib, q, k, v, lens, out, scale) -> int:
    b, h, d_h = q.shape
    _, g, n_max, _ = k.shape
    stream = torch.cuda.current_stream().cuda_stream
    return lib.mqa_decode_attention_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(),
                                            lens.data_ptr(), out.data_ptr(), b, h, g, d_h, n_max,
                                            float(scale), stream)


def test_noalloc_matches_the_allocating_entry_point_on_two_calls_in_a_row(api):
    B, lib = api
    dev = torch.device("cuda")
    # both shapes split their sequences across many CTAs, so the scratch array is used:
    # G = 4 with d_h = 128, then G = 16 with d_h = 64
    for b, h, g, d_h, lo, hi, seed in [(4, 32, 8, 128, 100, 3000, 600),
                                        (3, 16, 1, 64, 10, 900, 601)]:
        case = P.make_case(b, h, g, d_h, lo, hi, seed_id=seed)
        q = case["q"].to(dev)
        k, v = case["k"].to(dev), case["v"].to(dev)
        lens = case["lens"].to(dev)
        B.kv_append(case["k_new"].to(dev), case["v_new"].to(dev), k, v, case["pos"].to(dev))
        ref = B.decode_attention(q, k, v, lens, scale=case["scale"])
        out = torch.full_like(q, float("nan"))
        assert _call_noalloc(lib, q, k, v, lens, out, case["scale"]) == 0
        torch.cuda.synchronize()
        assert B.get_device_status() == 0
        P.assert_close(out, P.widen(ref), f"noalloc vs allocating entry point, b{b} h{h} g{g}")
        _, _, oracle_out = P.oracle_step(case)
        P.assert_close(out, oracle_out, f"noalloc vs the fp64 oracle, b{b} h{h} g{g}")


def test_noalloc_refuses_a_problem_larger_than_its_array(api):
    B, lib = api
    dev = torch.device("cuda")
    b, h, g, d_h, n_max = 256, 64, 1, 128, 1024
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    tiles = b * g * math.ceil(n_max / 64)
    ctas = max(1, min(sms, math.ceil(tiles / 4)))
    need = (ctas + b * g) * (h // g) * (d_h + 2) * 4
    assert need > NOALLOC_SCRATCH_BYTES - 4 * NOALLOC_MAX_SEGMENTS
    q = torch.zeros(b, h, d_h, dtype=torch.bfloat16, device=dev)
    k = torch.zeros(b, g, n_max, d_h, dtype=torch.bfloat16, device=dev)
    v = torch.zeros_like(k)
    lens = torch.full((b,), n_max, dtype=torch.int32, device=dev)
    out = torch.full_like(q, 3.0)
    assert _call_noalloc(lib, q, k, v, lens, out, 1.0 / math.sqrt(d_h)) == UNSUPPORTED
    torch.cuda.synchronize()
    assert np.all(P.bits(out) == P.bits(torch.full_like(q, 3.0)))


TIMEOUT = 5


def test_noalloc_after_a_timeout_that_left_arrival_counters_dirty(api):
    """A no-alloc call over 600 segments gives up after its CTAs have counted arrivals at split
    segments (testing stall 2). A small no-alloc call follows, then the large one again; both
    must match the oracle, so the clear after the timeout must cover the array's whole counter
    region."""
    B, lib = api
    dev = torch.device("cuda")
    big = P.make_case(300, 32, 2, 64, 500, 999, seed_id=610)
    small = P.make_case(2, 32, 2, 64, 500, 999, seed_id=611)

    def run(case, stall=0):
        q = case["q"].to(dev)
        k, v = case["k"].to(dev), case["v"].to(dev)
        lens = case["lens"].to(dev)
        B.kv_append(case["k_new"].to(dev), case["v_new"].to(dev), k, v, case["pos"].to(dev))
        out = torch.full_like(q, float("nan"))
        assert _call_noalloc(lib, q, k, v, lens, out, case["scale"]) == 0
        return out

    try:
        B.debug_set_wait_limit_ns(20_000_000)
        B.debug_stall(2)
        run(big)
        status = B.get_device_status()
        B.debug_timeout_site()
    finally:
        B.debug_stall(False)
        B.debug_set_wait_limit_ns(0)
    assert status == TIMEOUT, f"expected MQA_ERR_TIMEOUT, got {status}"
    for case, tag in ((small, "small"), (big, "large"), (big, "large again")):
        out = run(case)
        torch.cuda.synchronize()
        assert B.get_device_status() == 0
        P.assert_close(out, P.oracle_step(case)[2], f"noalloc {tag} call after the timeout")


def test_noalloc_calls_allowed_to_overlap_give_the_same_bits(api):
    """Back-to-back no-alloc calls on distinct caches, with and without launch overlap on the
    stream: the same outputs bit for bit (the array is written only after the call ahead has
    finished)."""
    B, lib = api
    dev = torch.device("cuda")
    cases = [P.make_case(4, 32, 4, 128, 300, 2000, seed_id=620 + i) for i in range(4)]
    dev_cases = []
    for c in cases:
        k, v = c["k"].to(dev), c["v"].to(dev)
        B.kv_append(c["k_new"].to(dev), c["v_new"].to(dev), k, v, c["pos"].to(dev))
        dev_cases.append((c["q"].to(dev), k, v, c["lens"].to(dev), c["scale"]))
    stream = torch.cuda.Stream()
    results = {}
    for on in (False, True):
        B.set_launch_overlap(on, stream)
        outs = [torch.full_like(q, float("nan")) for q, *_ in dev_cases]
        torch.cuda.synchronize()
        with torch.cuda.stream(stream):
            for rep in range(3):
                for (q, k, v, lens, scale), out in zip(dev_cases, outs):
                    assert _call_noalloc(lib, q, k, v, lens, out, scale) == 0
        stream.synchronize()
        assert B.get_device_status() == 0
        results[on] = [P.bits(o) for o in outs]
    B.set_launch_overlap(False, stream)
    for a, b in zip(results[False], results[True]):
        assert np.array_equal(a, b)
    for c, o in zip(cases, results[True]):
        ref = P.oracle_step(c)[2]
        out = torch.from_numpy(o.view(np.int16)).view(torch.bfloat16)
        P.assert_close(out, ref, "overlapped noalloc call vs the oracle")
