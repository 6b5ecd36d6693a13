"""Failure detection on the GPU without a fault: every in-kernel wait has a time limit, after which
the launch stops, reports MQA_ERR_TIMEOUT and where it gave up, and leaves the context usable.

The tests turn on a testing stall: before their first tile the consumer warps wait on a barrier
that nothing completes (a flag that nothing sets), with the wait limit shortened to 20 ms. That
wait runs out, the launch stops and reports where; nothing hangs, because the waits for a CTA's
own copies and MMAs still in flight keep the one-second limit. Then the hooks are reset and the
same step must give the oracle's result again on the same context. Each inner-product path is
covered, fused and unfused.
"""
from __future__ import annotations

import pytest
import torch

from tests import _parity as P

pytestmark = pytest.mark.gpu

TIMEOUT = 5
# the stall itself (14), or a wait that sits behind it and ran out first: the producer waiting for
# a free stage (1), the tcgen05 issuer waiting for a stage, for P or for a finished P V (5, 6, 13)
SITES_BEHIND_THE_STALL = {1, 5, 6, 13, 14}


@pytest.fixture(scope="module")
def mqa():
    import query_grouped_decode_kv_b300 as m
    m.debug_override(0, 0)
    m.debug_set_wait_limit_ns(0)
    m.debug_stall(False)
    yield m
    m.debug_override(0, 0)
    m.debug_set_wait_limit_ns(0)
    m.debug_stall(False)


def _fused(case, mqa):
    dev = torch.device("cuda")
    k, v = case["k"].to(dev), case["v"].to(dev)
    out = mqa.decode_step(case["q"].to(dev), case["k_new"].to(dev), case["v_new"].to(dev), k, v,
                          case["pos"].to(dev), case["lens"].to(dev), scale=case["scale"])
    return k, v, out


@pytest.mark.parametrize("fused", [False, True], ids=["two_launches", "fused"])
@pytest.mark.parametrize("path,shape", [
    (1, (4, 32, 8, 128, 500, 3000)),    # CUDA cores, G = 4 (eight warps, register split)
    (2, (4, 64, 8, 128, 500, 3000)),    # mma.sync, G = 8
    (3, (2, 64, 2, 128, 500, 3000)),    # tcgen05, G = 32
], ids=["cuda_cores", "mma_sync", "tcgen05"])
def test_a_wait_that_runs_out_reports_a_timeout_and_the_next_call_is_right(mqa, path, shape,
                                                                           fused):
    case = P.make_case(*shape, seed_id=800 + path)
    _, _, out_ref = P.oracle_step(case)
    run = _fused if fused else P.gpu_step
    mqa.debug_override(0, path)
    try:
        mqa.debug_set_wait_limit_ns(20_000_000)
        mqa.debug_stall(True)
        run(case, mqa)
        status = mqa.get_device_status()
        site = mqa.debug_timeout_site()
    finally:
        mqa.debug_stall(False)
        mqa.debug_set_wait_limit_ns(0)
    assert status == TIMEOUT, f"expected MQA_ERR_TIMEOUT, got {status}"
    assert site[0] in SITES_BEHIND_THE_STALL, f"unexpected wait site: {site}"
    try:
        _, _, out = run(case, mqa)
        torch.cuda.synchronize()
        assert mqa.get_device_status() == 0
        assert mqa.debug_timeout_site()[0] == 0
    finally:
        mqa.debug_override(0, 0)
    P.assert_close(out, out_ref, f"after a timeout, path {path}")


@pytest.mark.parametrize("h", [4, 32], ids=["cuda_cores_G2", "mma_sync_G16"])
def test_a_timeout_with_arrivals_counted_is_cleared_for_a_larger_later_call(mqa, h):
    """A launch over 600 (sequence, KV head) segments gives up after its CTAs have counted their
    arrivals at split segments (testing stall 2), leaving those counters non-zero. A small call
    follows on the same stream (4 segments), then the large shape again: both must match the
    oracle, so the clear after the timeout has to cover every counter of the workspace, not just
    the small call's."""
    big = P.make_case(300, h, 2, 64, 500, 999, seed_id=830 + h)
    small = P.make_case(2, h, 2, 64, 500, 999, seed_id=831 + h)
    _, _, ref_big = P.oracle_step(big)
    _, _, ref_small = P.oracle_step(small)
    try:
        mqa.debug_set_wait_limit_ns(20_000_000)
        mqa.debug_stall(2)
        P.gpu_step(big, mqa)
        status = mqa.get_device_status()
        site = mqa.debug_timeout_site()
    finally:
        mqa.debug_stall(False)
        mqa.debug_set_wait_limit_ns(0)
    assert status == TIMEOUT, f"expected MQA_ERR_TIMEOUT, got {status}"
    assert site[0] in SITES_BEHIND_THE_STALL, f"unexpected wait site: {site}"
    _, _, out_small = P.gpu_step(small, mqa)
    torch.cuda.synchronize()
    assert mqa.get_device_status() == 0
    P.assert_close(out_small, ref_small, "small call after the timeout")
    for rep in range(2):
        _, _, out_big = P.gpu_step(big, mqa)
        torch.cuda.synchronize()
        assert mqa.get_device_status() == 0
        P.assert_close(out_big, ref_big, f"large call after the timeout, run {rep}")
