"""Two-rank host logic on CPU (gloo): the whole-job timing and the batch sharding.

Under torchrun, bench.py runs one full replica of the step per rank and reports the slowest
rank's step time divided by the number of ranks. These tests run that reduction with two gloo
ranks. The decode step shards by sequence with no exchange on the data path: each of two ranks
appends and attends its half of the batch with the oracle, and the gathered halves equal the
whole batch's result bit for bit.
"""
from __future__ import annotations

import argparse
import os
import socket

import numpy as np
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

WORLD = 2


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _shard_step(case, b0: int, b1: int):
    """Append then attend sequences b0 .. b1 - 1 with the oracle (one rank's shard)."""
    import oracle
    from tests import _parity as P
    sl = slice(b0, b1)
    kb = np.ascontiguousarray(P.bits(case["k"])[sl])
    vb = np.ascontiguousarray(P.bits(case["v"])[sl])
    st = oracle.kv_append(np.ascontiguousarray(P.bits(case["k_new"])[sl]),
                          np.ascontiguousarray(P.bits(case["v_new"])[sl]), kb, vb,
                          np.ascontiguousarray(case["pos"].numpy()[sl]))
    assert st == oracle.OK
    out = oracle.decode_attention(np.ascontiguousarray(P.bits(case["q"])[sl]), kb, vb,
                                  np.ascontiguousarray(case["lens"].numpy()[sl]), case["scale"])
    return kb, vb, out


def _worker(rank: int, port: int):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=WORLD)
    try:
        import bench
        from tests import _parity as P

        # the job's step time is the slowest rank's, per quantity
        got = bench.max_over_ranks([1.0 + rank, 5.0 - rank, 0.25 * (rank + 1)],
                                   torch.device("cpu"))
        assert got == [2.0, 5.0, 0.5], got
        assert bench.whole_job_us_per_step(got[0], WORLD) == 1000.0

        # each rank takes two of four sequences; no exchange until the check
        case = P.make_case(4, 8, 2, 64, 1, 200, seed_id=950)
        per = case["q"].shape[0] // WORLD
        kb, vb, out = _shard_step(case, rank * per, (rank + 1) * per)
        parts = {}
        for name, arr in (("k", kb), ("v", vb), ("out", out)):
            # bf16 bit patterns travel widened to int32 (gloo has no 16-bit integers)
            t = torch.from_numpy(arr.astype(np.int32) if arr.dtype == np.uint16 else arr)
            bufs = [torch.empty_like(t) for _ in range(WORLD)]
            dist.all_gather(bufs, t)
            parts[name] = torch.cat(bufs).numpy()
        if rank == 0:
            k_ref, v_ref, out_ref = P.oracle_step(case)
            assert np.array_equal(parts["k"], k_ref.astype(np.int32))
            assert np.array_equal(parts["v"], v_ref.astype(np.int32))
            assert np.array_equal(parts["out"], out_ref)
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_reduce_timings_and_shard_the_batch():
    mp.start_processes(_worker, args=(_free_port(),), nprocs=WORLD, join=True,
                       start_method="spawn")


def test_whole_job_value_divides_the_slowest_rank_by_the_ranks():
    import bench
    assert bench.whole_job_us_per_step(8.0, 1) == 8000.0
    assert bench.whole_job_us_per_step(8.0, 4) == 2000.0


def test_reference_arm_runs_on_rank_zero_only(capsys):
    import bench
    args = argparse.Namespace(workload="mqa_tiny", steps=1, warmup=0, paged=0, kv="bf16",
                              tokens=1, gpus=2, impl="reference")
    assert bench.run_reference(args, WORLD, 1) == 0
    assert capsys.readouterr().out == ""
