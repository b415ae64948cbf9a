"""The benchmark's multi-rank logic on CPU: two gloo ranks, weak scaling.

Every rank times its own replica; the job time is the slowest rank's
(max over ranks) and the whole-job rate counts the work of all ranks.
"""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, results):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        t = bench.max_over_ranks(1.0 + rank, world, torch.device("cpu"))   # rank 1 is the slow one
        dist.barrier()
        results[rank] = (t, bench.whole_job_rate(100.0, world, t))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time_and_count_all_work():
    world = 2
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        results = m.dict()
        port = _free_port()
        procs = [ctx.Process(target=_rank_main, args=(r, world, port, results)) for r in range(world)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(timeout=120)
            assert p.exitcode == 0
        res = dict(results)
    assert res[0][0] == res[1][0] == 2.0
    assert res[0][1] == res[1][1] == pytest.approx(2 * 100.0 / 2.0)


def test_single_process_is_its_own_maximum():
    assert bench.max_over_ranks(3.5, 1, torch.device("cpu")) == 3.5
    assert bench.whole_job_rate(10.0, 1, 2.0) == 5.0


def test_few_heads_sweep_rotates_sets_until_twice_the_l2():
    """The h_q=16 sweep: a cache below twice the L2 is one of the fewest
    block-table sets whose rotation reads at least twice the L2, so that at
    least the L2 passes between two uses of one set; a larger cache is read
    as one set."""
    for b in (16, 32):
        for l in (512, 1024, 2048, 4096, 8192, 16384, 32768, 65536):
            w = bench.WORKLOADS[f"fewheads_fp16_h16_b{b}_l{l}"]
            assert (w["kind"], w["batch"], w["h_q"], w["lens"]) == ("few", b, 16, ("fixed", l))
            seqlens = bench.workload_seqlens(w)
            n = bench.few_table_sets(seqlens)
            per_set = sum(seqlens) * 1152
            assert n * per_set >= 2 * bench.L2_BYTES
            if n > 1:
                assert (n - 1) * per_set < 2 * bench.L2_BYTES     # no more sets than needed
                assert (n - 1) * per_set >= bench.L2_BYTES        # a set is gone from L2 when it returns
