"""The bench's multi-rank host logic on CPU: two gloo ranks (replicas) reduce
their times to the slowest rank's, and the whole-job value counts every
rank's work over that time.  Also: the reference arm runs on rank 0 only."""
import os
import socket

import pytest
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    import torch.distributed as dist
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank,
                            world_size=world)
    try:
        mine = [10.0 + 5.0 * rank, 3.0 - rank]           # per-rank total ms, second value
        got = bench.max_over_ranks(mine, "cpu")
        value = bench.whole_job_tflops(world, 2.0e12, 4, got[0])
        out.put((rank, got, value))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time_and_count_all_work():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, out)) for r in range(world)]
    for p in procs:
        p.start()
    res = {}
    for _ in range(world):
        rank, got, value = out.get(timeout=120)
        res[rank] = (got, value)
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    for rank in range(world):
        got, value = res[rank]
        assert got == [15.0, 3.0]                        # max over ranks, element-wise
        # 2 ranks x 4 steps x 2 TFLOP over the slowest rank's 15 ms
        assert value == pytest.approx(2 * 4 * 2.0e12 / 15e-3 / 1e12)


def test_single_rank_reduction_is_the_identity():
    assert bench.max_over_ranks([1.5, 2.5], "cpu") == [1.5, 2.5]
    assert bench.whole_job_tflops(1, 1.0e12, 10, 5.0) == pytest.approx(2000.0)


def test_reference_arm_runs_on_rank_zero_only(monkeypatch):
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("LOCAL_RANK", "1")
    args = bench.parse(["--impl", "reference", "--gpus", "2"])
    assert bench.run_reference(args) == 0                # returns at once, prints nothing


def test_profiling_switches_default_off():
    # the driver's plain `bench.py` run times the headline workload; the
    # profiling switches only narrow what a single run times
    args = bench.parse([])
    assert not args.only_strided and args.shape == "" and not args.all_extras
    assert bench.parse(["--only-strided"]).only_strided
