"""The multi-rank host logic of bench.py on the CPU: two gloo ranks on 127.0.0.1.

The path shards with no exchange (independent (sequence, head) units), so N GPUs run N
replicas; the bench takes the slowest rank's time (a max all-reduce) and reports the
whole-job throughput, and only rank 0 runs the reference arm and prints."""
import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def worker(rank, world, port, out):
    import sys
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    r, w, local = bench.dist_env()
    slowest = bench.max_over_ranks(10.0 + 5.0 * rank, w)  # rank 1 is the slow one
    value = bench.job_throughput(1000, 4, w, slowest)
    out[rank] = (r, w, local, slowest, value)
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_rank_and_sum_the_work():
    world = 2
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(worker, args=(world, free_port(), out), nprocs=world, join=True)
        res = dict(out)
    for rank in range(world):
        r, w, local, slowest, value = res[rank]
        assert (r, w, local) == (rank, world, rank)
        assert slowest == 15.0                      # the max over ranks, on every rank
        assert value == pytest.approx(2 * 1000 * 4 / 0.015)


def test_single_rank_needs_no_process_group():
    import sys
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.5, 1) == 3.5
    assert bench.job_throughput(16384, 10, 1, 2.0) == pytest.approx(16384 * 10 / 0.002)


def test_reference_arm_runs_on_rank_zero_only(monkeypatch, capsys):
    import sys
    import types
    sys.path.insert(0, ROOT)
    import bench
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    bench.run_reference(types.SimpleNamespace(steps=1, warmup=3, ref_budget=1.0))
    assert capsys.readouterr().out == ""  # no work, no line: rank 0 alone prints


def test_numa_pinning_degrades_gracefully_and_restores_affinity():
    """Without a readable GPU node (no GPU here) the e2e leg's NUMA placement is skipped and the
    process keeps its CPU affinity."""
    import sys
    sys.path.insert(0, ROOT)
    import bench
    before = os.sched_getaffinity(0)
    spec, prev = bench.pin_to_gpu_numa_node(torch.device("cpu"))
    assert prev == before
    if spec is None:
        assert os.sched_getaffinity(0) == before
    os.sched_setaffinity(0, prev)


def test_clock_summary_keeps_only_the_timed_window_and_reports_reasons():
    import sys
    sys.path.insert(0, ROOT)
    import bench
    c = bench.ClockSampler("GPU-none")
    c.samples = [(0.2, 1500.0, 2070.0, 500.0, []),                 # before the timed region
                 (1.0, 2070.0, 2070.0, 900.0, []),
                 (1.5, 1980.0, 2070.0, 1300.0, ["sw_power_cap"]),
                 (2.0, 2010.0, 2070.0, 1200.0, []),
                 (4.0, 300.0, 2070.0, 100.0, ["hw_slowdown"])]     # after it
    c.t0, c.t1 = 0.9, 2.5
    s = c.summary()
    assert s["samples"] == 3 and s["sm_mhz"] == 2010.0 and s["sm_max_mhz"] == 2070.0
    assert s["reasons"] == ["sw_power_cap"]
    assert s["temperature_c_max"] is None  # these samples carry no temperature
    c.samples = [(1.0, 2070.0, 2070.0, 900.0, [], 51.0), (1.5, 2070.0, 2070.0, 950.0, [], 58.0),
                 (3.0, 2070.0, 2070.0, 950.0, [], 90.0)]                  # the last one after it
    assert c.summary()["temperature_c_max"] == 58.0
    c.t0, c.t1 = 2.1, 2.9  # a window with no sample is reported as such, not guessed
    assert c.summary()["reasons"] == ["unavailable"]
