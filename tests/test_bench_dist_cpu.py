"""Multi-rank host logic of bench.py on CPU: two gloo ranks, no GPU.

Under torchrun every rank quantizes its own copy of the workload (weak
scaling, no collective on the data path); the only cross-rank steps are the
max of the timed region over ranks and the whole-job throughput.
"""
import os
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _rank_main(rank, world, port, q):
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import bench

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    slowest = bench.all_ranks_max(10.0 + 5.0 * rank, dist, "cpu")
    value = bench.aggregate_gbs(1e9, 4, world, slowest)
    dist.barrier()
    dist.destroy_process_group()
    q.put((rank, slowest, value))


def test_two_gloo_ranks_agree_on_max_time_and_whole_job_throughput():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = 29500 + os.getpid() % 1000
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    results = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, slowest, value in results:
        assert slowest == 15.0                     # the slower rank's time
        assert value == pytest.approx(1e9 * 4 * 2 / 15e-3 / 1e9)


def test_reference_arm_other_ranks_do_no_work(monkeypatch, capsys):
    sys.path.insert(0, ROOT)
    import bench

    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    class A:
        workload = "small_128x256"; steps = 3; warmup = 1; gpus = 2; impl = "reference"
    assert bench.run_reference(A()) is None
    assert capsys.readouterr().out == ""


def test_single_process_helpers_without_a_group():
    sys.path.insert(0, ROOT)
    import bench

    assert bench.all_ranks_max(3.5) == 3.5
    assert bench.aggregate_gbs(954204160, 2000, 1, 2000 * 0.159) == pytest.approx(6001.3, rel=1e-4)
