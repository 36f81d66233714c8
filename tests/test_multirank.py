"""Multi-rank host logic of the benchmark on CPU (gloo, world size 2).

The (batch, KV head) units are independent, so ranks never exchange data: each rank
compresses its own layer with its own seed, and the only collective is the max over ranks
of the timed region.  These tests run that logic in two gloo processes."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    import torch.distributed as dist

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ms = bench.max_over_ranks(10.0 + 5.0 * rank, world, dist, "cpu")
    rate = bench.job_throughput(1000.0, 4, world, ms)
    seed = bench.rank_seed(7, rank)
    dist.barrier()
    out.put((rank, ms, rate, seed))
    dist.destroy_process_group()


def test_max_over_ranks_and_whole_job_rate():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    (r0, ms0, rate0, s0), (r1, ms1, rate1, s1) = res
    assert ms0 == ms1 == 15.0                 # both ranks report the slowest rank's time
    assert rate0 == rate1 == 1000.0 * 4 * 2 / 0.015
    assert s0 != s1                           # each rank compresses a different layer


def test_single_rank_is_identity():
    import bench
    assert bench.max_over_ranks(3.5, 1, None, "cpu") == 3.5


def test_reference_arm_other_ranks_exit_without_work(monkeypatch, capsys):
    import bench

    class A:
        config = "tova_prefill_s512"
        steps = 1
        warmup = 0
        gpus = 2

    monkeypatch.setenv("RANK", "1")
    bench.run_reference(A())
    assert capsys.readouterr().out == ""
