"""The multi-GPU bookkeeping of bench.py (replicas, max-over-ranks timing, whole-job throughput)
run as two gloo ranks on the CPU."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ms = [1.0, 3.0][rank]                      # rank 1 is the slow one
    mx = bench.max_over_ranks(ms, world)
    bench.barrier(world)
    q.put((rank, mx, bench.job_throughput(1e9, mx, world)))
    dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_rank_and_sum_the_bytes():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = sorted(q.get(timeout=120) for _ in range(2))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, mx, gbs in got:
        assert mx == 3.0                       # both ranks see the max
        assert gbs == pytest.approx(2e9 / 3e-3 / 1e9)


def test_reference_arm_runs_on_rank_zero_only(monkeypatch, capsys):
    import bench
    monkeypatch.setenv("RANK", "1")

    class A:
        warmup, steps = 3, 1
    bench.run_reference(A())
    assert capsys.readouterr().out == ""
