"""The benchmark's multi-rank host logic on CPU: two gloo ranks, each timing its
own replica, agree on the slowest rank's step time and on the whole-job
throughput; the reference arm does its work on rank 0 only."""
import os
import socket

import pytest
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        local_ms = [2.5, 4.0][rank]
        ms = bench.max_over_ranks(local_ms)
        out.put((rank, ms, bench.job_gbs(1_000_000, ms, world)))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_job_throughput_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r[1] for r in res] == [4.0, 4.0]
    # 2 ranks x 1 MB in 4 ms = 0.5 GB/s
    assert res[0][2] == res[1][2] == pytest.approx(0.5)


def test_single_process_is_identity():
    assert bench.max_over_ranks(3.25) == 3.25
    assert bench.job_gbs(2e9, 1000.0, 1) == pytest.approx(2.0)


def test_reference_arm_runs_on_rank0_only(monkeypatch, capsys):
    monkeypatch.setenv("RANK", "1")
    bench.run_reference(None)          # returns before touching its arguments
    assert capsys.readouterr().out == ""
