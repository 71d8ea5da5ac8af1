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


def test_traffic_record_only_for_its_workload_and_current_sources():
    """The committed DRAM-traffic record applies to the workload it was captured on
    and only while the kernel sources still hash to what was profiled."""
    import hashlib
    import json
    import os
    from synth import workload as wl
    rec = json.load(open(os.path.join(bench.ROOT, "profiles", f"ncu_dram_traffic_{bench.TRAFFIC_WORKLOAD}.json")))
    w_prof = next(w for w in wl.WORKLOADS.values() if w.name == bench.TRAFFIC_WORKLOAD)
    w_other = next(w for w in wl.WORKLOADS.values() if w.name != bench.TRAFFIC_WORKLOAD)
    for kernel, r in rec.items():
        assert bench._traffic(kernel, w_other) is None
        src = os.path.join(bench.ROOT, "sparse_kv_cache_quest_gb300", "csrc", r["source"])
        current = hashlib.sha256(open(src, "rb").read()).hexdigest() == r["source_sha256"]
        assert bench._traffic(kernel, w_prof) == (r["dram_bytes_per_launch"] if current else None)
