"""The bench's multi-rank host logic on CPU: two ranks over gloo (127.0.0.1).

Under torchrun every rank runs an independent replica (its own seed); the job
time is the slowest rank's and the work is the sum of the ranks' work, so
`value` is all ranks' visible-tile FLOPs over the max time.  The reference arm
runs on rank 0 only.
"""
import multiprocessing as mp
import os
import socket
import types

import pytest

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, queue):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import torch.distributed as dist

    import bench as b

    dist.init_process_group("gloo", rank=rank, world_size=world)
    env = b.rank_env()
    # rank r: step region 10 + r ms, e2e region 30 - r ms, work 100 (r + 1)
    times, work = b.reduce_over_ranks(dist, "cpu", (10.0 + rank, 30.0 - rank), 100.0 * (rank + 1))
    dist.barrier()
    dist.destroy_process_group()
    queue.put({"rank": rank, "env": env, "times": times, "work": work,
               "seed": b.replica_seed(b.WORKLOADS[2], rank)})


def test_two_ranks_reduce_max_time_and_sum_work():
    ctx = mp.get_context("spawn")
    queue = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, queue)) for r in range(2)]
    for p in procs:
        p.start()
    results = [queue.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    results.sort(key=lambda r: r["rank"])
    for r in results:
        assert r["env"] == (2, r["rank"], r["rank"])
        assert r["times"] == [11.0, 30.0]          # slowest rank of each region
        assert r["work"] == 300.0                  # 100 + 200
    assert results[0]["seed"] != results[1]["seed"]  # independent replicas


def test_single_process_defaults(monkeypatch):
    for k in ("WORLD_SIZE", "RANK", "LOCAL_RANK"):
        monkeypatch.delenv(k, raising=False)
    assert bench.rank_env() == (1, 0, 0)
    w = bench.WORKLOADS[2]
    assert bench.replica_seed(w, 0) == w.seed


def test_reference_arm_runs_on_rank_zero_only(monkeypatch, capsys):
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    args = types.SimpleNamespace(workload=1, warmup=3, steps=1, gpus=2, ref_sample_tokens=512)
    bench.run_reference(args)          # returns without work or output
    assert capsys.readouterr().out == ""


def test_reference_arm_line_on_rank_zero(monkeypatch, capsys):
    pytest.importorskip("numpy")
    monkeypatch.setenv("RANK", "0")
    monkeypatch.setenv("WORLD_SIZE", "1")
    args = types.SimpleNamespace(workload=1, warmup=3, steps=2, gpus=1, ref_sample_tokens=512)
    bench.run_reference(args)
    import json
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["value"] > 0 and line["steps"] == 2
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["cpu_baseline"]["kind"] == "oracle"
