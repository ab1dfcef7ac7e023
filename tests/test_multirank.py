"""The N > 1 path of bench.py on CPU: two gloo ranks (127.0.0.1).  The path is
replicas only (each rank attends over its own micro-batch; no data-path
collective), so what crosses ranks is the timing aggregate: the slowest
rank's times and the sum of the ranks' useful FLOPs.  Also: each rank draws a
different seeded micro-batch, and rank 0 alone prints."""
import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, ws, port, out):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(ws),
                      LOCAL_RANK=str(rank))
    import bench
    from packed_varlen_attention_aware_gb300 import workloads as wl

    dist.init_process_group("gloo", rank=rank, world_size=ws)
    w_ws, w_rank, w_local = bench.dist_setup()
    times, flops = bench.aggregate_over_ranks([10.0 * (rank + 1), 20.0 - rank, 1.5 + rank], 1000 * (rank + 1), ws,
                                              "cpu")
    lengths = wl.workload("mb32k", 3 + rank).lengths
    dist.barrier()
    dist.destroy_process_group()
    out.put((rank, (w_ws, w_rank, w_local), times, flops, lengths))


def test_two_gloo_ranks_aggregate():
    ws, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, ws, port, q)) for r in range(ws)]
    for p in procs:
        p.start()
    res = {}
    for _ in range(ws):
        rank, env, times, flops, lengths = q.get(timeout=120)
        res[rank] = (env, times, flops, lengths)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank in range(ws):
        env, times, flops, _ = res[rank]
        assert env == (ws, rank, rank)
        assert times == [20.0, 20.0, 2.5]  # max over ranks
        assert flops == 3000.0              # sum over ranks
    assert res[0][3] != res[1][3]           # replicas run different micro-batches
    assert sum(res[0][3]) == sum(res[1][3]) == 32768


def test_job_throughput_and_single_rank():
    sys.path.insert(0, ROOT)
    import bench

    # two ranks of 3e12 useful FLOPs a step, 4 steps, slowest rank 8 ms: 3000 TFLOP/s
    assert bench.job_throughput(6e12, 4, 8.0) == pytest.approx(3000.0)
    times, flops = bench.aggregate_over_ranks([1.0, 2.0], 5, 1, "cpu")
    assert times == [1.0, 2.0] and flops == 5.0


def test_reference_arm_runs_on_rank_zero_only(capsys):
    """Under torchrun the reference arm (the oracle on host cores) runs and
    prints on rank 0; every other rank exits 0 without work or output."""
    sys.path.insert(0, ROOT)
    import argparse

    import bench

    args = argparse.Namespace(workload="tiny", seed=0, steps=1, warmup=3, gpus=2, mode="fused", cpu_seconds=0.1)
    assert bench.reference_arm(args, 1) == 0
    assert capsys.readouterr().out == ""


def test_gpus_flag_starts_that_many_ranks():
    """`bench.py --gpus 2` outside torchrun starts two ranks itself (torchrun,
    127.0.0.1); rank 0 alone prints, and the line's n_gpus is the world size.
    The reference arm (the oracle on host cores) needs no GPU, so the launcher
    runs here."""
    import json
    import subprocess

    env = {k: v for k, v in os.environ.items() if k not in ("WORLD_SIZE", "RANK", "LOCAL_RANK", "MASTER_ADDR",
                                                              "MASTER_PORT")}
    cmd = [sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2", "--workload",
           "tiny", "--steps", "1", "--warmup", "3", "--ref-step-seconds", "0.2"]
    r = subprocess.run(cmd, env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["n_gpus"] == 2


def test_gpus_flag_must_match_the_world_size(monkeypatch):
    sys.path.insert(0, ROOT)
    import bench

    monkeypatch.setenv("WORLD_SIZE", "3")
    monkeypatch.setenv("RANK", "0")
    monkeypatch.setenv("LOCAL_RANK", "0")
    with pytest.raises(SystemExit):
        bench.main(["--impl", "reference", "--gpus", "2", "--workload", "tiny"])
