"""The N > 1 path of bench.py on CPU: gloo ranks (world size 2) for the
barrier, the max over ranks and the whole-job throughput of independent
replicas, and the reference arm launched by torchrun."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, world: int, port: int, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    sys.path.insert(0, ROOT)
    import torch
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        bench._barrier(dist)
        seconds = [2.0, 3.0][rank]                  # the second replica is slower
        m = bench._max_over_ranks(dist, seconds, torch.device("cpu"))
        v = bench._job_throughput(dist, world, 100, seconds, torch.device("cpu"))
        bench._barrier(dist)
        q.put((rank, m, v))
    finally:
        dist.destroy_process_group()


def test_replica_aggregation_over_gloo_ranks():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(world))
    for rank, m, v in got:
        assert m == 3.0                              # every rank sees the slowest time
        assert v == pytest.approx(2 * 100 / 3.0)     # all ranks' tokens over it


def test_reference_arm_under_torchrun_prints_one_line():
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py", "--impl", "reference",
           "--gpus", "2", "--steps", "1", "--warmup", "0", "--ref-step-seconds", "0.2", "--workload", "tiny"]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1                           # rank 0 alone prints
    j = json.loads(lines[0])
    assert j["impl"] == "reference" and j["n_gpus"] == 2 and j["value"] > 0
    assert j["e2e"]["h2d_bytes_per_step"] == 0 and j["cpu_baseline"]["kind"] == "oracle"
    # the same config object as the measured arm prints for this workload and world size
    sys.path.insert(0, ROOT)
    import bench
    from moe_layer_bit_gb300 import workloads as wk
    assert j["config"] == bench.bench_config(wk.by_name("tiny"), 2)
