"""The benchmark's multi-rank path on the CPU, with two gloo ranks.

bench.py runs one independent replica per rank under torchrun. The job's time is that of
the slowest rank (an all-reduce MAX), and the job's throughput counts every rank's units.
The reference arm runs on rank 0 alone. No GPU is needed for either check.
"""
import json
import os
import socket
import subprocess
import sys

import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, times, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import importlib.util
    spec = importlib.util.spec_from_file_location("bench", os.path.join(ROOT, "bench.py"))
    bench = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(bench)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        slowest = bench.max_over_ranks(times[rank], world)
        rate = bench.job_rate(64, 10, world, slowest)
        q.put((rank, slowest, rate))
    finally:
        dist.destroy_process_group()


def test_slowest_rank_sets_the_job_time():
    world, times = 2, [3.5, 7.25]
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, times, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(world))
    for rank, slowest, rate in got:
        assert slowest == max(times)
        # 64 tokens x 10 steps on each of 2 ranks over the slowest rank's 7.25 ms
        assert abs(rate - 64 * 10 * 2 / 7.25e-3) < 1e-6 * rate


def test_reference_arm_under_torchrun_runs_on_rank_zero_only():
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(free_port()), os.path.join(ROOT, "bench.py"),
           "--impl", "reference", "--workload", "b1_l512", "--steps", "1", "--warmup", "3", "--ref-seqs", "1"]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [json.loads(l) for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    line = lines[0]
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle"
