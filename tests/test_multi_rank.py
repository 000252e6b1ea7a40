"""The benchmark's multi-process path on CPU (gloo, world size 2): the
attention step shards by request with no exchange, so N GPUs run N
replicas; what N > 1 adds is host logic -- rank set-up, the barrier around
the timed region and the max over ranks of the measured time -- and rank 0
alone printing the line.  No GPU is used."""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, ws, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(ws))
    sys.path.insert(0, ROOT)
    import bench
    r, n = bench.dist_init()
    bench.barrier(n)
    # each rank measured a different time; every rank must get the largest
    got = bench.allmax(1.5 + rank, n)
    bench.barrier(n)
    q.put((r, n, got))
    import torch.distributed as dist
    dist.destroy_process_group()


def test_allmax_and_barrier_over_two_gloo_ranks():
    import multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(2))
    assert res == [(0, 2, 2.5), (1, 2, 2.5)]


def test_reference_arm_under_torchrun_two_ranks():
    """`bench.py --impl reference --gpus 2` launched as the driver launches
    it: both ranks exit 0 and exactly one JSON line (rank 0's) is printed."""
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.join(ROOT, "bench.py"),
           "--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "1"]
    env = dict(os.environ, OMP_NUM_THREADS="2")
    out = subprocess.run(cmd, capture_output=True, text=True, timeout=600, cwd=ROOT, env=env)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [ln for ln in out.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, out.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
    for key in ("metric", "unit", "steps", "warmup", "ms_per_step", "higher_is_better", "config",
                "cpu_baseline", "e2e"):
        assert key in d
    # the same metric, unit, direction and config object as the GPU arm's line
    sys.path.insert(0, ROOT)
    import bench
    import synth
    assert d["metric"] == bench.METRIC and d["unit"] == "tokens/s" and d["higher_is_better"] is True
    assert d["config"] == json.loads(json.dumps(bench.headline_config(dict(synth.WORKLOADS[bench.WORKLOAD]))))
