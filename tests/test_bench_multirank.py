"""bench.py's multi-rank logic on CPU: world size 2 over gloo (no GPU). Ranks run independent replicas
of the workload; the job's time is the slowest rank's and its value counts every rank's units."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, ws, port, q):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(ws))
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    import bench
    local_ms = [12.5, 20.0][rank]
    mx = bench.max_over_ranks(local_ms, ws)
    dist.barrier()
    q.put((rank, mx, bench.whole_job_rate(1_000_000, mx * 1e-3, ws)))
    dist.destroy_process_group()


def _short_worker(rank, ws, port, q):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(ws))
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    import bench
    # rank 1 asks for more host memory than any machine has; rank 0 for one byte
    q.put((rank, bench._e2e_host_memory_short(1 if rank == 0 else 10**18, ws)))
    dist.destroy_process_group()


def test_e2e_host_memory_decision_is_collective_gloo():
    """A rank that cannot pin its gradients leaves the end-to-end leg out on every rank, so no rank waits at
    that leg's barrier for one that skipped it."""
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_short_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = dict(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert out[1].startswith("host memory:") and "GB available" in out[1]
    assert out[0] == "host memory: another rank of this job has too little to pin its gradients"


def test_host_memory_short_alone():
    sys.path.insert(0, ROOT)
    import bench
    assert bench._e2e_host_memory_short(1, 1) is None
    assert bench._host_memory_short(10**18, 1).startswith("host memory: 1 rank(s)")


def test_max_over_ranks_and_whole_job_rate_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [o[1] for o in out] == [20.0, 20.0]          # both ranks see the slowest rank's time
    assert all(abs(o[2] - 2 * 1_000_000 / 0.020 / 1e9) < 1e-12 for o in out)


def test_single_rank_helpers():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.0, 1) == 3.0
    assert bench.whole_job_rate(10 ** 9, 2.0, 1) == 0.5


def test_reference_arm_rank1_exits_silently():
    """Under torchrun only rank 0 runs the reference arm and prints; other ranks exit 0 without output."""
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "3",
                        "--warmup", "3", "--workload", "tiny"], capture_output=True, text=True, env=env, timeout=300)
    assert r.returncode == 0 and r.stdout.strip() == ""


def test_reference_arm_rank0_prints_one_line():
    env = dict(os.environ, RANK="0", WORLD_SIZE="1", LOCAL_RANK="0")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "3",
                        "--warmup", "3", "--workload", "tiny"], capture_output=True, text=True, env=env, timeout=600)
    assert r.returncode == 0, r.stderr
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["value"] > 0 and line["cpu_baseline"]["kind"] == "oracle"
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["unit"] == "Gparams/s"
