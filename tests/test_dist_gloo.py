"""Multi-rank host logic of the benchmark on CPU (gloo, world size 2): each
rank runs its own replica of the workload, the job's step time is the
slowest rank's, and the job's throughput is the sum over replicas."""
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


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ms = bench.max_over_ranks(1.0 + rank * 0.5)
    gbs = bench.job_throughput(2e9, ms, world)
    dist.barrier()
    q.put((rank, ms, gbs))
    dist.destroy_process_group()


def test_two_rank_replicas_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(2))
    assert [r[1] for r in res] == [1.5, 1.5]                  # max over ranks
    assert all(abs(r[2] - 2 * 2e9 / 1.5e-3 / 1e9) < 1e-6 for r in res)


def test_single_process_passthrough():
    import bench
    assert bench.max_over_ranks(3.25) == 3.25
    assert bench.job_throughput(1e9, 2.0, 1) == pytest.approx(500.0)


def test_gpus_flag_without_torchrun_starts_replicas():
    # --gpus 2 outside torchrun starts two local replica processes with the
    # rendezvous variables set; only rank 0 prints, and the line reports both
    import json
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    env = {k: v for k, v in os.environ.items() if k not in ("RANK", "WORLD_SIZE", "LOCAL_RANK", "MASTER_PORT")}
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--gpus", "2", "--steps", "1",
                        "--warmup", "0", "--workload", "taco_tiny", "--ref-rows", "8"],
                       cwd=root, env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["n_gpus"] == 2
