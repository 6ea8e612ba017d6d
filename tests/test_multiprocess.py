"""The multi-process host logic of bench.py on CPU (gloo, world size 2).

The product does not shard (every configuration fits one GPU), so N GPUs run
N independent replicas: each rank times its own steps, the job's time is the
largest over ranks, and the job's rate counts every rank's work.  These
tests run that logic on two CPU processes with the gloo backend, and check
that the reference arm's extra ranks leave without work or output."""
import os
import socket
import subprocess
import sys

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    r, w, lr = bench.dist_env()
    local_ms = 10.0 + 5.0 * rank                 # rank 1 is the slower replica
    job_ms = bench.max_over_ranks(local_ms, dist)
    rate = bench.job_rate(1000.0, 4, w, job_ms)
    dist.barrier()
    dist.destroy_process_group()
    with open(out, "w") as f:
        f.write(f"{r} {w} {lr} {job_ms} {rate}\n")


def test_timing_is_max_over_ranks_and_rate_counts_all(tmp_path):
    import torch.multiprocessing as mp
    port = _free_port()
    outs = [str(tmp_path / f"r{i}.txt") for i in range(2)]
    ctx = mp.get_context("spawn")
    procs = [ctx.Process(target=_worker, args=(i, 2, port, outs[i])) for i in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    for i, o in enumerate(outs):
        r, w, lr, job_ms, rate = open(o).read().split()
        assert (int(r), int(w), int(lr)) == (i, 2, i)
        assert float(job_ms) == 15.0                       # the slower rank's time, on both
        assert float(rate) == pytest.approx(1000.0 * 4 * 2 / 0.015)


def test_single_process_defaults():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.5) == 3.5
    assert bench.job_rate(10.0, 2, 1, 1000.0) == 20.0


def test_reference_arm_extra_rank_exits_quietly():
    """Under torchrun only rank 0 runs and prints the reference line."""
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--gpus", "2", "--steps", "1", "--warmup", "0",
                        "--workload", "tiny_uniform"],
                       capture_output=True, text=True, env=env, timeout=300)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == ""
