"""The replica path of bench.py on CPU: two processes over gloo (127.0.0.1), as
torchrun launches them on a GPU node (one replica per GPU, no gradient
exchange).  Checked: the replicas read disjoint token windows of the stream,
the job's time is the slowest replica's (all ranks agree on it), the job's
throughput counts every replica's tokens, and the reference arm runs on rank
0 only."""
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    import torch.distributed as dist

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = 10.0 + 5.0 * rank  # rank 1 is the slow one
        job = bench.max_over_ranks(ms, dist, "cpu")
        out.put((rank, job, bench.rank_micro_steps(rank, 7, 3)))
    finally:
        dist.destroy_process_group()


def test_two_replicas_over_gloo():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = [q.get(timeout=120) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    res.sort()
    assert [r[1] for r in res] == [15.0, 15.0]  # every rank reports the slowest replica's time
    w0 = {m for row in res[0][2] for m in row}
    w1 = {m for row in res[1][2] for m in row}
    assert len(w0) == len(w1) == 7 * 3 and not (w0 & w1)
    # throughput of the whole job: both replicas' tokens over the slowest time
    assert bench.job_throughput(2, 20, 16384, 15.0 * 20) == pytest.approx(2 * 20 * 16384 / 0.3)


def test_single_process_needs_no_collective():
    assert bench.max_over_ranks(12.5, None, "cpu") == 12.5
    assert bench.rank_micro_steps(0, 2, 2) == [[0, 1], [2, 3]]


def test_reference_arm_runs_on_rank_zero_only():
    """Under torchrun the reference arm's other ranks exit 0 without work or output."""
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2",
                        "--steps", "1", "--warmup", "1"], env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0
    assert r.stdout.strip() == ""
