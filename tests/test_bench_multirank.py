"""Host-side logic of bench.py's multi-GPU path, on CPU with the gloo backend.

With N > 1 the bench runs N independent replicas (the convolution has no
cross-GPU exchange on one node here): every rank times its own steps, the job
time is the slowest rank's (all-reduce MAX) and the throughput counts every
rank's units.  The reference arm runs on rank 0 alone; other ranks exit without
work.  Two gloo ranks on 127.0.0.1 check both.
"""

import os
import socket
import subprocess
import sys

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms_local = [4.0, 6.5][rank]
        ms, value = bench.job_throughput(ms_local, 320_000, world)
        q.put((rank, ms, value))
    finally:
        dist.destroy_process_group()


def test_job_throughput_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=5) for _ in range(2))
    for rank, ms, value in got:
        assert ms == 6.5                              # the slowest rank sets the job time
        assert value == pytest.approx(2 * 320_000 / 6.5e-3)


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    ms, value = bench.job_throughput(5.0, 1000, 1)
    assert ms == 5.0 and value == pytest.approx(1000 / 5e-3)


def test_reference_arm_runs_on_rank_zero_only():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "0"], env=env, capture_output=True, text=True,
                       timeout=120)
    assert r.returncode == 0
    assert r.stdout.strip() == ""
