"""The multi-replica path of bench.py (N > 1 ranks), run as two gloo ranks on the CPU.

bench.py --gpus N runs N independent replicas of the decode step: the method
has no data exchange between GPUs ("replicas only").  The only cross-rank
steps are a barrier around the timed region, the maximum of the ranks'
times, and the whole-job rate (all ranks' bytes over the slowest rank's
time).  These are checked here with world_size 2 over gloo.
"""

import importlib.util
import os
import socket

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench():
    spec = importlib.util.spec_from_file_location("bench_under_test", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        b = _bench()
        b.rank_barrier(world)
        ms = 2.0 + rank  # rank 1 is the slower one
        slowest = b.rank_max(ms, world, device="cpu")
        rate = b.job_rate(1e6, world, slowest)
        b.rank_barrier(world)
        out.put((rank, slowest, rate))
    finally:
        dist.destroy_process_group()


def test_two_ranks_take_the_slowest_time_and_add_their_units():
    torch = pytest.importorskip("torch")
    mp = torch.multiprocessing.get_context("spawn")
    world, port = 2, _free_port()
    q = mp.Queue()
    procs = [mp.Process(target=_rank, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    assert all(p.exitcode == 0 for p in procs)
    res = sorted(q.get(timeout=5) for _ in range(world))
    for rank, slowest, rate in res:
        assert slowest == 3.0  # max over ranks, the same on every rank
        assert rate == pytest.approx(2 * 1e6 / 3e-3)  # both ranks' units over the slowest time


def test_one_rank_is_the_identity():
    b = _bench()
    assert b.rank_max(4.5, 1) == 4.5
    b.rank_barrier(1)
    assert b.job_rate(10.0, 1, 2.0) == pytest.approx(5000.0)


def test_reference_arm_runs_on_rank_zero_only():
    """Under torchrun the oracle arm runs and prints on rank 0 alone; the other ranks exit 0 at once."""
    import subprocess
    import sys
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2",
                          "--steps", "1", "--warmup", "3"], capture_output=True, text=True, env=env, cwd=ROOT,
                         timeout=120)
    assert out.returncode == 0, out.stderr[-2000:]
    assert out.stdout.strip() == ""
