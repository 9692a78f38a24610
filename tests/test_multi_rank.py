"""The multi-GPU path's host logic (one process per GPU, each decoding its
own sequences, the step time taken as the maximum over ranks), run as two
gloo ranks on the CPU.  The path has no data exchange, so this is all there
is to its N > 1 behaviour besides the launch itself."""
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    import synthetic as syn
    ms = 10.0 + 2.5 * rank  # the second rank is the slower one
    slowest = bench.max_over_ranks(ms, world, "cpu")
    value = bench.job_value(world, 64, 100, slowest)
    cfg = bench.rank_config(2, rank)
    qI = syn.indexer_query(cfg, 2, 1)["qI"].view(torch.uint8)
    out.put((rank, slowest, value, cfg, int(qI.long().sum())))
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_shard_by_sequence_and_time_by_the_slowest():
    ctx = mp.get_context("spawn")
    out = ctx.SimpleQueue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    res = sorted(out.get() for _ in range(2))
    (r0, m0, v0, c0, s0), (r1, m1, v1, c1, s1) = res
    assert (r0, r1) == (0, 1)
    assert m0 == m1 == 12.5                      # both ranks see the slowest rank's time
    assert v0 == v1 == pytest.approx(2 * 64 * 100 / 12.5e-3)  # whole-job queries/s
    assert c0 != c1 and s0 != s1                 # each rank draws its own sequences


def test_reference_arm_prints_on_rank_zero_only():
    env = dict(os.environ, WORLD_SIZE="2", RANK="1", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference"], env=env,
                       capture_output=True, text=True, timeout=120)
    assert r.returncode == 0
    assert r.stdout.strip() == ""


def test_the_faster_launch_form_gives_the_value():
    """bench.py times the decode loop eagerly and as replayed CUDA graphs and
    reports the faster per step; without a graph it keeps the eager timing."""
    import bench
    assert bench.pick_launch(170.0, 2000, 164.0, 1984)[::3] == (1984, True)  # graphs faster per step
    assert bench.pick_launch(170.0, 2000, 171.0, 1984)[::3] == (2000, False)  # eager faster per step
    assert bench.pick_launch(170.0, 2000, None, 0) == (2000, 170.0, "eager stream launches", False)
