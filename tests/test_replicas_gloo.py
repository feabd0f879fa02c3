"""The N-GPU path of bench.py is N independent replicas: a barrier and a
max over ranks around the timed region, whole-job tokens/s = N x tokens per
rank / the slowest rank's time.  Checked here with two gloo ranks on the
CPU (the timing helpers bench.py uses), and the reference arm's rule that
only rank 0 runs under torchrun."""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _rank_main(rank, world, port, out):
    import torch.distributed as tdist
    sys.path.insert(0, ROOT)
    import bench
    tdist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    local_s = [0.5, 2.0][rank]                       # rank 1 is the slow one
    slowest = bench.max_over_ranks(local_s, "cpu")
    rate = bench.whole_job_rate(64 * 10, slowest, world)
    tdist.barrier()
    tdist.destroy_process_group()
    out.put((rank, slowest, rate))


def test_two_gloo_ranks_take_the_slowest_rank_and_sum_the_tokens():
    import torch.multiprocessing as mp
    port = 29500 + os.getpid() % 1000
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, slowest, rate in res:
        assert slowest == 2.0
        assert rate == pytest.approx(2 * 640 / 2.0)


def test_reference_arm_runs_on_rank_zero_only():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "0", "--ref-budget", "0.5"], env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0
    assert r.stdout.strip() == ""
