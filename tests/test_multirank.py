"""The N > 1 host logic of bench.py, run as two gloo ranks on the CPU.

On N GPUs every rank publishes its own batch into its own replicas (weak
scaling, no data-path collective).  The host side takes a barrier around
the timed region, the maximum of the ranks' times, and reports all ranks'
rows over that maximum; only rank 0 prints.  The reference arm runs on
rank 0 alone and the other ranks exit without work.
"""

import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out_dir):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench

    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank,
                            world_size=world)
    try:
        bench.barrier()
        slowest = bench.max_over_ranks(1.5 + rank)        # rank 1 is the slow one
        value = bench.whole_job_rate(world, 1000.0, slowest)
        bench.barrier()
        with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as f:
            json.dump({"slowest": slowest, "value": value}, f)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_max_time_and_sum_the_work(tmp_path):
    world, port = 2, _free_port()
    mp.start_processes(_rank, args=(world, port, str(tmp_path)), nprocs=world,
                       start_method="spawn", join=True)
    got = [json.load(open(tmp_path / f"rank{r}.json")) for r in range(world)]
    for g in got:
        assert g["slowest"] == pytest.approx(2.5)
        # 2 ranks x 1000 units in 2.5 ms
        assert g["value"] == pytest.approx(2 * 1000 / 2.5e-3)


def test_reference_arm_runs_on_rank_zero_only():
    env = dict(os.environ, WORLD_SIZE="2", RANK="1", LOCAL_RANK="1")
    res = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--steps", "3", "--warmup", "3"], env=env, capture_output=True,
                         text=True, timeout=120)
    assert res.returncode == 0
    assert res.stdout.strip() == ""


def test_gpus_two_relaunches_under_torchrun_and_prints_one_line():
    """--gpus 2 outside torchrun starts two local ranks; the reference arm
    runs on rank 0 alone, so exactly one JSON line comes back, for 2 GPUs."""
    env = {k: v for k, v in os.environ.items()
           if k not in ("WORLD_SIZE", "RANK", "LOCAL_RANK", "MASTER_ADDR", "MASTER_PORT")}
    res = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--gpus", "2", "--steps", "3", "--warmup", "3", "--ref-seconds", "1"],
                         env=env, capture_output=True, text=True, timeout=300)
    assert res.returncode == 0, res.stderr[-2000:]
    lines = [l for l in res.stdout.splitlines() if l.strip()]
    assert len(lines) == 1, res.stdout
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["n_gpus"] == 2


def test_single_process_rate_is_units_over_time():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.whole_job_rate(1, 3_497_984, 0.768) == pytest.approx(3_497_984 / 0.768e-3)
    assert bench.max_over_ranks(4.0) == 4.0       # no process group: identity
