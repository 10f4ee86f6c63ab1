"""The multi-rank host logic of bench.py, on CPU with gloo (world size 2):
each rank draws its own rows, the elapsed time is the maximum over ranks, the
whole-job value counts every rank's bytes over that time; and the reference
arm under torchrun runs on rank 0 only."""
import json
import os
import subprocess
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _rank_main(rank, world, port, results):
    sys.path.insert(0, ROOT)
    import bench
    from memory_bound_row_rmsnorm_gb300 import synthetic as syn

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # every rank's batch is its own: gather a fingerprint of set 0
        x = syn.normal_rows(64, 32, "f32", bench.rank_seed(rank, 0), "cpu")
        fp = torch.tensor([float(x.sum()), float(x[0, 0])], dtype=torch.float64)
        allfp = [torch.zeros_like(fp) for _ in range(world)]
        dist.all_gather(allfp, fp)
        # slowest rank decides the time
        mine = 10.0 + 5.0 * rank
        mx = bench.max_over_ranks(mine, dist, "cpu")
        results[rank] = (mx, [t.tolist() for t in allfp])
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks():
    world, port = 2, 29517 + os.getpid() % 1000
    mgr = mp.get_context("spawn").Manager()
    results = mgr.dict()
    mp.start_processes(_rank_main, args=(world, port, results), nprocs=world, start_method="spawn")
    (mx0, fps), (mx1, _) = results[0], results[1]
    assert mx0 == mx1 == 15.0
    assert fps[0] != fps[1], "ranks must draw different rows"


def test_whole_job_value_counts_every_rank():
    sys.path.insert(0, ROOT)
    import bench
    one = bench.whole_job_tbs(10 ** 9, 1, 100, 50.0)
    two = bench.whole_job_tbs(10 ** 9, 2, 100, 50.0)
    assert two == pytest.approx(2 * one)
    assert one == pytest.approx(10 ** 9 * 100 / 0.05 / 1e12)


def _reference(env_extra):
    env = dict(os.environ, **env_extra)
    return subprocess.run(
        [sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "2",
         "--warmup", "3", "--ref-seconds", "2", "--workload", "softmax_f32_1024x4096"],
        capture_output=True, text=True, env=env, timeout=300)


def test_reference_arm_prints_on_rank_zero_only():
    r1 = _reference({"WORLD_SIZE": "2", "RANK": "1", "LOCAL_RANK": "1"})
    assert r1.returncode == 0 and r1.stdout.strip() == ""
    r0 = _reference({"WORLD_SIZE": "2", "RANK": "0", "LOCAL_RANK": "0"})
    assert r0.returncode == 0, r0.stderr
    line = json.loads(r0.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["unit"] == "TB/s" and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["steps"] == 2
