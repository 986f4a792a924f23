"""Host-side checks of the multi-GPU path, which is replicas only (each GPU
runs its own sequences; no exchange on the data path): two gloo ranks on the
CPU go through bench.py's process-group set-up, barrier, max-over-ranks timing
and whole-job aggregation, and the reference arm does its work on rank 0 only."""
import json
import os
import socket
import sys

import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(world), RANK=str(rank),
                      LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import argparse
    import torch.distributed as dist
    import bench
    w, r, local = bench.dist_setup(world)
    backend = dist.get_backend()
    bench.barrier(w)
    slowest = bench.max_over_ranks(w, 10.0 + rank)  # rank 1 is the slow one
    gbs = bench.whole_job_gbs(w, 1 << 30, slowest)
    # the reference arm: rank 0 works and prints, the others return at once
    ran = False
    if r != 0:
        args = argparse.Namespace(steps=1, warmup=0, reference_budget=1.0)
        bench.bench_reference(args, w, r)
        ran = True
    bench.barrier(w)
    dist.destroy_process_group()
    with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as f:
        json.dump({"world": w, "rank": r, "backend": backend, "slowest": slowest, "gbs": gbs,
                   "reference_returned": ran}, f)


@pytest.mark.skipif(torch.cuda.is_available(), reason="host-side test: with a GPU the group would use NCCL")
def test_two_gloo_replicas(tmp_path):
    world = 2
    mp.start_processes(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world, start_method="spawn")
    recs = [json.load(open(tmp_path / f"rank{r}.json")) for r in range(world)]
    for r, rec in enumerate(recs):
        assert rec["world"] == world and rec["rank"] == r and rec["backend"] == "gloo"
        assert rec["slowest"] == 11.0  # the max over ranks, seen by every rank
        assert rec["gbs"] == pytest.approx(2 * (1 << 30) / 11e-3 / 1e9)
    assert recs[1]["reference_returned"] is True


def test_reference_arm_line(tmp_path):
    """The reference arm (the oracle on the host cores) prints one JSON line
    with the contract's keys, runs at least 3 warm-up steps, reports the
    metric of the decode arm, and times whole steps of every layer: its
    ms_per_step times its steps fits inside the run's own wall time (here a
    2-layer step keeps the CPU suite short)."""
    import subprocess
    import time
    cmd = [sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "2", "--warmup", "0",
           "--reference-budget", "5", "--layers", "2"]
    t0 = time.perf_counter()
    res = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600)
    wall = time.perf_counter() - t0
    assert res.returncode == 0, res.stderr[-2000:]
    lines = [l for l in res.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    rec = json.loads(lines[0])
    assert rec["impl"] == "reference" and rec["n_gpus"] == 1 and rec["warmup"] >= 3
    assert rec["unit"] == "GB/s" and rec["higher_is_better"] is True and rec["value"] > 0
    assert rec["config"]["workload"] == "hybrid_step_l32768_bs784_x16"
    assert rec["cpu_baseline"]["kind"] == "oracle" and rec["cpu_baseline"]["cores"] >= 1
    assert rec["cpu_baseline"]["value"] == rec["value"]
    assert rec["e2e"] == {"value": rec["value"], "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
    assert rec["config"]["layers"] == 2 and 1 <= rec["steps"] <= 2
    assert (rec["steps"] + rec["warmup"]) * rec["ms_per_step"] * 1e-3 <= wall
    # the value is the bytes of a whole step over the measured step time
    bytes_step = 2 * 32768 * 4096
    assert rec["value"] == pytest.approx(bytes_step / (rec["ms_per_step"] * 1e-3) / 1e9, rel=1e-9)
