"""The multi-rank host path of bench.py on CPU (gloo, world size 2).

On a GPU node each rank runs one replica of the workload (weak scaling, no
collective on the data path); the only cross-rank steps are the barriers
around the timed region and the max over ranks of the elapsed time.  These
tests run those steps with the gloo backend in two spawned processes, and run
the reference arm under torchrun to check that rank 0 alone prints its line.
"""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, world: int, port: int, out_dir: str):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    w, r, local = bench.dist_setup()
    assert (w, r, local) == (world, rank, rank)
    bench.dist_init(w, "gloo")
    bench.barrier(w)
    elapsed = 10.0 + 5.0 * rank                      # rank 1 is the slow one
    worst = bench.max_over_ranks(elapsed, w, torch.device("cpu"))
    bench.barrier(w)
    with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as f:
        json.dump({"worst": worst}, f)
    import torch.distributed as dist
    dist.destroy_process_group()


def test_barrier_and_max_over_ranks_gloo(tmp_path):
    port = _free_port()
    mp.start_processes(_rank_main, args=(2, port, str(tmp_path)), nprocs=2, join=True, start_method="spawn")
    for rank in range(2):
        with open(tmp_path / f"rank{rank}.json") as f:
            assert json.load(f)["worst"] == 15.0, rank      # every rank sees the slowest rank's time


def test_reference_arm_prints_once_under_torchrun(tmp_path):
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes", "1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py", "--impl", "reference",
           "--workload", "c1", "--steps", "1", "--warmup", "3", "--reference-rows", "4"]
    p = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert p.returncode == 0, p.stderr[-2000:]
    lines = [ln for ln in p.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, p.stdout
    rec = json.loads(lines[0])
    assert rec["impl"] == "reference" and rec["n_gpus"] == 2 and rec["value"] > 0
    assert rec["cpu_baseline"]["kind"] == "oracle"
