"""The multi-rank path of bench.py on CPU: two gloo ranks (world size 2).

The layer is token-parallel, so N GPUs run N replicas on their own tokens with
no collective on the data path; the only cross-rank steps are the barrier and
the max over ranks of the timed region.  These tests check that host logic."""
import json
import os
import socket
import subprocess
import sys
from pathlib import Path

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench
import workloads as W

ROOT = Path(__file__).resolve().parents[1]


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    w = W.WORKLOADS["tiny"]
    hidden = bench.replica_hidden(w, rank)
    local_ms = 10.0 + 5.0 * rank           # the slower rank decides
    slowest = bench.max_over_ranks(local_ms, world, torch.device("cpu"))
    dist.barrier()
    res = {"rank": rank, "slowest": slowest, "hidden_sum": int(hidden.astype(np.int64).sum()),
           "value": bench.job_throughput(world, w.T, 7, slowest)}
    Path(out_dir, f"r{rank}.json").write_text(json.dumps(res))
    dist.destroy_process_group()


def test_two_gloo_ranks_max_time_and_distinct_tokens(tmp_path):
    world = 2
    mp.start_processes(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world, start_method="spawn")
    r = [json.loads((tmp_path / f"r{i}.json").read_text()) for i in range(world)]
    assert r[0]["slowest"] == r[1]["slowest"] == 15.0
    assert r[0]["hidden_sum"] != r[1]["hidden_sum"]          # each replica has its own tokens
    w = W.WORKLOADS["tiny"]
    assert r[0]["value"] == pytest.approx(world * w.T * 7 / 15e-3)
    # rank 0's tokens are the workload's own (a one-GPU run is the workload itself)
    assert np.array_equal(bench.replica_hidden(w, 0), W.router_inputs(w)[0])


def test_reference_arm_runs_on_rank0_only():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    p = subprocess.run([sys.executable, str(ROOT / "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "3"], env=env, capture_output=True, text=True, timeout=120)
    assert p.returncode == 0
    assert p.stdout.strip() == ""                               # no work, no line, on ranks > 0


def test_single_rank_is_a_noop_reduction():
    assert bench.max_over_ranks(3.5, 1) == 3.5
