"""bench.py's host logic without a GPU: the replica arithmetic over ranks (two gloo processes),
and the reference arm's JSON line, alone and under torchrun with two ranks."""

import json
import os
import socket
import subprocess
import sys

import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    ms = [7.5, 9.25][rank]  # per-rank step times
    out[rank] = (bench.max_over_ranks_of(ms, world, "cpu"), bench.replica_seed(4, rank))
    dist.destroy_process_group()


def test_replicas_over_two_gloo_ranks():
    world = 2
    out = mp.Manager().dict()
    mp.spawn(_rank_main, args=(world, _free_port(), out), nprocs=world, join=True)
    # every rank sees the slowest rank's time; every rank draws its own problem
    assert out[0][0] == out[1][0] == 9.25
    assert out[0][1] == 4 and out[1][1] != out[0][1]
    # the job's value counts every rank's work over that time
    assert bench.job_tflops(1e12, world, 9.25) == 2 * bench.job_tflops(1e12, 1, 9.25)


def test_single_rank_needs_no_process_group():
    assert bench.max_over_ranks_of(3.0, 1, "cpu") == 3.0


def _reference_lines(cmd):
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    return [json.loads(ln) for ln in r.stdout.splitlines() if ln.startswith("{")]


REF_ARGS = ["--impl", "reference", "--shape", "1,4,2,128,64", "--steps", "1", "--warmup", "0"]


def test_reference_arm_line():
    (line,) = _reference_lines([sys.executable, "bench.py"] + REF_ARGS)
    assert line["impl"] == "reference" and line["n_gpus"] == 1 and line["value"] > 0
    assert line["metric"] == bench.METRIC and line["unit"] == "TFLOP/s" and line["higher_is_better"] is True
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["value"] == line["value"]
    assert line["e2e"] == {"value": line["value"], "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                           "d2h_bytes_per_step": 0}


def test_reference_arm_under_torchrun_prints_once():
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()), "bench.py", "--gpus", "2"] + REF_ARGS
    lines = _reference_lines(cmd)
    assert len(lines) == 1 and lines[0]["impl"] == "reference" and lines[0]["n_gpus"] == 2
