"""The multi-rank host path of bench.py on CPU: world_size-2 gloo process groups.

Every box of this build has one GPU, so `bench.py --gpus N` runs N independent replicas. The
replicas' only interaction is host-side: a barrier before the timed region, the maximum of the
per-rank times (the slowest rank sets the job's time), and rank 0 alone printing the line.
These tests run that logic with gloo on the host, no GPU involved.
"""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.distributed as tdist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    sys.path.insert(0, ROOT)
    import bench

    tdist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        bench.barrier()
        got = bench.max_over_ranks(1.5 + rank * 2.25)  # ranks report 1.5 and 3.75 ms
        same = bench.max_over_ranks(7.0)
        out[rank] = (got, same)
    finally:
        tdist.destroy_process_group()


def test_max_over_ranks_with_gloo_world_2():
    port = _free_port()
    manager = mp.get_context("spawn").Manager()
    out = manager.dict()
    mp.start_processes(_rank_main, args=(2, port, out), nprocs=2, join=True, start_method="spawn")
    assert dict(out) == {0: (3.75, 7.0), 1: (3.75, 7.0)}


def test_max_over_ranks_without_a_group_is_the_identity():
    sys.path.insert(0, ROOT)
    import bench

    assert not tdist.is_initialized()
    assert bench.max_over_ranks(2.5) == 2.5
    bench.barrier()  # no group: a no-op
    assert bench.process_group_backend() == ("nccl" if torch.cuda.is_available() else "gloo")


@pytest.mark.skipif(torch.cuda.is_available(), reason="the launch below uses gloo ranks on a host without GPUs")
def test_reference_arm_under_torchrun_prints_one_line_from_rank_0():
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py", "--impl", "reference",
           "--config", "conv_block", "--gpus", "2", "--steps", "1", "--warmup", "0", "--ref-budget", "1"]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=240)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    rec = json.loads(lines[0])
    assert rec["impl"] == "reference" and rec["n_gpus"] == 2 and rec["metric"] == "conv_hbm_gbs"
    assert rec["cpu_baseline"]["kind"] == "oracle" and rec["e2e"]["h2d_bytes_per_step"] == 0
