"""Multi-process (replicas) logic of bench.py on the CPU: two ranks over gloo.

The forward pass has no data-path collective (every rank runs its own batch,
weak scaling); what the N > 1 path needs is the rendezvous, the barrier around
the timed region, the max over ranks of the measured time, and the reference
arm printing once.  These run here with world size 2 on 127.0.0.1.
"""
import io
import json
import multiprocessing as mp
import os
import socket
import sys
from contextlib import redirect_stdout

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _env(rank, ws, port):
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(ws), LOCAL_RANK=str(rank),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)


def _barrier_worker(rank, ws, port, q):
    _env(rank, ws, port)
    import torch
    import bench
    w, r, local = bench.dist_setup()
    bench.barrier(w)
    # each rank reports a different time; every rank must see the slowest
    m = bench.max_over_ranks(1.5 * (rank + 1), w, torch.device("cpu"))
    bench.barrier(w)
    q.put((r, w, local, m))
    torch.distributed.destroy_process_group()


def _reference_worker(rank, ws, port, q):
    _env(rank, ws, port)
    import argparse
    import torch
    import bench
    args = argparse.Namespace(gpus=ws, steps=1, warmup=1)
    buf = io.StringIO()
    with redirect_stdout(buf):
        bench.run_reference_arm(args, bench.WORKLOADS["tiny_moe_f32"])
    q.put((rank, buf.getvalue()))
    if torch.distributed.is_initialized():
        torch.distributed.destroy_process_group()


def _run(target, ws=2):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=target, args=(r, ws, port, q)) for r in range(ws)]
    for p in procs:
        p.start()
    out = [q.get(timeout=180) for _ in range(ws)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    return sorted(out)


def test_two_ranks_meet_and_take_the_max_time():
    res = _run(_barrier_worker)
    assert [r[0] for r in res] == [0, 1]
    assert all(r[1] == 2 for r in res)
    assert [r[2] for r in res] == [0, 1]
    assert all(r[3] == pytest.approx(3.0) for r in res)


def test_reference_arm_prints_once_under_two_ranks():
    res = _run(_reference_worker)
    assert res[1][1] == ""                         # rank 1 exits without output
    line = json.loads(res[0][1].strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["n_gpus"] == 2
    assert line["value"] > 0 and line["cpu_baseline"]["kind"] == "oracle"
    assert line["e2e"]["h2d_bytes_per_step"] == 0
    # the same config object as the GPU arm prints for this workload
    sys.path.insert(0, ROOT)
    import bench
    assert line["config"] == bench.workload_config(bench.WORKLOADS["tiny_moe_f32"], 2)
