"""bench.py's N > 1 path on the CPU, with gloo (no GPU).

Multi-GPU is replicas only: ranks run independent copies of the workload
and meet only to time it (a barrier, then the slowest rank's time). These
tests run two gloo ranks on the CPU:
* the timing reduction gives every rank the largest time, and the whole-job
  throughput counts every rank's bytes over that time;
* the reference arm under torchrun: rank 0 alone works and prints one JSON
  line, the other rank exits 0."""
import importlib.util
import json
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench():
    spec = importlib.util.spec_from_file_location("bench", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    bench = _bench()
    local_ms = [3.0, 7.5][rank]
    dist.barrier()
    got = bench.max_over_ranks(local_ms, world, dist, "cpu")
    q.put((rank, got, bench.throughput(10**9, world, got)))
    dist.barrier()
    dist.destroy_process_group()


def test_max_over_ranks_and_throughput_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
    assert all(p.exitcode == 0 for p in procs)
    res = sorted(q.get(timeout=5) for _ in range(2))
    assert [r[1] for r in res] == [7.5, 7.5]                    # both see the slowest rank
    assert res[0][2] == pytest.approx(2 * 10**9 / 7.5e-3 / 1e9)  # bytes of both ranks


def test_single_rank_needs_no_collective():
    bench = _bench()
    assert bench.max_over_ranks(4.25, 1, None, "cpu") == 4.25


def test_reference_arm_under_torchrun_prints_once():
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()),
           os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2",
           "--steps", "1", "--warmup", "0"]
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["value"] > 0 and d["e2e"]["h2d_bytes_per_step"] == 0
