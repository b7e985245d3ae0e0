"""Multi-process host logic of the benchmark on CPU (gloo, world size 2).

The operation has no cross-GPU exchange: under torchrun every rank runs an
independent replica and the only collective is the timing reduction (the
slowest rank's time) plus barriers.  These tests run that logic with the gloo
backend on CPU, and check that the reference arm prints from rank 0 only.
"""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _worker(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    sys.path.insert(0, ROOT)
    import bench
    out = bench.reduce_max([1.0 + rank, 10.0 - rank], world)
    dist.barrier()
    q.put((rank, out))
    dist.destroy_process_group()


def test_reduce_max_over_two_gloo_ranks():
    import multiprocessing as mp
    import socket
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = dict(q.get(timeout=120) for _ in range(2))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert res[0] == res[1] == [2.0, 10.0]


def test_reference_arm_prints_on_rank0_only():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--config", "1",
                        "--steps", "3", "--warmup", "3"], env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0 and r.stdout.strip() == ""
    env = dict(os.environ, RANK="0", WORLD_SIZE="1", LOCAL_RANK="0")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--config", "1",
                        "--steps", "3", "--warmup", "3"], env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["unit"] == "GB/s" and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["e2e"]["h2d_bytes_per_step"] == 0


def test_bench_rejects_short_warmup():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--warmup", "2"],
                       capture_output=True, text=True, timeout=120)
    assert r.returncode != 0


def test_clock_sampling_follows_visible_devices(monkeypatch):
    """nvidia-smi is asked about the physical GPU behind CUDA device `local`."""
    sys.path.insert(0, ROOT)
    import bench
    monkeypatch.setenv("CUDA_VISIBLE_DEVICES", "3, 5")
    assert bench.smi_index(0) == "3" and bench.smi_index(1) == "5"
    monkeypatch.delenv("CUDA_VISIBLE_DEVICES")
    assert bench.smi_index(1) == "1"


def test_nominal_hbm_query_never_raises():
    """The second roofline denominator comes from CUDA device attributes; with
    no device (or no runtime) it is None rather than an error or a guess."""
    sys.path.insert(0, ROOT)
    import bench
    v = bench.nominal_hbm_gbs(0)
    assert v is None or v > 0
