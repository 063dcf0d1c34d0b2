"""The multi-rank parts of bench.py, run as two gloo ranks on the CPU.

Decode shards into independent (sequence, KV head) units with no exchange, so
N GPUs run N replicas.  What N > 1 adds is host logic: the barrier around the
timed region, the job time taken as the slowest rank's, the unit counts summed
over ranks, and the reference arm printing on rank 0 only.
"""
import json
import os
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _worker(rank, world, port, q):
    import torch
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        bench.barrier(world)
        # rank r "took" 1 + r seconds and processed 10 * (r + 1) units
        t = bench.max_over_ranks(1.0 + rank, world, torch.device("cpu"))
        n = bench.sum_over_ranks(10.0 * (rank + 1), world, torch.device("cpu"))
        bench.barrier(world)
        q.put((rank, t, n))
    finally:
        dist.destroy_process_group()


def _free_port():
    import socket
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_max_and_sum_over_two_gloo_ranks():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
    got = sorted(q.get(timeout=5) for _ in range(world))
    # every rank sees the slowest rank's time and the total of the units
    assert got == [(0, 2.0, 30.0), (1, 2.0, 30.0)]


def test_single_rank_helpers_are_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.5, 1) == 3.5
    assert bench.sum_over_ranks(7.0, 1) == 7.0
    bench.barrier(1)


def _reference_arm(rank, world):
    env = dict(os.environ, RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank),
               CUDA_VISIBLE_DEVICES="", OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1")
    cmd = [sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
           "--workload", "tiny_fp32_mha", "--steps", "2", "--warmup", "3"]
    return subprocess.run(cmd, env=env, capture_output=True, text=True, timeout=300)


def test_reference_arm_prints_on_rank_zero_only():
    r1 = _reference_arm(1, 2)
    assert r1.returncode == 0, r1.stderr
    assert not [x for x in r1.stdout.splitlines() if x.startswith("{")]
    r0 = _reference_arm(0, 2)
    assert r0.returncode == 0, r0.stderr
    lines = [json.loads(x) for x in r0.stdout.splitlines() if x.startswith("{")]
    assert len(lines) == 1
    d = lines[0]
    assert d["impl"] == "reference" and d["unit"] == "GB/s" and d["value"] > 0
    assert d["steps"] == 2 and d["warmup"] == 3
    assert d["cpu_baseline"]["kind"] == "oracle"
    assert d["e2e"] == {"value": d["value"], "unit": "GB/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}


@pytest.mark.parametrize("name", ["tiny_prefill_bf16", "chunked_prefill_7b_fp8",
                                  "chunked_prefill_7b_int8"])
def test_prefill_reference_arm(name):
    """The prefill reference arm (the oracle on sampled query rows; 8-bit caches
    through their codes) prints one TFLOP/s line."""
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="", OMP_NUM_THREADS="1",
               OPENBLAS_NUM_THREADS="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--workload", name, "--steps", "2", "--warmup", "3"],
                       env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    lines = [json.loads(x) for x in r.stdout.splitlines() if x.startswith("{")]
    assert len(lines) == 1
    d = lines[0]
    assert d["impl"] == "reference" and d["unit"] == "TFLOP/s" and d["value"] > 0
    assert d["config"]["workload"] == name and d["cpu_baseline"]["kind"] == "oracle"
