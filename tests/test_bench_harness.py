"""bench.py's host logic on CPU: the replica aggregation over world_size 2 with
gloo, and the reference arm (the oracle) end to end."""
import json
import os
import subprocess
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _worker(rank, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE="2", LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=2)
    try:
        # rank 0 processed 100 rows in 50 ms, rank 1 300 rows in 200 ms
        rows, ms = (100.0, 50.0) if rank == 0 else (300.0, 200.0)
        value, slowest = bench.replica_throughput(rows, ms, 2)
        bench.barrier_sync(2)
        out[rank] = (value, slowest)
    finally:
        dist.destroy_process_group()


def test_replica_throughput_gloo_world_size_2():
    port = 29500 + os.getpid() % 1000
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_worker, args=(port, out), nprocs=2, join=True)
        results = dict(out)
    for rank in (0, 1):
        value, slowest = results[rank]
        assert slowest == 200.0
        assert value == pytest.approx(400.0 / 0.2)  # all rows over the slowest rank's time


def test_reference_arm_prints_one_json_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "2", "--warmup", "3", "--ref-rows", "8"],
                       capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "rows/s" and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["value"] == d["value"]
    assert d["config"]["workload"] == "ce_bf16_16384x128256"


def test_workload_entry_arithmetic():
    sys.path.insert(0, ROOT)
    import bench
    e = bench.entry("w", "k", 2.0, 1000, 4e9, 8000.0, gated=True)
    assert e["rows_per_s"] == pytest.approx(5e5)
    assert e["gbs"] == pytest.approx(2000.0) and e["frac"] == pytest.approx(0.25)
    assert e["gated"] and e["traffic"] is None


def test_gated_workloads_are_the_large_vocabulary_ones():
    sys.path.insert(0, ROOT)
    import bench
    import workloads
    assert set(bench.GATED_CE) <= set(workloads.CE_WORKLOADS)
    assert "ce_f32_64x1000" not in bench.GATED_CE
