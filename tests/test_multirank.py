"""The multi-rank path of bench.py (replicas, weak scaling) on CPU with the
gloo backend and two processes: every rank gets the maximum of the per-rank
timings, the job value counts all ranks' work in the slowest rank's time, and
the reference arm prints on rank 0 only."""
import json
import os
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def _worker(rank, world, port, out):
    import torch
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    torch.distributed.init_process_group("gloo", rank=rank, world_size=world)
    try:
        local = [10.0 + rank, 7.0 - rank, 1.5 * (rank + 1)]
        got = bench.max_over_ranks(local)
        out.put((rank, got))
    finally:
        torch.distributed.destroy_process_group()


def test_max_over_ranks_gloo_two_processes():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = 29500 + os.getpid() % 1000
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = dict(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert res[0] == res[1] == [11.0, 7.0, 3.0]


def test_job_value_weak_scaling():
    import bench
    one = bench.job_value(1, 16.5e12, 5.5)
    assert abs(one - 3000.0) < 1e-9
    assert abs(bench.job_value(4, 16.5e12, 5.5) - 4 * one) < 1e-9


def test_flop_convention_reproduces_the_pages_table():
    # 2*M*N*K / t reproduces the torch TFLOP/s column of the routing PR's kernel
    # table, e.g. 8320 x 5376 x 21504 in 1351.1 us -> 1424 TFLOP/s
    import bench
    for (M, K, N), us, printed in zip(bench.SHAPES, bench.H100_TORCH_US, [1424, 1431, 1351, 1361, 1520]):
        assert round(bench.flops(M, K, N) / (us * 1e-6) / 1e12) == printed


def test_reference_arm_nonzero_rank_prints_nothing():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "3"], env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0 and r.stdout.strip() == ""


def test_reference_arm_prints_the_contract_line():
    # the reference arm (the CPU oracle on a bounded sample) runs without a GPU and
    # prints one JSON line with the native arm's metric and the reference keys
    import json
    import os
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    r = subprocess.run([sys.executable, os.path.join(root, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "3", "--ref-rows", "2"], capture_output=True, text=True, timeout=600,
                       cwd=root, env=dict(os.environ, RANK="0", WORLD_SIZE="1"))
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "TFLOP/s" and d["value"] > 0
    assert d["higher_is_better"] is True and d["steps"] == 1 and d["warmup"] == 3
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0
    assert "metric" in d and "config" in d
