"""The bench's multi-rank path on CPU (gloo, world size 2): the job time is
the maximum over ranks, the whole-job value counts every rank's calls, and
the reference arm under torchrun prints one line from rank 0 only."""

import json
import os
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _worker(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = bench.max_over_ranks(10.0 + 5.0 * rank, world)
        q.put((rank, ms, bench.whole_job_gbs(1000, 100, world, ms)))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_whole_job_value():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = 29500 + os.getpid() % 1000
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(2))
    for rank, ms, gbs in got:
        assert ms == 15.0                                       # the slower rank's time
        assert abs(gbs - 2 * 100 * 1000 / 15e-3 / 1e9) < 1e-12  # both ranks' bytes


def test_single_rank_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.25, 1) == 3.25
    assert bench.whole_job_gbs(2000, 10, 1, 1.0) == 2000 * 10 / 1e-3 / 1e9


def test_reference_arm_under_torchrun_prints_once():
    port = 30500 + os.getpid() % 1000
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr", "127.0.0.1", "--master-port", str(port),
           os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2", "--steps", "3", "--warmup", "3"]
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["e2e"]["h2d_bytes_per_step"] == 0


def test_mxfp4_bytes_and_summary():
    """The mxfp4 side measurement: algorithmic bytes (4-bit codes, one scale byte
    per 32, bf16 x and y) and the fields and fractions of its JSON object."""
    sys.path.insert(0, ROOT)
    import bench
    N, K = 15360, 3840
    assert bench.mx_algorithmic_bytes(N, K, 1) == N * K // 2 + N * K // 32 + 2 * (K + N) == 31372800
    assert bench.mx_algorithmic_bytes(N, K, 13) == 31372800 + 12 * 2 * (K + N)
    mx = dict(N=N, K=K, R=10, set_bytes=31334400, steps=1000, ms1=12.0, ms13=84.0,
              clocks13={"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": [], "samples": 9})
    out = bench.mx_summary(mx, 6773.5, 80.5)
    assert out["workload"] == bench.MX_WORKLOAD and out["N"] == N and out["K"] == K
    m1, m13 = out["m1"], out["m13"]
    assert m1["us_per_call"] == 12.0 and m13["us_per_call"] == 84.0
    assert abs(m1["achieved_gbs"] - 31372800 / 12e-6 / 1e9) < 0.01
    assert abs(m1["hbm_frac"] - m1["achieved_gbs"] / 6773.5) < 1e-4
    assert abs(m13["fp32_tflops"] - 2.0 * N * K * 13 / 84e-6 / 1e12) < 0.01
    assert abs(m13["fp32_frac"] - m13["fp32_tflops"] / 80.5) < 1e-3
    assert m13["ratio_to_m1"] == 7.0 and m13["clocks"]["reasons"] == []
    assert "cpu_oracle" not in out
    t, runs = bench.mx_oracle_timing(K, rows=8, seconds=0.05)
    assert t > 0 and runs >= 1
    cpu = bench.mx_summary(mx, 6773.5, 80.5, cpu=(8, t, runs))["cpu_oracle"]
    assert cpu["kind"] == "oracle" and cpu["cores"] == 1
    assert abs(cpu["value"] - bench.mx_algorithmic_bytes(8, K, 1) / t / 1e9) < 1e-4
