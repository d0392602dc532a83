"""Host-side logic of bench.py, on the CPU: the multi-rank reduction of the
replicas path (two gloo ranks), the whole-job throughput, and the reference
arm's JSON line."""
import json
import os
import subprocess
import sys

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        got = bench.max_over_ranks([1.0 + rank, 10.0 - rank, 5.0])
        env = bench.dist_env()
        out.put((rank, got, env))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_with_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = 29500 + (os.getpid() % 1000)
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, got, env in res:
        assert got == [2.0, 10.0, 5.0]
        assert env == (2, rank, rank)


def test_max_over_ranks_without_a_group_is_identity():
    assert bench.max_over_ranks([3, 1.5]) == [3.0, 1.5]


def test_replica_throughput_counts_every_rank():
    assert bench.replica_throughput(10.0, 4, 2.0) == 20.0


def test_flop_count_convention():
    assert bench.fwd_flops(1, 128, 1024, 128, False) == 4.0 * 128 * 1024 * 1024 * 128
    assert bench.fwd_flops(1, 128, 1024, 128, True) == 2.0 * 128 * 1024 * 1024 * 128


def test_reference_arm_prints_one_contract_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "3", "--ref-seconds", "0.2", "--n", "2048"],
                       capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    j = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "config", "cpu_baseline", "e2e"):
        assert key in j, key
    assert j["impl"] == "reference" and j["unit"] == "TFLOP/s" and j["value"] > 0
    assert j["e2e"]["h2d_bytes_per_step"] == 0 and j["cpu_baseline"]["kind"] == "oracle"


def test_reference_arm_is_silent_on_other_ranks():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--ref-seconds", "0.2", "--n", "1024"],
                       capture_output=True, text=True, timeout=300, cwd=ROOT, env=env)
    assert r.returncode == 0 and r.stdout.strip() == ""


def test_timeline_summary_on_a_hand_made_timeline():
    """Three chunks (copy-in done, kernel reached, kernel done, copy-out done,
    ms from the call's start): kernels [1, 4], [3.5, 6] and [7, 9] -> busy
    5 (the first two overlap) + 2 = 7 ms of a 10 ms call, one 1 ms gap,
    chunk 2's copy-in ending 0.5 ms after chunk 1's kernel; with 4 ms of
    copies alone, the call hid (7 + 4 - 10) / 4 of them."""
    import bench
    tl = [(1.0, 1.0, 4.0, 4.5), (2.0, 3.5, 6.0, 6.5), (6.5, 7.0, 9.0, 10.0)]
    s = bench.timeline_summary(tl, 4.0)
    assert s["chunks"] == 3 and s["wall_ms"] == 10.0
    assert s["kernel_busy_ms"] == 7.0 and s["idle_ms"] == 3.0
    assert s["kernel_ms_sum"] == 3.0 + 2.5 + 2.0
    assert s["first_kernel_ms"] == 1.0 and s["after_last_kernel_ms"] == 1.0
    assert s["max_gap_ms"] == 1.0
    assert s["copy_in_late_ms"] == 0.5  # chunk 2 (6.5) after chunk 1's kernel (6.0); chunk 1 was early
    assert s["overlap_frac"] == 0.25
