"""Host logic of bench.py without a GPU: the max-over-ranks timing of the
replicas (two gloo ranks on CPU), the whole-job value, the algorithmic bytes,
and the reference arm's JSON line on a small workload."""
import json
import os
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402
from speculative_decoding_draft_tcgen05_gb300 import workloads as wl  # noqa: E402


def _rank_main(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    local_ms = [120.0, 135.5][rank]  # rank 1 is the slow replica
    m = bench.max_over_ranks(local_ms, world)
    q.put((rank, m, bench.whole_job_value(1, world, 1000, m)))
    dist.destroy_process_group()


def test_replicas_take_the_slowest_rank():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = 29500 + os.getpid() % 1000
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [m for _, m, _ in out] == [135.5, 135.5]
    # 2 replicas x 1 block x 1000 steps in 135.5 ms
    assert out[0][2] == pytest.approx(2 * 1000 / 0.1355)


def test_single_rank_needs_no_process_group():
    assert bench.max_over_ranks(3.5, 1) == 3.5
    assert bench.whole_job_value(8, 1, 100, 50.0) == pytest.approx(8 * 100 / 0.05)


def test_algorithmic_bytes_of_the_headline_workload():
    w = wl.WORKLOADS["4b_b1"]
    k1, step = bench.algorithmic_bytes(w, G=152, N=7)
    assert k1 == 151936 * 2560 * 2 + 256 * 2560 * 2 + 7 * 2560 * 2 + 152 * 7 * 16 * 8 + 7 * 256 * 4
    assert step > k1 and step - k1 < 5e6


def test_reference_arm_prints_one_line():
    env = dict(os.environ, OMP_NUM_THREADS="2")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload", "tiny",
                        "--steps", "3", "--warmup", "1"], capture_output=True, text=True, env=env, timeout=300)
    assert r.returncode == 0, r.stderr
    lines = [ln for ln in r.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    j = json.loads(lines[0])
    assert j["impl"] == "reference" and j["value"] > 0 and j["unit"] == "blocks/s"
    assert j["cpu_baseline"]["kind"] == "oracle" and j["e2e"]["h2d_bytes_per_step"] == 0


def test_reference_arm_other_ranks_exit_quietly():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload", "tiny",
                        "--steps", "1", "--warmup", "1"], capture_output=True, text=True, env=env, timeout=120)
    assert r.returncode == 0 and r.stdout.strip() == ""
