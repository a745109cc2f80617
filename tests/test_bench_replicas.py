"""The benchmark's multi-rank logic on CPU: world_size-2 gloo ranks run the
max-over-ranks time reduction and the whole-job rate, and the reference arm
runs on rank 0 only.  No GPU is used."""
import os
import subprocess
import sys

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        t = bench.reduce_max(10.0 + 5.0 * rank, dist)  # rank 1 is the slower one
        rate = bench.whole_job_rate(100.0, 4, world, t)
        q.put((rank, t, rate))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_whole_job_rate():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = 29500 + os.getpid() % 1000
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, t, rate in res:
        assert t == 15.0  # every rank sees the slowest rank's time
        assert rate == pytest.approx(100.0 * 4 * 2 / 0.015)


def test_reduce_max_single_process_is_identity():
    assert bench.reduce_max(3.5, None) == 3.5
    assert bench.whole_job_rate(1e9, 10, 1, 1000.0) == pytest.approx(1e10)


def test_reference_arm_other_ranks_exit_quietly():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "0"], capture_output=True, text=True, env=env, timeout=300)
    assert r.returncode == 0
    assert r.stdout.strip() == ""


@pytest.mark.parametrize("op", ["fwd", "bwd_data"])
def test_reference_arm_json_line(op):
    """Rank 0 of the reference arm prints one JSON line with the contract's keys,
    for the forward pass and for backward data (the oracle on the host cores)."""
    import json

    env = dict(os.environ, RANK="0", WORLD_SIZE="1", LOCAL_RANK="0")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--op", op,
                        "--workload", "grouped2d_f32_smoke", "--steps", "2", "--warmup", "1"],
                       capture_output=True, text=True, env=env, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["config"]["op"] == op
    assert ("bwd_data" in d["metric"]) == (op == "bwd_data")
    for k in ("value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "cpu_baseline",
              "e2e"):
        assert k in d, k
    assert d["value"] > 0 and d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0
