"""The N > 1 path of bench.py on CPU: two gloo ranks (replicas). Each rank
times its own replica; the job's time is the maximum over ranks and its value
the FLOPs of all ranks over that time. Only rank 0 runs the reference arm."""
import json
import os
import subprocess
import sys

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _rank(rank, world, port, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        local_ms = [3.0, 5.0][rank]
        total = bench.max_over_ranks(local_ms, "cpu")
        dist.barrier()
        out[rank] = (total, bench.whole_job_tflops(world, 2e12, total))
    finally:
        dist.destroy_process_group()


def _free_port():
    import socket
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_two_gloo_ranks_take_the_slowest_time():
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        out = m.dict()
        mp.start_processes(_rank, args=(2, _free_port(), out), nprocs=2, join=True,
                           start_method="spawn")
        res = dict(out)
    assert res[0] == res[1]
    total, value = res[0]
    assert total == 5.0
    # two replicas of 2 TFLOP each in 5 ms
    assert value == pytest.approx(2 * 2e12 / 5e-3 / 1e12)


def test_single_process_is_its_own_maximum():
    assert bench.max_over_ranks(7.5, "cpu") == 7.5
    assert bench.whole_job_tflops(1, 1e12, 1.0) == pytest.approx(1000.0)


def test_reference_arm_runs_on_rank_zero_only():
    """Under torchrun the ranks other than 0 exit at once without output."""
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--workload", "tiny_ring", "--steps", "1", "--warmup", "1"],
                       env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == ""


def test_reference_arm_prints_the_contract_line():
    """Rank 0 of the reference arm (the oracle on the host cores) prints one
    JSON line with the contract's keys: impl, metric and unit, the step
    counts, a cpu_baseline describing the run and an e2e with no host-device
    bytes."""
    env = {k: v for k, v in os.environ.items() if k not in ("RANK", "WORLD_SIZE", "LOCAL_RANK")}
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--workload", "tiny_ring", "--steps", "1", "--warmup", "1"],
                       env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr
    lines = [x for x in r.stdout.strip().splitlines() if x.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["value"] > 0 and d["steps"] == 1 and d["warmup"] == 1
    for key in ("metric", "unit", "n_gpus", "ms_per_step", "higher_is_better", "dtype", "config"):
        assert key in d, key
    assert d["config"]["workload"] == "tiny_ring"
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["sample"] and cb["value"] == d["value"]
    e2e = d["e2e"]
    assert e2e["value"] == d["value"] and e2e["unit"] == d["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0
