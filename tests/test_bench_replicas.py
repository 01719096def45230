"""The multi-process side of bench.py on CPU: with N > 1 every rank runs a
replica of the single-GPU step, the step time is the max over ranks, and
the whole-job throughput counts every rank's tokens.  Checked with two gloo
ranks; the reference arm's non-zero ranks exit without output."""
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


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        local = [1.25, 3.5][rank]  # the second replica is slower
        t = bench.replica_time(local, world, "cpu")
        out[rank] = (t, bench.replica_throughput(world, 32768, t))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_replica():
    world = 2
    with mp.Manager() as m:
        out = m.dict()
        mp.start_processes(_worker, args=(world, _free_port(), out), nprocs=world, join=True,
                           start_method="spawn")
        res = dict(out)
    assert res[0][0] == pytest.approx(3.5) and res[1][0] == pytest.approx(3.5)
    assert res[0][1] == pytest.approx(2 * 32768 / 3.5e-3)


def test_single_process_is_a_no_op():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.replica_time(2.0, 1, "cpu") == 2.0
    assert bench.replica_throughput(1, 1000, 1.0) == pytest.approx(1e6)


def test_reference_arm_other_ranks_exit_quietly():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "3", "--workload", "tiny"],
                       env=env, capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == ""


@pytest.mark.parametrize("workload", ["tiny", "ssd32k"])
def test_reference_arm_prints_one_contract_line(workload):
    """Rank 0 of the reference arm (the fp64 oracle on host cores) prints one
    JSON line with the contract's keys and its own e2e and cpu_baseline."""
    env = dict(os.environ, RANK="0", WORLD_SIZE="1", LOCAL_RANK="0")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "3", "--workload", workload],
                       env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr
    lines = [ln for ln in r.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config", "e2e",
                "cpu_baseline", "gpu_launches"):
        assert key in d, key
    assert d["impl"] == "reference" and d["value"] > 0 and d["config"]["workload"] == workload
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"]["value"] == d["value"] and d["e2e"]["h2d_bytes_per_step"] == 0
