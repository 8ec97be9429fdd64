"""The multi-GPU form of the benchmark is replicas only (rows are independent
and nothing is exchanged): each rank runs the whole workload, and the job's
rate is all ranks' rows over the slowest rank's time.  Checked here with two
gloo ranks on the CPU."""
import os
import socket
import subprocess
import sys

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, results):
    sys.path.insert(0, ROOT)
    import bench

    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank,
                            world_size=world)
    try:
        local_ms = [100.0, 250.0][rank]  # rank 1 is the slow one
        value, max_ms, w = bench.replica_throughput(torch, local_ms, rows_per_step=8192, steps=10,
                                                    dist=dist)
        results[rank] = (value, max_ms, w)
    finally:
        dist.destroy_process_group()


def test_replica_throughput_two_gloo_ranks():
    port = _free_port()
    with mp.Manager() as mgr:
        results = mgr.dict()
        mp.spawn(_rank_main, args=(2, port, results), nprocs=2, join=True)
        got = dict(results)
    want = 8192 * 10 * 2 / 0.250
    for rank in (0, 1):
        value, max_ms, w = got[rank]
        assert w == 2
        assert max_ms == 250.0
        assert value == pytest.approx(want)


def test_replica_throughput_single_process():
    sys.path.insert(0, ROOT)
    import bench

    value, max_ms, w = bench.replica_throughput(torch, 200.0, rows_per_step=16, steps=5)
    assert (w, max_ms) == (1, 200.0)
    assert value == pytest.approx(16 * 5 / 0.2)


def test_reference_arm_other_ranks_exit_without_work():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "3"], env=env, capture_output=True, text=True,
                       timeout=120)
    assert r.returncode == 0
    assert r.stdout.strip() == ""


def test_reference_arm_json_line():
    """The reference arm (the oracle on the host cores) prints one JSON line
    with the contract's keys, on the headline workload."""
    import json

    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "3"], capture_output=True, text=True,
                       timeout=600, env=dict(os.environ, RANK="0", WORLD_SIZE="1"))
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference"
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "config", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["unit"] == "rows/s" and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] == 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0


def test_oracle_throughput_on_all_host_cores():
    """The whole-host oracle figure runs the same oracle on several threads,
    each on its own rows, and counts every row it merged."""
    sys.path.insert(0, ROOT)
    import bench
    import workloads

    m = workloads.random_merge(3, 64, 4, 256, mode="bf16")
    v, rows, secs = bench.cpu_oracle_sample_threads(m, 2, budget_s=0.5)
    assert rows > 0 and secs > 0 and abs(v - rows / secs) < 1e-6 * v
