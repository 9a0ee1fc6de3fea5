"""bench.py's command-line contract on the CPU: the reference arm (the CPU oracle on a bounded
sample of the n=40 workload) prints one JSON line with the keys the driver reads."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_prints_one_json_line():
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                          "--warmup", "3"], capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [ln for ln in out.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference"
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e", "gpu_launches"):
        assert key in d, key
    assert d["value"] > 0 and d["steps"] == 1 and d["warmup"] == 3 and d["higher_is_better"] is True
    assert d["config"]["workload"].startswith("n=40 dense QUBO")
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["cpu_baseline"]["kind"] == "oracle"


def test_max_over_ranks_single_process_group():
    # the step-time reduction with a one-rank gloo group returns its input
    import socket
    torch = __import__("pytest").importorskip("torch")
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=0, world_size=1)
    try:
        assert bench.max_over_ranks([1.5, 2.0], "cpu") == [1.5, 2.0]
    finally:
        dist.destroy_process_group()


def test_self_check_against_the_stored_full_search():
    # the timed answer is compared with tests/golden/full_oracle_n40_int32.txt; a wrong energy,
    # rank or tie count raises, so bench.py exits non-zero instead of printing a rate
    import pytest
    sys.path.insert(0, ROOT)
    import bench
    e, r, t = bench.golden("n40_int32")
    assert bench.check_result("n40_int32", e, r, t)
    for bad in ((e + 1, r, t), (e, r + 1, t), (e, r, t + 1)):
        with pytest.raises(bench.ResultMismatch):
            bench.check_result("n40_int32", *bad)
    e36, r36, t36 = bench.golden("n36_fp32")
    assert bench.check_result("n36_fp32", e36 + 1e-9, r36, t36, tol=1e-6)
    with pytest.raises(bench.ResultMismatch):
        bench.check_result("n36_fp32", e36 + 1e-3, r36, t36, tol=1e-6)


def test_sharded_step_records_combine():
    # the all-gathered result records of the multi-GPU step: lowest energy wins, equal energies
    # keep the lowest rank and add their ties, a failed shard raises
    import numpy as np
    import pytest
    sys.path.insert(0, ROOT)
    import bench
    dt = np.dtype([("status", np.int32), ("reserved", np.int32), ("min_energy", np.float64),
                   ("argmin_rank", np.uint64), ("tie_count", np.uint64)])
    recs = np.zeros(3, dt)
    recs["min_energy"] = [-7.0, -9.0, -9.0]
    recs["argmin_rank"] = [5, 40, 12]
    recs["tie_count"] = [1, 2, 3]
    assert bench.combine_gathered(recs.tobytes(), 3, dt) == (-9.0, 12, 5)
    recs["status"][1] = -2
    with pytest.raises(RuntimeError):
        bench.combine_gathered(recs.tobytes(), 3, dt)
