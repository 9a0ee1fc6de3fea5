"""The bench's multi-GPU path (one n=40 search sharded by contiguous slice ranges, one all-gather
of the per-rank records over NCCL) run as a one-rank torchrun group on the CUDA path: the same
code the N-GPU bench runs, with its answer checked against the stored full oracle search."""
import json
import os
import socket
import subprocess
import sys

import pytest

from conftest import ROOT, read_golden

pytestmark = pytest.mark.gpu


def test_sharded_bench_path_in_a_one_rank_group():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "1",
           "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.join(ROOT, "bench.py"),
           "--sharded", "--steps", "2", "--warmup", "3"]
    env = dict(os.environ, NCCL_NVLS_ENABLE="0")
    out = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [ln for ln in out.stdout.splitlines() if ln.startswith("{")]
    line = json.loads(lines[-1])
    assert line["n_gpus"] == 1 and line["config"]["slices_per_rank"] == 1 << line["config"]["shard_k_prefix"]
    assert line["result"]["checks"]["sharded_step"] == "matches the full oracle search"
    (row,) = read_golden("full_oracle_n40_int32.txt")
    assert line["result"]["min_energy"] == float(row[0]) and line["result"]["tie_count"] == int(row[2])
    assert line["value"] > 0 and line["e2e"]["value"] > 0 and line["gpu_launches"] > 0
