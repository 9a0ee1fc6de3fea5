"""Multi-process host logic of the sharded search (CPU, gloo, world sizes 2 and 3).

Each rank searches its contiguous share of the 2^k_prefix slices and one all-gather combines the
shard records. Here the per-rank search is the CPU oracle's slice solver, so the exchange and
the reduction are checked without a GPU; the whole-problem oracle solve is the expected value.
"""
import json
import os
import socket

import numpy as np
import pytest

import oracle
import qubo_instances as qi

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

from exact_qubo_exhaustive_gb300 import distributed as qd  # noqa: E402


def free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def oracle_range(Q, k, first, count):
    """Oracle result over slices [first, first + count): per-slice solves, reduced here."""
    O = oracle.get()
    recs = []
    for p in range(first, first + count):
        e, x, t = O.solve_slice(Q, k, p)
        recs.append((e, oracle.rank_of_bits(x), t))
    e, r, t = qd.combine(recs)
    return e, oracle.bits_of_rank(Q.shape[0], r), t


def _worker(rank, world, port, case_file, out_dir):
    os.environ["GLOO_SOCKET_IFNAME"] = "lo"
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        case = np.load(case_file)
        Q, k = case["Q"], int(case["k"])
        seen = []

        def solver(Qm, kk, first, count):
            seen.append((first, count))
            return oracle_range(Qm, kk, first, count)

        e, x, t = qd.solve_distributed(Q, k, solver=solver)
        with open(os.path.join(out_dir, f"r{rank}.json"), "w") as f:
            json.dump({"e": float(e), "x": [int(b) for b in x], "t": int(t), "seen": seen}, f)
    finally:
        dist.destroy_process_group()


def run_ranks(tmp_path, Q, k, world):
    case_file = str(tmp_path / "case.npz")
    np.savez(case_file, Q=Q, k=k)
    mp.start_processes(_worker, args=(world, free_port(), case_file, str(tmp_path)), nprocs=world,
                       start_method="spawn", join=True)
    return [json.load(open(tmp_path / f"r{r}.json")) for r in range(world)]


def check_against_oracle(outs, Q, k, world):
    want_e, want_x, want_t = oracle.get().solve(Q)
    for r, o in enumerate(outs):
        assert o["e"] == float(want_e)
        assert o["x"] == [int(b) for b in want_x]
        assert o["t"] == int(want_t)
        first, count = qd.shard_range(1 << k, r, world)
        assert o["seen"] == ([[first, count]] if count else [])


def test_shard_range_partitions_contiguously():
    for total in (0, 1, 2, 7, 8, 1 << 14):
        for world in (1, 2, 3, 5, 8):
            spans = [qd.shard_range(total, r, world) for r in range(world)]
            pos = 0
            for first, count in spans:
                assert first == pos and count >= 0
                pos += count
            assert pos == total
            counts = [c for _, c in spans]
            assert max(counts) - min(counts) <= 1
    with pytest.raises(ValueError):
        qd.shard_range(8, 2, 2)


def test_combine_rule():
    # lowest energy wins; among equal energies the lowest rank wins and ties add; empty shards skip
    assert qd.combine([(-3, 9, 1), None, (-5, 7, 2), (-5, 4, 3)]) == (-5, 4, 5)
    assert qd.combine([(0, 0, 4)]) == (0, 0, 4)
    with pytest.raises(ValueError):
        qd.combine([None, None])


def test_two_ranks_random_int(tmp_path):
    Q = qi.random_upper_int(14, -100, 100, 611)
    check_against_oracle(run_ranks(tmp_path, Q, 4, 2), Q, 4, 2)


def test_three_ranks_uneven_shards_and_all_ties(tmp_path):
    # Q = 0: every one of the 2^12 states ties; 8 slices split 3 / 3 / 2
    Q = np.zeros((12, 12), np.int32)
    outs = run_ranks(tmp_path, Q, 3, 3)
    check_against_oracle(outs, Q, 3, 3)
    assert outs[0]["t"] == 1 << 12 and outs[0]["x"] == [0] * 12


def test_rank_without_slices(tmp_path):
    # 2 slices over 3 ranks: the last rank searches nothing and still receives the result
    Q = qi.mattis_planted(12, 612)[0]
    check_against_oracle(run_ranks(tmp_path, Q, 1, 3), Q, 1, 3)


def test_two_ranks_fp32(tmp_path):
    Q = qi.random_symmetric_normal_f32(12, 613)
    check_against_oracle(run_ranks(tmp_path, Q, 3, 2), Q, 3, 2)


def test_two_ranks_fp64(tmp_path):
    # fp64 input: the combined energy keeps its fraction (integer input alone is returned as int)
    Q = qi.random_symmetric_normal_f32(12, 614).astype(np.float64) * 0.37
    outs = run_ranks(tmp_path, Q, 3, 2)
    check_against_oracle(outs, Q, 3, 2)
    assert outs[0]["e"] != int(outs[0]["e"])


def test_fp64_tie_across_shards(tmp_path):
    # x_0 is free (Q_00 = 0, no coupling), so the two minimisers differ only in x_0 and lie in
    # different shards of the k_prefix = 1 split; E_min = -2.25 is not an integer
    Q = np.diag([0.0] + [-0.25] * 9)
    outs = run_ranks(tmp_path, Q, 1, 2)
    check_against_oracle(outs, Q, 1, 2)
    assert outs[0]["e"] == -2.25 and outs[0]["t"] == 2 and outs[0]["x"] == [0] + [1] * 9


def _bench_worker(rank, world, port, out_dir):
    os.environ["GLOO_SOCKET_IFNAME"] = "lo"
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        import bench
        got = bench.max_over_ranks([10.0 + rank, 5.0 - rank, 7.5 * (rank + 1)], "cpu")
        with open(os.path.join(out_dir, f"b{rank}.json"), "w") as f:
            json.dump(got, f)
    finally:
        dist.destroy_process_group()


def test_bench_takes_the_slowest_rank(tmp_path):
    # bench.py reports the whole job's step time as the maximum over ranks
    mp.start_processes(_bench_worker, args=(2, free_port(), str(tmp_path)), nprocs=2, start_method="spawn",
                       join=True)
    for r in range(2):
        assert json.load(open(tmp_path / f"b{r}.json")) == [11.0, 5.0, 15.0]
