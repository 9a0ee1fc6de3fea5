"""The batched workload itself (4096 independent n=24 int32 instances, entries uniform in
[-50, 50], instance i from seed + i) through the device entry point, against the CPU oracle.

Terastate-per-second QUBO Brute-Force on a Single GPU, §III-C1: independent subproblems, here
one problem per instance. The whole batch runs in one call at the workload's full size (the
persistent-grid work split, the workspace and the per-instance strides at batch = 4096); a seeded
sample of 256 instances is compared bit-exactly with the oracle's exhaustive search, and every
instance's returned state is re-evaluated by the oracle.
"""
import numpy as np
import pytest

import oracle
import qubo_instances as qi

pytestmark = pytest.mark.gpu

O = oracle.get()
BATCH, N = 4096, 24


@pytest.fixture(scope="module")
def batched_result():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import exact_qubo_exhaustive_gb300 as q
    Qs = qi.workload_batched()
    assert Qs.shape == (BATCH, N, N)
    dq = torch.from_numpy(np.ascontiguousarray(Qs)).cuda()
    nb = max(q.batched_workspace_bytes(BATCH, N), 256)
    ws = torch.empty(nb, dtype=torch.uint8, device="cuda")
    res = torch.zeros(BATCH * 32, dtype=torch.uint8, device="cuda")
    s = torch.cuda.current_stream()
    q.solve_batched_device(BATCH, N, dq, ws, nb, s.cuda_stream, res)
    torch.cuda.synchronize()
    r = np.frombuffer(res.cpu().numpy().tobytes(), dtype=q.RESULT_DTYPE).copy()
    return Qs, r


def test_every_instance_reports_a_state_with_its_energy(batched_result):
    Qs, r = batched_result
    assert (r["status"] == 0).all()
    assert (r["tie_count"] >= 1).all()
    for b in range(BATCH):
        x = oracle.bits_of_rank(N, int(r["argmin_rank"][b]))
        assert O.energy_i64(O.fold_i32(Qs[b]), x) == int(r["min_energy"][b]), b


def test_sampled_instances_match_the_oracle_exactly(batched_result):
    Qs, r = batched_result
    sample = np.unique(qi.Stream(4096024).integers(0, BATCH - 1, 256))
    sample = np.union1d(sample, [0, BATCH - 1])  # both ends of the batch's strides
    for b in sample:
        e, x, t = O.solve(Qs[b])
        got = (int(r["min_energy"][b]), int(r["argmin_rank"][b]), int(r["tie_count"][b]))
        assert got == (e, oracle.rank_of_bits(x), t), (int(b), got, (e, oracle.rank_of_bits(x), t))


def test_device_entry_matches_the_host_entry(batched_result):
    import exact_qubo_exhaustive_gb300 as q
    Qs, r = batched_result
    e, x, t = q.solve_batched(Qs)
    ranks = np.array([oracle.rank_of_bits(v) for v in x], dtype=np.uint64)
    assert (e == r["min_energy"].astype(np.int64)).all()
    assert (ranks == r["argmin_rank"]).all() and (t == r["tie_count"]).all()


def test_without_block_bounds_the_same_results(batched_result):
    # the packed pass of the batch with block bounds (the default) against the one without
    torch = pytest.importorskip("torch")
    import exact_qubo_exhaustive_gb300 as q
    Qs, r = batched_result
    q.enable_block_bounds(False)
    try:
        e, x, t = q.solve_batched(Qs[:512])
    finally:
        q.enable_block_bounds(True)
    assert (e == r["min_energy"][:512]).all() and (t == r["tie_count"][:512]).all()
    assert [oracle.rank_of_bits(v) for v in x] == [int(v) for v in r["argmin_rank"][:512]]
