"""The allocation-free entry point against the ordinary device entry point.

qubo_solve_device_no_alloc() exists for callers that cannot call cudaMalloc when they need a
result (a latency-critical loop, or a plug-in whose host framework owns all device memory). It
must give exactly the results of qubo_solve_device(), call after call, although every call reuses
the same fixed scratch array. This file is named to be collected last.
"""
import numpy as np
import pytest

import qubo_instances as qi

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def env():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import exact_qubo_exhaustive_gb300 as q
    return q, torch


def record(q, t):
    return np.frombuffer(t.cpu().numpy().tobytes(), dtype=q.RESULT_DTYPE)[0]


def with_workspace(q, torch, n, Q, dtype):
    dq = torch.from_numpy(Q).cuda()
    nb = q.workspace_bytes(n, dtype)
    ws = torch.empty(nb, dtype=torch.uint8, device="cuda")
    res = torch.zeros(32, dtype=torch.uint8, device="cuda")
    q.solve_device(n, dq, dtype, ws, nb, torch.cuda.current_stream().cuda_stream, res)
    torch.cuda.synchronize()
    return record(q, res)


def no_alloc(q, torch, n, Q, dtype):
    dq = torch.from_numpy(Q).cuda()
    res = torch.zeros(32, dtype=torch.uint8, device="cuda")
    q.solve_device_no_alloc(n, dq, dtype, torch.cuda.current_stream().cuda_stream, res)
    torch.cuda.synchronize()
    return record(q, res)


def test_two_calls_in_a_row_match_the_workspace_entry_point(env):
    q, torch = env
    cases = [(32, qi.random_upper_int(32, -1000, 1000, 71), q.INT32),
             (24, qi.random_upper_int(24, -1, 1, 72), q.INT32),   # many ties: exercises the resolve pass
             (26, qi.random_symmetric_normal_f32(26, 73), q.FP32)]
    for n, Q, dt in cases:
        want = with_workspace(q, torch, n, Q, dt)
        assert want["status"] == 0
        for _ in range(2):  # the second call sees the first call's leftovers in the array
            got = no_alloc(q, torch, n, Q, dt)
            assert got["status"] == 0
            assert got["min_energy"] == want["min_energy"]  # exact for int32, bit-identical fp64 for fp32
            assert got["argmin_rank"] == want["argmin_rank"]
            assert got["tie_count"] == want["tie_count"]


def test_interleaved_problems_of_every_minimum_pass(env):
    # every minimum pass works in the shared array: the block-bounded biased pass (narrow and
    # wide-but-below-2^22 int32 input, fp32 input's fixed-point image; its block table and group
    # words live in the array too), the int32 pass on int32 input beyond 2^22 (n >= 30) and on a
    # small problem; two rounds, so every call follows another problem's leftovers
    q, torch = env
    cases = [(32, qi.random_upper_int(32, -3, 3, 81), q.INT32),
             (31, qi.random_symmetric_normal_f32(31, 82), q.FP32),
             (33, qi.random_upper_int(33, -1000, 1000, 83), q.INT32),
             (20, qi.random_upper_int(20, -1, 1, 84), q.INT32),
             (30, qi.random_upper_int(30, -(1 << 17), 1 << 17, 85), q.INT32)]
    plans = [q.plan(n, dt) for n, _, dt in cases]
    assert plans[0]["pruned"] == 1 and plans[1]["pruned"] == 1 and plans[2]["pruned"] == 1
    assert int(np.abs(cases[4][1].astype(np.int64)).sum()) > (1 << 22)  # the int32 pass owns it
    wants = [with_workspace(q, torch, n, Q, dt) for n, Q, dt in cases]
    for _ in range(2):
        for (n, Q, dt), want in zip(cases, wants):
            got = no_alloc(q, torch, n, Q, dt)
            assert got["status"] == 0 and want["status"] == 0
            assert (got["min_energy"], got["argmin_rank"], got["tie_count"]) == \
                (want["min_energy"], want["argmin_rank"], want["tie_count"]), n


def test_largest_problem_that_fits_the_array(env):
    # the largest n whose default-plan workspace fits the array is accepted and exact
    q, torch = env
    n = max(m for m in range(20, 63) if q.workspace_bytes(m) <= q.NO_ALLOC_SCRATCH_BYTES)
    assert q.workspace_bytes(n + 1) > q.NO_ALLOC_SCRATCH_BYTES
    Q = qi.random_upper_int(n, -1000, 1000, 86)
    want = with_workspace(q, torch, n, Q, q.INT32)
    for _ in range(2):
        got = no_alloc(q, torch, n, Q, q.INT32)
        assert got["status"] == 0
        assert (got["min_energy"], got["argmin_rank"], got["tie_count"]) == \
            (want["min_energy"], want["argmin_rank"], want["tie_count"])


def test_problems_beyond_the_array_are_rejected(env):
    q, torch = env
    n = 52
    assert q.workspace_bytes(n) > q.NO_ALLOC_SCRATCH_BYTES
    dq = torch.zeros((n, n), dtype=torch.int32, device="cuda")
    res = torch.zeros(32, dtype=torch.uint8, device="cuda")
    with pytest.raises(q.QuboError) as ei:
        q.solve_device_no_alloc(n, dq, q.INT32, torch.cuda.current_stream().cuda_stream, res)
    assert ei.value.status == -1
