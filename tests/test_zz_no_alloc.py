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


def test_problems_beyond_the_array_are_rejected(env):
    q, torch = env
    n = 52
    assert q.workspace_bytes(n) > q.NO_ALLOC_SCRATCH_BYTES
    dq = torch.zeros((n, n), dtype=torch.int32, device="cuda")
    res = torch.zeros(32, dtype=torch.uint8, device="cuda")
    with pytest.raises(q.QuboError) as ei:
        q.solve_device_no_alloc(n, dq, q.INT32, torch.cuda.current_stream().cuda_stream, res)
    assert ei.value.status == -1
