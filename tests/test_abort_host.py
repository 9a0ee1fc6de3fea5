"""Cancellation on the host (qubo_request_abort): a pending request refuses new calls before any
device work, and clearing it re-arms them (CPU; no GPU is touched)."""
import numpy as np
import pytest

import qubo_instances as qi


@pytest.fixture
def q():
    import exact_qubo_exhaustive_gb300 as lib
    lib.clear_abort()
    yield lib
    lib.clear_abort()


def test_pending_abort_refuses_calls(q, tmp_path):
    Q = qi.random_upper_int(12, -9, 9, 1)
    q.request_abort()
    for call in (lambda: q.solve(Q), lambda: q.solve_slices(Q, 2, [0, 1]), lambda: q.solve_lowest(Q, 3),
                 lambda: q.solve_batched(np.stack([Q, Q])), lambda: q.solve_checkpointed(Q, 2, str(tmp_path / "a")),
                 # the abort check comes before any use of these (never dereferenced) device pointers
                 lambda: q.solve_device_no_alloc(12, 256, q.INT32, None, 512),
                 lambda: q.solve_device(12, 256, q.INT32, 1024, 1 << 20, None, 512)):
        with pytest.raises(q.QuboError) as ei:
            call()
        assert ei.value.status == -7
    assert not (tmp_path / "a").exists()  # nothing was written


def test_clear_rearms(q):
    Q = qi.random_upper_int(12, -9, 9, 2)
    q.request_abort()
    q.clear_abort()
    torch = pytest.importorskip("torch")
    if torch.cuda.is_available():
        q.solve(Q)  # runs normally
    else:
        with pytest.raises(q.QuboError) as ei:
            q.solve(Q)
        assert ei.value.status == -6  # got past the abort check, stopped at the device check
