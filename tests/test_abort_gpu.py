"""Cancellation of running searches on the GPU: the request is seen between kernel launches
(never polled inside a kernel), the call returns QUBO_ERR_ABORTED, the device stays usable, and a
checkpointed run keeps its progress."""
import threading
import time

import numpy as np
import pytest

import oracle
import qubo_instances as qi

pytestmark = pytest.mark.gpu


@pytest.fixture
def q():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import exact_qubo_exhaustive_gb300 as lib
    lib.clear_abort()
    yield lib
    lib.clear_abort()


def run_in_thread(fn):
    out = {}

    def body():
        t0 = time.perf_counter()
        try:
            out["value"] = fn()
        except Exception as exc:  # the QuboError is the expected outcome
            out["error"] = exc
        out["seconds"] = time.perf_counter() - t0

    th = threading.Thread(target=body)
    th.start()
    return th, out


def test_abort_a_long_search(q):
    Q = qi.random_upper_int(44, -1000, 1000, 40)  # 2^44 states: about a second uninterrupted
    th, out = run_in_thread(lambda: q.solve(Q))
    time.sleep(0.25)
    q.request_abort()
    th.join(timeout=30)
    assert not th.is_alive()
    assert isinstance(out.get("error"), q.QuboError) and out["error"].status == -7
    q.clear_abort()
    small = qi.random_upper_int(16, -50, 50, 41)
    e, x, t = q.solve(small)  # the device is still usable
    want = oracle.get().solve(small)
    assert (e, t) == (want[0], want[2]) and (x == want[1]).all()


def test_abort_keeps_checkpointed_progress(q, tmp_path):
    Q = qi.random_upper_int(42, -1000, 1000, 42)
    path = str(tmp_path / "run.ckpt")
    th, out = run_in_thread(lambda: q.solve_checkpointed(Q, 7, path, slices_per_chunk=2))
    # abort as soon as a chunk is on disk (no fixed sleep: a slow start cannot make it early)
    deadline = time.perf_counter() + 30
    while time.perf_counter() < deadline and th.is_alive():
        try:
            if q.checkpoint_read(path)["next_slice"] > 0:
                break
        except q.QuboError:
            pass  # no chunk written yet
        time.sleep(0.002)
    q.request_abort()
    th.join(timeout=30)
    assert isinstance(out.get("error"), q.QuboError) and out["error"].status == -7
    q.clear_abort()
    done_before = q.checkpoint_read(path)["next_slice"]
    assert 0 < done_before < 128
    complete, e, x, t, n_done = q.solve_checkpointed(Q, 7, path, slices_per_chunk=2)
    assert complete and n_done == 128
    whole = q.solve(Q)
    assert (e, t) == (whole[0], whole[2]) and (x == whole[1]).all()
