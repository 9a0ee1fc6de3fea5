"""GPU runs of the checkpointed long-run driver: chunked, budget-limited calls resumed from the
file reach exactly the result of one uninterrupted search (and of the oracle)."""
import numpy as np
import pytest

import oracle
import qubo_instances as qi

pytestmark = pytest.mark.gpu

O = oracle.get()


@pytest.fixture(scope="module")
def q():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import exact_qubo_exhaustive_gb300 as lib
    return lib


def oracle_prefix(Q, k, upto):
    """Oracle record over slices [0, upto): lowest energy, lowest rank, summed ties."""
    best = None
    for p in range(upto):
        e, x, t = O.solve_slice(Q, k, p)
        r = oracle.rank_of_bits(x)
        if best is None or e < best[0]:
            best = [e, r, t]
        elif e == best[0]:
            best[1] = min(best[1], r)
            best[2] += t
    return best


def test_one_uninterrupted_call_equals_solve(q, tmp_path):
    Q = qi.random_upper_int(30, -500, 500, 3100)
    done, e, x, t, n_done = q.solve_checkpointed(Q, 6, str(tmp_path / "a.ckpt"))
    want = q.solve(Q)
    assert done and n_done == 64 and (e, t) == (want[0], want[2]) and (x == want[1]).all()
    r = q.checkpoint_read(str(tmp_path / "a.ckpt"))
    assert r["next_slice"] == 64 and r["min_energy"] == want[0]
    # a finished file answers at once
    again = q.solve_checkpointed(Q, 6, str(tmp_path / "a.ckpt"))
    assert again[0] and again[1] == e and again[3] == t


def test_budgeted_calls_resume_chunk_by_chunk(q, tmp_path):
    n, k, chunk = 22, 5, 4
    Q = qi.random_upper_int(n, -40, 40, 3101)  # small range: many ties across slices
    path = str(tmp_path / "b.ckpt")
    calls = 0
    while True:
        done, e, x, t, n_done = q.solve_checkpointed(Q, k, path, slices_per_chunk=chunk, time_budget_s=1e-9)
        calls += 1
        assert n_done == min(calls * chunk, 1 << k)
        want = oracle_prefix(Q, k, n_done)
        assert (e, oracle.rank_of_bits(x), t) == tuple(want)
        if done:
            break
    assert calls == (1 << k) // chunk
    full = O.solve(Q)
    assert (e, t) == (full[0], full[2]) and (x == full[1]).all()


def test_fp32_checkpointed(q, tmp_path):
    Q = qi.random_symmetric_normal_f32(24, 3102)
    path = str(tmp_path / "c.ckpt")
    while True:
        done, e, x, t, n_done = q.solve_checkpointed(Q, 4, path, slices_per_chunk=3, time_budget_s=1e-9)
        if done:
            break
    want = q.solve(Q)
    assert e == want[0] and (x == want[1]).all() and t == want[2]
