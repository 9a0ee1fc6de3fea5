"""GPU parity of the k-lowest-energies entry point (through the C ABI) against the oracle."""
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


def keys(e, x):
    return [(int(a), oracle.rank_of_bits(b)) for a, b in zip(e, x)]


@pytest.mark.parametrize("n,lo,hi,k,seed", [(10, -50, 50, 64, 1), (18, -1000, 1000, 1, 2), (18, -1000, 1000, 1000, 3),
                                            (22, -300, 300, 500, 4), (20, -1, 1, 5000, 5), (16, -9, 9, 3000, 6)])
def test_lowest_against_oracle(q, n, lo, hi, k, seed):
    Q = qi.random_upper_int(n, lo, hi, 3000 + seed)
    e, x = q.solve_lowest(Q, k)
    we, wx = O.lowest(Q, k)
    assert keys(e, x) == keys(we, wx)


def test_lowest_whole_spectrum_of_a_small_problem(q):
    Q = qi.random_full_int(6, -30, 30, 3010)
    e, x = q.solve_lowest(Q, 100)  # only 64 states exist
    we, wx = O.lowest(Q, 100)
    assert len(e) == 64 and keys(e, x) == keys(we, wx)


def test_lowest_fully_degenerate_spectrum(q):
    # Q = 0: all 2^20 states tie, more than the candidate buffer: the rank bisection path
    e, x = q.solve_lowest(np.zeros((20, 20), np.int32), 100)
    assert (e == 0).all() and [oracle.rank_of_bits(s) for s in x] == list(range(100))


def test_lowest_k1_matches_solve_and_n32_properties(q):
    n, k = 32, 200
    Q = qi.random_upper_int(n, -1000, 1000, 3020)
    e, x = q.solve_lowest(Q, k)
    s = q.solve(Q)
    assert e[0] == s[0] and (x[0] == s[1]).all()
    ks = keys(e, x)
    assert ks == sorted(ks) and len(set(r for _, r in ks)) == k
    U = O.fold_i32(Q)
    for (E, _), st in zip(ks, x):
        assert O.energy_i64(U, st) == E
    # completeness on sampled slices: every state of a slice whose key is below the k-th key is
    # in the result
    kth = ks[-1]
    got = set(ks)
    kp = 12
    for p in qi.Stream(3021).integers(0, (1 << kp) - 1, 3):
        lo = int(p) << (n - kp)
        se, sx = O.lowest(Q, k, lo, lo + (1 << (n - kp)))
        for key in keys(se, sx):
            if key < kth:
                assert key in got


def test_lowest_argument_errors(q):
    with pytest.raises(q.QuboError) as ei:
        q.solve_lowest(qi.random_symmetric_normal_f32(8, 1), 4)
    assert ei.value.status == -1
    with pytest.raises(q.QuboError):
        q.solve_lowest(np.zeros((8, 8), np.int32), 0)
