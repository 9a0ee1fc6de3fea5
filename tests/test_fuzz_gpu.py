"""Seeded random parity sweep: many small problems of every representation against the oracle.

Each trial draws a size, an entry range (packed-narrow, biased, wide int32, non-negative or
fp32 N(0,1)), a few decoupled variables (zero rows and columns, which multiply the minimum's
multiplicity), and sometimes an explicit (k_prefix, cache_bits) split; batched trials mix
instances of different ranges in one call. int32 results must be bit-exact (energy, lowest-rank
argmin, tie count); fp32 energies within 1e-3 * sum|Q| * 2^-20 with the oracle's argmin.
"""
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


def _instance(rng, n, kind, seed):
    if kind == "fp32":
        Q = qi.random_symmetric_normal_f32(n, seed)
    else:
        lo, hi = {"narrow": (-int(rng.integers(1, 20)), int(rng.integers(1, 20))), "mid": (-1000, 1000),
                  "wide": (-(1 << 20), 1 << 20), "pos": (0, 5)}[kind]
        Q = qi.random_upper_int(n, lo, hi, seed)
    for v in rng.choice(n, size=int(rng.integers(0, min(4, n) + 1)), replace=False):
        Q[v, :] = 0
        Q[:, v] = 0
    return Q


@pytest.mark.parametrize("seed", [1, 2])
def test_random_single_problems(q, seed):
    rng = np.random.default_rng(seed)
    checked = 0
    while checked < 60:
        n = int(rng.integers(1, 25))
        kind = str(rng.choice(["narrow", "mid", "wide", "pos", "fp32"]))
        Q = _instance(rng, n, kind, int(rng.integers(0, 1 << 30)))
        kw = {}
        if rng.random() < 0.4 and n > 2:
            kw = dict(k_prefix=int(rng.integers(0, n)), cache_bits=int(rng.integers(0, n)))
        try:
            e, x, t = q.solve(Q, **kw)
        except q.QuboError as err:
            assert kw and err.status == -4, (n, kind, kw, err.status)  # QUBO_ERR_PLAN: infeasible split
            continue
        want = O.solve(Q)
        if kind == "fp32":
            assert abs(e - want[0]) <= 1e-3 * float(np.abs(Q.astype(np.float64)).sum()) * 2.0 ** -20
            assert (x == want[1]).all() and t == want[2], (n, kw)
        else:
            assert (e, t) == (want[0], want[2]) and (x == want[1]).all(), (n, kind, kw)
        checked += 1


@pytest.mark.parametrize("seed", [3, 4])
def test_random_batches(q, seed):
    rng = np.random.default_rng(seed)
    for _ in range(4):
        n = int(rng.integers(18, 25))
        batch = int(rng.integers(1, 12))
        base = int(rng.integers(0, 1 << 30))
        Qs = np.stack([_instance(rng, n, str(rng.choice(["narrow", "mid", "pos"])), base + b) for b in range(batch)])
        e, x, t = q.solve_batched(Qs)
        for b in range(batch):
            want = O.solve(Qs[b])
            assert (int(e[b]), int(t[b])) == (want[0], want[2]) and (x[b] == want[1]).all(), (n, b)


@pytest.mark.parametrize("seed", [5])
def test_random_lowest_spectra(q, seed):
    # the k lowest (energy, rank) keys, bit-exact against the oracle's sorted top-k
    rng = np.random.default_rng(seed)
    for _ in range(20):
        n = int(rng.integers(2, 21))
        Q = _instance(rng, n, str(rng.choice(["narrow", "mid", "pos"])), int(rng.integers(0, 1 << 30)))
        k = int(rng.integers(1, 400))
        e, x = q.solve_lowest(Q, k)
        we, wx = O.lowest(Q, k)
        assert np.array_equal(e, we) and np.array_equal(x, wx), (n, k)


@pytest.mark.parametrize("seed", [5, 6])
def test_random_problems_of_the_bounded_pass(q, seed):
    # n >= 30 with 2^12 columns: the block-bounded biased pass (every range that fits the fp32
    # binade, and fp32 input) or the int32 pass (wide); decoupled variables put minimisers in
    # many units and blocks at once; slices give each group its own threshold
    rng = np.random.default_rng(seed)
    for _ in range(3):
        n = int(rng.integers(30, 32))
        kind = str(rng.choice(["narrow", "mid", "wide", "pos", "fp32"]))
        Q = _instance(rng, n, kind, int(rng.integers(0, 1 << 30)))
        e, x, t = q.solve(Q)
        want = O.solve(Q)
        if kind == "fp32":
            assert abs(e - want[0]) <= 1e-3 * float(np.abs(Q.astype(np.float64)).sum()) * 2.0 ** -20
            assert (x == want[1]).all() and t == want[2], (n, kind)
        else:
            assert (e, t) == (want[0], want[2]) and (x == want[1]).all(), (n, kind)
    for _ in range(2):
        n, k = int(rng.integers(34, 38)), int(rng.integers(6, 9))
        kind = str(rng.choice(["narrow", "mid", "pos", "fp32"]))
        Q = _instance(rng, n, kind, int(rng.integers(0, 1 << 30)))
        ids = np.unique(rng.integers(0, 1 << k, 3)).astype(np.uint64)
        e, x, t = q.solve_slices(Q, k, ids)
        for i, sid in enumerate(ids):
            want = O.solve_slice(Q, k, int(sid))
            if kind == "fp32":
                assert abs(float(e[i]) - want[0]) <= 1e-3 * float(np.abs(Q.astype(np.float64)).sum()) * 2.0 ** -20
                assert (x[i] == want[1]).all() and int(t[i]) == want[2], (n, k, int(sid))
            else:
                assert (int(e[i]), int(t[i])) == (want[0], want[2]) and (x[i] == want[1]).all(), (n, k, int(sid))
