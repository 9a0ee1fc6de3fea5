"""GPU parity of the k-lowest-energies entry point (through the C ABI) against the oracle."""
import itertools

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


# ---------------------------------------------------------------- n >= 30: the bounded driver
# From 30 variables the driver's minimum pass runs with block bounds and a margin that it widens
# until k states lie within it. Two instance families whose k lowest keys are known exactly at
# that size pin it.

def _full_rank(bits_by_pos, n):
    """Ranks of the rows of a (m, n) bit matrix whose column i is variable x_i."""
    w = np.array([1 << (n - 1 - i) for i in range(n)], dtype=np.uint64)
    return (bits_by_pos.astype(np.uint64) * w).sum(axis=1)


@pytest.mark.parametrize("n,n0,k,seed,scale,rng_core,rng_d", [
    (30, 18, 1000, 1, 1, 1000, 400), (31, 19, 4000, 2, 1, 1000, 400), (32, 20, 300, 3, 1, 1000, 400),
    (30, 18, 1000, 4, 1024, 1000, 400), (30, 18, 500, 5, 1, 9, 5)])
def test_lowest_bounded_separable_instances(q, n, n0, k, seed, scale, rng_core, rng_d):
    # n0 coupled variables at random positions and n - n0 variables with a diagonal term only:
    # E(x) = E_core(x_core) + sum_i d_i x_i. If c lies beyond the core's k lowest (ties at the
    # k-th energy included), k core states c' have E(c') < E(c), and every (c', y) lies strictly
    # below (c, y); so the k lowest keys combine the core's k lowest (the oracle's) with all
    # 2^(n - n0) diagonal parts. scale 1024 puts sum |U| above 2^22 (the int32 bounded pass);
    # entries to 9 keep it below 2^14 (the packed bounded pass)
    rng = qi.Stream(3100 + seed)
    pos = np.sort(np.argsort(rng.raw(n))[:n0])
    free = np.array([i for i in range(n) if i not in set(pos.tolist())])
    core = qi.random_upper_int(n0, -rng_core, rng_core, 3110 + seed) * np.int32(scale)
    d = rng.integers(-rng_d, rng_d, n - n0) * scale
    Q = np.zeros((n, n), np.int32)
    Q[np.ix_(pos, pos)] = core
    Q[free, free] = d
    assert q.plan(n)["pruned"] == 1
    # the core's k lowest keys and every other core state at the k-th energy
    kc = k + 1
    ce, cx = O.lowest(core, kc)
    while len(ce) == kc and ce[-1] == ce[k - 1]:
        kc *= 2
        ce, cx = O.lowest(core, kc)
    keep = ce <= ce[k - 1]
    ce, cx = ce[keep], cx[keep]
    f = n - n0
    fx = ((np.arange(1 << f)[:, None] >> np.arange(f - 1, -1, -1)[None, :]) & 1).astype(np.uint8)
    fe = fx.astype(np.int64) @ d.astype(np.int64)
    # energy and rank of (core state a, diagonal part b): each the sum of its two parts
    wbit = np.array([1 << (n - 1 - i) for i in range(n)], dtype=np.uint64)
    cr = (cx.astype(np.uint64) * wbit[pos]).sum(axis=1)
    fr = (fx.astype(np.uint64) * wbit[free]).sum(axis=1)
    E = (ce[:, None] + fe[None, :]).reshape(-1)
    R = (cr[:, None] + fr[None, :]).reshape(-1)
    order = np.lexsort((R, E))[:k]
    e, x = q.solve_lowest(Q, k)
    assert np.array_equal(e, E[order])
    assert np.array_equal(_full_rank(x, n), R[order])
    U = O.fold_i32(Q)
    for i in (0, k // 2, k - 1):
        assert O.energy_i64(U, x[i]) == int(e[i])


@pytest.mark.parametrize("k", [1, 100, 1500, 6000])
def test_lowest_bounded_equal_weight_mattis(q, k):
    # J_ij = -s*_i s*_j (i < j), h = 0, as a QUBO: Q_ij = 4 J_ij, Q_ii = -2 sum_j J_ij. With
    # m = n - 2 L the overlap of the spins with s* at Hamming distance L, H = -(m^2 - n) / 2, so
    # the k lowest keys are the states at distance L = 0, 1, 2, ... from x* or from its
    # complement, by level and then by rank. The level gaps (62, 58, 54 at n = 32) exceed
    # sum |U| / 64, so the driver's first margin holds only the two ground states
    n = 32
    s = qi.Stream(3200).signs(n).astype(np.int64)
    J = -np.outer(s, s)
    Q = np.zeros((n, n), np.int64)
    for i in range(n):
        for j in range(i + 1, n):
            Q[i, j] = 4 * J[i, j]
        Q[i, i] = -2 * (J[i].sum() - J[i, i])
    Q = Q.astype(np.int32)
    xs = ((s + 1) // 2).astype(np.uint8)
    states, levels = [], []
    for L in range(4):
        for c in itertools.combinations(range(n), L):
            y = xs.copy()
            y[list(c)] ^= 1
            states += [y, 1 - y]
            levels += [L, L]
    states = np.array(states, np.uint8)
    levels = np.array(levels)
    R = _full_rank(states, n)
    order = np.lexsort((R, levels))[:k]
    assert k <= len(order)
    e, x = q.solve_lowest(Q, k)
    assert np.array_equal(_full_rank(x, n), R[order])
    U = O.fold_i32(Q)
    E0 = O.energy_i64(U, xs)
    assert int(e[0]) == E0
    m0 = n
    for i in range(k):
        m = n - 2 * int(levels[order[i]])
        assert int(e[i]) == E0 + (m0 * m0 - m * m) // 2
    for i in sorted({0, k // 3, k - 1}):
        assert O.energy_i64(U, x[i]) == int(e[i])
