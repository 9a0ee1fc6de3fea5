"""Pins for the CPU oracle against what the pages and the mathematics fix (no GPU needed).

Each pin is chosen so that a plausible slip in the oracle (a dropped term, a wrong sign or
index, a transposed operand, a wrong tie rule) fails at least one of them; the mutant builds
in test_oracle_mutants.py check exactly that.
"""
import itertools
import math

import numpy as np
import pytest

import oracle
import qubo_instances as qi
from conftest import read_golden

O = oracle.get()


def brute_raw(Q):
    """Pure-Python brute force straight from E(x) = sum_{i,j} Q_ij x_i x_j (tiny n only)."""
    n = len(Q)
    best, arg, ties = None, None, 0
    for r, x in enumerate(itertools.product((0, 1), repeat=n)):  # lexicographic = rank order
        e = sum(int(Q[i][j]) for i in range(n) for j in range(n) if x[i] and x[j])
        if best is None or e < best:
            best, arg, ties = e, r, 1
        elif e == best:
            ties += 1
    return best, arg, ties


# ---------------------------------------------------------------- Gray code (Fig. 5)

def test_gray_sequence_matches_fig5():
    rows = read_golden("gray3_fig5.txt")
    for idx, code in rows:
        assert format(O.gray_code(int(idx)), "03b") == code


def test_gray_flip_is_single_bit_of_fig5():
    codes = [int(c, 2) for _, c in read_golden("gray3_fig5.txt")]
    for i in range(len(codes) - 1):
        diff = codes[i] ^ codes[i + 1]
        assert diff & (diff - 1) == 0 and diff != 0
        assert diff == 1 << O.gray_flip_bit(i)


def test_walker_visits_fig5_order():
    # With x_0 as the leftmost bit, the walker's state sequence for n = 3 is Fig. 5's.
    U = O.fold_i32(qi.random_upper_int(3, -5, 5, 1))
    _, R = O.gray_trace_i64(U)
    assert [format(int(r), "03b") for r in R] == [c for _, c in read_golden("gray3_fig5.txt")]


def test_gray_visits_every_state_once():
    for n in (1, 5, 10):
        seq = [O.gray_code(i) for i in range(1 << n)]
        assert sorted(seq) == list(range(1 << n))


# ---------------------------------------------------------------- energies

@pytest.mark.parametrize("seed", range(5))
def test_energy_basics(seed):
    n = 9
    Q = qi.random_full_int(n, -50, 50, seed)
    U = O.fold_i32(Q)
    zero = np.zeros(n, np.uint8)
    assert O.energy_i64(U, zero) == 0 == O.energy_raw_i32(Q, zero)  # E(0) = 0
    for i in range(n):
        e = np.zeros(n, np.uint8)
        e[i] = 1
        assert O.energy_i64(U, e) == Q[i, i] == O.energy_raw_i32(Q, e)  # E(e_i) = Q_ii
    rng = np.random.default_rng(seed)
    for _ in range(50):
        x = rng.integers(0, 2, n).astype(np.uint8)
        e = O.energy_raw_i32(Q, x)
        assert O.energy_i64(U, x) == e  # folding keeps E
        assert O.energy_raw_i32(Q.T.copy(), x) == e  # E(Q) = E(Q^T)
        assert O.energy_raw_i32(Q + Q.T, x) == 2 * e  # E(Q + Q^T) = 2 E(Q)
        assert O.energy_i64(O.fold_i32(Q.T.copy()), x) == e


def test_fold_is_upper_triangle():
    Q = qi.random_full_int(6, -9, 9, 3)
    U = O.fold_i32(Q)
    for i in range(6):
        for j in range(6):
            if j < i:
                assert U[i, j] == 0
            elif j == i:
                assert U[i, j] == Q[i, i]
            else:
                assert U[i, j] == Q[i, j] + Q[j, i]


def test_eval64_matches_integer_energy_when_exact():
    n = 10
    Q = qi.random_full_int(n, -1000, 1000, 7)
    Ui = O.fold_i32(Q)
    Uf = O.fold_f32(Q.astype(np.float32))
    rng = np.random.default_rng(0)
    for _ in range(100):
        x = rng.integers(0, 2, n).astype(np.uint8)
        assert O.eval64(Uf, x) == float(O.energy_i64(Ui, x))


def test_walker_energies_equal_direct_energies():
    # Walker (local fields, incremental) against from-scratch evaluation, every state, n <= 12.
    for n, seed in ((1, 0), (2, 1), (7, 2), (12, 3)):
        Q = qi.random_full_int(n, -300, 300, seed)
        U = O.fold_i32(Q)
        E, R = O.gray_trace_i64(U)
        for e, r in zip(E, R):
            assert e == O.energy_i64(U, oracle.bits_of_rank(n, int(r)))


# ---------------------------------------------------------------- searches vs brute force

@pytest.mark.parametrize("n,lo,hi,seed", [(1, -3, 3, 0), (2, -3, 3, 1), (3, -2, 2, 2), (5, -2, 2, 3),
                                          (6, -1, 1, 4), (7, -5, 5, 5), (8, -3, 3, 6), (8, -100, 100, 7)])
def test_searches_equal_python_brute_force(n, lo, hi, seed):
    Q = qi.random_full_int(n, lo, hi, seed)
    want = brute_raw(Q.tolist())
    U = O.fold_i32(Q)
    assert O.direct_i64(U) == want
    assert O.gray_i64(U) == want
    Uf = O.fold_f32(Q.astype(np.float32))
    e, r, t = O.direct_f64(Uf)
    assert (e, r, t) == (float(want[0]), want[1], want[2])
    e, r, t = O.gray_f64(Uf)
    assert (e, r, t) == (float(want[0]), want[1], want[2])


@pytest.mark.parametrize("n,seed", [(14, 0), (16, 1), (18, 2)])
def test_direct_equals_gray_walker(n, seed):
    U = O.fold_i32(qi.random_upper_int(n, -100, 100, seed))
    assert O.direct_i64(U) == O.gray_i64(U)


def test_direct_equals_gray_walker_with_many_ties():
    U = O.fold_i32(qi.random_upper_int(15, -1, 1, 11))
    d = O.direct_i64(U)
    assert d == O.gray_i64(U)
    assert d[2] > 1


# ---------------------------------------------------------------- closed forms

@pytest.mark.parametrize("n", [1, 5, 13])
def test_zero_matrix(n):
    U = np.zeros((n, n), np.int64)
    assert O.gray_i64(U) == (0, 0, 1 << n)
    assert O.direct_i64(U) == (0, 0, 1 << n)


@pytest.mark.parametrize("seed", range(4))
def test_diagonal_matrix(seed):
    n = 12
    d = qi.Stream(seed).integers(-3, 3, n)
    Q = np.diag(d).astype(np.int32)
    e_want = int(np.minimum(d, 0).sum())
    x_want = (d < 0).astype(np.uint8)  # zero diagonal: x_i = 0 has the lower rank
    ties_want = 1 << int((d == 0).sum())
    e, x, t = O.solve(Q)
    assert (e, t) == (e_want, ties_want) and (x == x_want).all()
    e, x, t = O.solve(Q, method="direct")
    assert (e, t) == (e_want, ties_want) and (x == x_want).all()


def test_positive_matrix_has_unique_zero_minimum():
    Q = qi.random_upper_int(13, 1, 9, 5)
    e, x, t = O.solve(Q)
    assert e == 0 and t == 1 and not x.any()


# ---------------------------------------------------------------- planted instances

def test_ising_to_qubo_conversion_by_brute_force():
    n = 6
    s = qi.Stream(9)
    J = np.triu(s.integers(-5, 5, n * n).reshape(n, n), 1)
    h = s.integers(-4, 4, n)
    Q, offset = qi.ising_to_qubo(J, h)
    for x in itertools.product((0, 1), repeat=n):
        sp = [2 * b - 1 for b in x]
        H = sum(J[i, j] * sp[i] * sp[j] for i in range(n) for j in range(i + 1, n)) + sum(h[i] * sp[i] for i in range(n))
        assert H == O.energy_raw_i32(Q.astype(np.int32), np.array(x, np.uint8)) + offset


@pytest.mark.parametrize("n", [4, 8, 12, 16])
def test_mattis_unit_weights_matches_page_ground_energy(n):
    want = {int(a): int(b) for a, b in read_golden("mattis_ground_energy.txt")}
    Q, s_star, w, offset = qi.mattis_planted(n, 100 + n, wlo=1, whi=1)
    e, x, t = O.solve(Q)
    assert 2 * (e + offset) == -n * (n - 1)  # the page's form 2E = -n(n-1)
    assert e + offset == want[n]
    assert t == 2


@pytest.mark.parametrize("n,seed", [(10, 0), (14, 1), (18, 2), (20, 3)])
def test_mattis_planted_closed_form(n, seed):
    Q, s_star, w, offset = qi.mattis_planted(n, seed)
    differ = np.not_equal.outer(s_star, s_star)
    e_want = -2 * int(np.triu(w * differ, 1).sum())
    xs = ((1 + s_star) // 2).astype(np.uint8)
    x_want = xs if xs[0] == 0 else 1 - xs
    e, x, t = O.solve(Q)
    assert e == e_want and t == 2 and (x == x_want).all()


# ---------------------------------------------------------------- the subproblem split (§III-C1)

def test_slice_identity_and_slice_minima():
    n, k = 11, 4
    Q = qi.random_full_int(n, -60, 60, 21)
    U = O.fold_i32(Q)
    E, R = O.gray_trace_i64(U)
    energy_by_rank = np.empty(1 << n, np.int64)
    energy_by_rank[R.astype(np.int64)] = E
    best = None
    for p in range(1 << k):
        c, Qr = O.subproblem_i64(U, k, p)
        m = n - k
        for xr_rank in range(1 << m):
            xr = oracle.bits_of_rank(m, xr_rank)
            assert c + O.energy_i64(Qr, xr) == energy_by_rank[(p << m) | xr_rank]
        sl = O.gray_i64(U, k, p)
        block = energy_by_rank[p << m:(p + 1) << m]
        emin = int(block.min())
        assert sl == (emin, (p << m) + int(np.argmin(block)), int((block == emin).sum()))
        assert O.direct_i64(U, p << m, (p + 1) << m) == sl
        best = emin if best is None else min(best, emin)
    assert best == O.gray_i64(U)[0]


# ---------------------------------------------------------------- fp64 path

@pytest.mark.parametrize("n,seed", [(9, 0), (13, 1), (15, 2)])
def test_fp64_walker_equals_direct(n, seed):
    Q = qi.random_symmetric_normal_f32(n, seed)
    U = O.fold_f32(Q)
    assert O.gray_f64(U) == O.direct_f64(U)


def test_fp64_band_is_tiny_and_min_is_below_every_sampled_state():
    Q = qi.random_symmetric_normal_f32(16, 4)
    U = O.fold_f32(Q)
    assert O.walk_bound_f64(U, 10) < 1e-6
    e, r, t = O.gray_f64(U)
    rng = np.random.default_rng(1)
    for _ in range(200):
        x = rng.integers(0, 2, 16).astype(np.uint8)
        assert O.eval64(U, x) >= e
    assert O.eval64(U, oracle.bits_of_rank(16, r)) == e


def test_fp64_diagonal_closed_form():
    d = np.array([0.5, -1.25, 0.0, -3.0, 2.0, -0.125], np.float32)
    Q = np.diag(d)
    e, x, t = O.solve(Q)
    assert e == float(np.minimum(d, 0).astype(np.float64).sum()) and t == 2
    assert (x == (d < 0)).all()


def test_generator_stream_definition():
    # Block form equals the scalar definition; rejection sampling stays in range.
    for k in range(1, 20):
        assert int(qi.splitmix64_block(123, k - 1, 1)[0]) == qi.splitmix64_scalar(123, k)
    v = qi.Stream(5).integers(-1000, 1000, 5000)
    assert v.min() >= -1000 and v.max() <= 1000
    z = qi.Stream(6).normals(20000)
    assert abs(z.mean()) < 0.05 and abs(z.std() - 1) < 0.05


# ---------------------------------------------------------------- Ising form (§I)

def brute_ising(J, h):
    """Pure-Python H(s) = sum_{i,j} J_ij s_i s_j + sum_i h_i s_i over all s (tiny n only)."""
    n = len(J)
    best, arg, ties = None, None, 0
    for r, x in enumerate(itertools.product((0, 1), repeat=n)):
        s = [2 * b - 1 for b in x]
        H = sum(int(J[i][j]) * s[i] * s[j] for i in range(n) for j in range(n)) + sum(int(h[i]) * s[i] for i in range(n))
        if best is None or H < best:
            best, arg, ties = H, r, 1
        elif H == best:
            ties += 1
    return best, arg, ties


def test_ising_two_spin_example():
    # H = s0 s1: the two anti-aligned states are the ground states, H = -1; x = (0, 1) has rank 1
    H, s, t = O.ising_direct(np.array([[0, 1], [0, 0]], np.int64))
    assert (H, t) == (-1, 2) and list(s) == [-1, 1]


def test_ising_field_only_closed_form():
    h = np.array([3, -2, 0, 5, -1], np.int64)
    H, s, t = O.ising_direct(np.zeros((5, 5), np.int64), h)
    assert H == -int(np.abs(h).sum()) and t == 2  # one free spin (h = 0)
    assert list(s) == [-1, 1, -1, -1, 1]          # s_i = -sign(h_i); the free spin takes -1 (rank)


@pytest.mark.parametrize("seed", [1, 2, 3])
def test_ising_direct_matches_brute_force(seed):
    st = qi.Stream(700 + seed)
    n = 7
    J = st.integers(-9, 9, n * n).reshape(n, n)
    h = st.integers(-9, 9, n)
    H, s, t = O.ising_direct(J, h)
    bh, br, bt = brute_ising(J, h)
    assert (H, t) == (bh, bt)
    assert list(s) == [2 * ((br >> (n - 1 - i)) & 1) - 1 for i in range(n)]
    Hf, sf, tf = O.ising_direct(J.astype(np.float64), h.astype(np.float64))  # fp64 twin
    assert (Hf, tf) == (float(bh), bt) and (sf == s).all()


def test_ising_direct_invariances():
    st = qi.Stream(711)
    n = 9
    J = st.integers(-20, 20, n * n).reshape(n, n)
    h = st.integers(-20, 20, n)
    H, s, t = O.ising_direct(J, h)
    assert O.ising_direct(J.T, h)[0] == H                        # only J_ij + J_ji matters
    Jd = J + np.diag(st.integers(-5, 5, n))
    assert O.ising_direct(Jd, h)[0] == H + int(np.diag(Jd - J).sum())  # J_ii s_i^2 is a constant
    assert O.ising_direct(J, -h)[0] == O.ising_direct(J, h)[0]   # s -> -s symmetry of the pair terms


@pytest.mark.parametrize("n,seed", [(10, 4), (14, 5), (18, 6)])
def test_ising_direct_mattis_closed_form(n, seed):
    s_star, w, J = qi.mattis_couplings(n, 1, 100, seed)
    H, s, t = O.ising_direct(J)
    assert H == -int(np.triu(w, 1).sum()) and t == 2
    want = s_star if s_star[0] == -1 else -s_star
    assert (s == want).all()


# ---------------------------------------------------------------- lowest part of the spectrum

def brute_spectrum(Q):
    """All (E, rank) pairs of x^T Q x sorted by energy then rank (pure Python, tiny n)."""
    n = len(Q)
    keys = []
    for r, x in enumerate(itertools.product((0, 1), repeat=n)):
        keys.append((sum(int(Q[i][j]) for i in range(n) for j in range(n) if x[i] and x[j]), r))
    return sorted(keys)


@pytest.mark.parametrize("seed", [1, 2])
def test_lowest_matches_sorted_brute_force(seed):
    n = 8
    Q = qi.random_full_int(n, -20, 20, 730 + seed)
    want = brute_spectrum(Q)
    for k in (1, 5, 37, 1 << n, (1 << n) + 10):
        e, x = O.lowest(Q, k)
        got = [(int(a), oracle.rank_of_bits(b)) for a, b in zip(e, x)]
        assert got == want[:k]


def test_lowest_k1_is_the_minimum_and_ranges_merge():
    Q = qi.random_upper_int(14, -50, 50, 733)
    e, x = O.lowest(Q, 1)
    m = O.solve(Q)
    assert e[0] == m[0] and (x[0] == m[1]).all()
    k, n = 40, 14
    whole = O.lowest(Q, k)
    a, b = O.lowest(Q, k, 0, 5000), O.lowest(Q, k, 5000, 1 << n)
    merged = sorted([(int(v), oracle.rank_of_bits(s)) for v, s in zip(*a)] +
                    [(int(v), oracle.rank_of_bits(s)) for v, s in zip(*b)])[:k]
    assert merged == [(int(v), oracle.rank_of_bits(s)) for v, s in zip(*whole)]


def test_lowest_degenerate_and_diagonal_closed_forms():
    e, x = O.lowest(np.zeros((10, 10), np.int32), 7)  # every state ties: ranks 0..6
    assert (e == 0).all() and [oracle.rank_of_bits(s) for s in x] == list(range(7))
    d = np.array([-5, 3, -2, 0], np.int32)  # E = sum of the chosen diagonal entries
    e, x = O.lowest(np.diag(d), 16)
    sub = sorted((int(sum(d[i] for i in range(4) if (r >> (3 - i)) & 1)), r) for r in range(16))
    assert [(int(a), oracle.rank_of_bits(b)) for a, b in zip(e, x)] == sub
