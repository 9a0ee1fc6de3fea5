"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle on identical seeded inputs.

int32: bit-exact (minimum energy, lowest-rank argmin, tie count).
fp32:  the returned energy is the fixed-order fp64 energy of the returned state, and it lies
       within 1e-3 * sum|Q_ij| * 2^-20 of the oracle's fp64 minimum.
"""
import contextlib

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


def fp32_tol(Q):
    return 1e-3 * float(np.abs(Q.astype(np.float64)).sum()) * 2.0 ** -20


def check_int(q, Q, **kw):
    e, x, t = q.solve(Q, **kw)
    want = O.solve(Q)
    assert (e, t) == (want[0], want[2]), (e, t, want)
    assert (x == want[1]).all()
    return e, x, t


@contextlib.contextmanager
def no_bounds(q):
    """Calls planned inside take the minimum passes without block bounds (packed or biased)."""
    q.enable_block_bounds(False)
    try:
        yield
    finally:
        q.enable_block_bounds(True)


# ---------------------------------------------------------------- exhaustive small sweeps

@pytest.mark.parametrize("n", list(range(1, 17)))
def test_small_n_sweep(q, n):
    for seed, (lo, hi) in enumerate([(-100, 100), (-2, 2), (-1, 1), (0, 3)]):
        check_int(q, qi.random_upper_int(n, lo, hi, 1000 * n + seed))
    check_int(q, qi.random_full_int(n, -50, 50, 7 * n))  # non-triangular input


@pytest.mark.parametrize("n", [1, 2, 7, 12, 17, 20])
def test_zero_matrix_all_states_tie(q, n):
    e, x, t = q.solve(np.zeros((n, n), np.int32))
    assert e == 0 and t == 1 << n and not x.any()


@pytest.mark.parametrize("n", [5, 14, 19])
def test_diagonal_closed_form(q, n):
    d = qi.Stream(n).integers(-3, 3, n)
    e, x, t = q.solve(np.diag(d).astype(np.int32))
    assert e == int(np.minimum(d, 0).sum())
    assert (x == (d < 0)).all()
    assert t == 1 << int((d == 0).sum())


# every kernel variant and split: explicit (k_prefix, cache_bits)
@pytest.mark.parametrize("n,k,c", [
    (16, 0, 9), (17, 0, 12), (18, 1, 12), (20, 3, 12), (20, 0, 9), (21, 4, 10), (22, 2, 11),
    (20, 6, 9), (14, 2, 6), (12, 0, 10), (13, 5, 3), (15, 14, 1), (10, 4, 6), (18, 8, 10), (9, 9, 0),
])
def test_explicit_plans(q, n, k, c):
    for seed, (lo, hi) in enumerate([(-100, 100), (-1, 1)]):
        Q = qi.random_upper_int(n, lo, hi, 77 * n + 3 * k + c + seed)
        check_int(q, Q, k_prefix=k, cache_bits=c)


def test_infeasible_explicit_plan_is_an_error(q):
    Q = qi.random_upper_int(20, -9, 9, 2)
    with pytest.raises(q.QuboError) as ei:
        q.solve(Q, k_prefix=2, cache_bits=16)
    assert ei.value.status == -4


def test_plans_pick_fast_kernel_for_large_n(q):
    p = q.plan(40)
    assert p["variant"] == 1 and p["cache_bits"] == 12 and p["units"] >= 1024
    # the bounded passes; the packed one is planned too (it checks sum |U| < 2^14 on the device
    # and exits at once otherwise, leaving the biased or int32 pass to run)
    assert p["pruned"] == 1 and p["biased"] == 1 and p["packed"] == 1
    with no_bounds(q):
        p = q.plan(40)
        assert p["pruned"] == 0 and p["biased"] == 1 and p["packed"] == 1
        assert q.plan(40, q.FP32)["pruned"] == 0
    assert q.plan(40)["pruned"] == 1
    assert q.plan(8)["variant"] == 0
    # fp32 input: its fixed-point image is scaled into the biased pass's range; never packed
    assert q.plan(36, q.FP32)["biased"] == 1 and q.plan(36, q.FP32)["packed"] == 0


@pytest.mark.parametrize("n,seed", [(16, 1), (17, 2), (19, 3), (23, 4), (27, 5)])
def test_fast_split_boundaries(q, n, seed):
    # the smallest splits of the register-row kernel, wide and narrow entries
    check_int(q, qi.random_upper_int(n, -1000, 1000, seed))
    check_int(q, qi.random_upper_int(n, -3, 3, seed + 100))


def _with_abs_sum(Q, total):
    """Q with Q[0, 0] changed so that sum |Q_ij| (upper triangle) is exactly `total`."""
    Q = Q.copy()
    Q[0, 0] = 0
    rest = int(np.abs(Q.astype(np.int64)).sum())
    assert 0 <= total - rest < (1 << 31)
    Q[0, 0] = -(total - rest)
    assert int(np.abs(Q.astype(np.int64)).sum()) == total
    return Q


@pytest.mark.parametrize("sign", ["mixed", "negative", "positive"])
def test_biased_walk_range_limit_is_exact(q, sign):
    # The biased minimum walk, with and without block bounds, keeps column energies in the fp32
    # binade [2^23, 2^24) for sum |U| <= 2^22 - 1; above, the int32 walk runs. Both sides of the
    # limit through both passes and the k-lowest driver, with running values pushed to the
    # extremes: all-negative entries reach E = -sum |U| at x = 1, all-positive ones +sum |U|.
    n = 30
    lo, hi = {"mixed": (-15000, 15000), "negative": (-15000, -1), "positive": (1, 15000)}[sign]
    for total in ((1 << 22) - 1, 1 << 22):
        Q = np.triu(qi.random_upper_int(n, lo, hi, 2300 + total % 7))
        if sign == "positive":
            Q = np.abs(Q)
            Q[0, 0] = 0
            Q[0, 0] = total - int(np.abs(Q.astype(np.int64)).sum())
        else:
            Q = _with_abs_sum(Q, total)
        assert int(np.abs(Q.astype(np.int64)).sum()) == total
        assert q.plan(n)["pruned"] == 1
        e, x, t = check_int(q, Q)
        if sign == "negative":
            assert e == -total and x.all()
        with no_bounds(q):
            assert q.plan(n)["pruned"] == 0
            check_int(q, Q)
        le, lx = q.solve_lowest(Q, 1)
        assert int(le[0]) == e and (lx[0] == x).all()


def test_int32_walk_large_values(q):
    # sum |U| near 2^29: the minimum walk stays in int32 on the fast kernel
    Q = qi.random_upper_int(28, -(1 << 21), 1 << 21, 2301)
    assert int(np.abs(Q.astype(np.int64)).sum()) > (1 << 22)
    check_int(q, Q)


def test_fewer_threads_than_variables(q):
    # cache_bits = 9 gives 32-thread blocks (16 columns each) while n = 44 > 32: every variable's
    # per-unit linear term must still be formed
    n, k = 44, 22
    Q = qi.random_upper_int(n, -200, 200, 2470)
    assert q.plan(n, q.INT32, 0, 9)["threads_per_block"] < n
    ids = qi.Stream(2471).integers(0, (1 << k) - 1, 3).astype(np.uint64)
    e, x, t = q.solve_slices(Q, k, ids, cache_bits=9)
    for i, sid in enumerate(ids):
        want = O.solve_slice(Q, k, int(sid))
        assert (int(e[i]), int(t[i])) == (want[0], want[2]) and (x[i] == want[1]).all()


# ---------------------------------------------------------------- packed 16x2 minimum pass
# Narrow inputs (sum |U| < 2^14) take the packed pass, with block bounds by default and without
# them through the switch: both are checked, and the k-lowest driver on the same inputs.

@pytest.mark.parametrize("n,lo,hi,seed", [(30, -30, 30, 1), (30, -9, 9, 3), (31, -3, 3, 4), (31, 0, 2, 5)])
def test_packed_pass_small_range(q, n, lo, hi, seed):
    Q = qi.random_upper_int(n, lo, hi, 2400 + seed)
    assert int(np.abs(Q.astype(np.int64)).sum()) <= (1 << 14) - 1
    assert q.plan(n)["packed"] == 1 and q.plan(n)["pruned"] == 1
    e, x, t = check_int(q, Q)  # the bounded packed pass
    with no_bounds(q):
        assert q.plan(n)["packed"] == 1 and q.plan(n)["pruned"] == 0
        check_int(q, Q)  # the packed pass: every unit minimum feeds the tie and argmin passes
    le, lx = q.solve_lowest(Q, 1)
    assert int(le[0]) == e and (lx[0] == x).all()


@pytest.mark.parametrize("sign", ["mixed", "negative", "positive"])
def test_packed_range_limit_is_exact(q, sign):
    # sum |U| = 2^14 - 1 runs the packed pass (values pushed to +-sum |U|), 2^14 the biased
    # one; with and without block bounds
    n = 30
    lo, hi = {"mixed": (-50, 50), "negative": (-50, -1), "positive": (1, 50)}[sign]
    for total in ((1 << 14) - 1, 1 << 14):
        Q = np.triu(qi.random_upper_int(n, lo, hi, 2450 + total % 5))
        if sign == "positive":
            Q = np.abs(Q)
            Q[0, 0] = 0
            Q[0, 0] = total - int(np.abs(Q.astype(np.int64)).sum())
        else:
            Q = _with_abs_sum(Q, total)
        assert int(np.abs(Q.astype(np.int64)).sum()) == total
        e, x, t = check_int(q, Q)
        if sign == "negative":
            assert e == -total and x.all()
        with no_bounds(q):
            assert q.plan(n)["packed"] == 1  # planned; on the device it runs below 2^14 only
            check_int(q, Q)
        le, lx = q.solve_lowest(Q, 1)
        assert int(le[0]) == e and (lx[0] == x).all()


def test_packed_pass_all_ties(q):
    # Q = 0: every state ties; every block's bound equals the threshold, so the bounded packed
    # pass walks every block exactly, and the resolve pass counts 2^n; so does the unbounded one
    Z = np.zeros((30, 30), np.int32)
    e, x, t = q.solve(Z)
    assert (e, t) == (0, 1 << 30) and not x.any()
    with no_bounds(q):
        assert q.solve(Z)[2] == 1 << 30
    le, lx = q.solve_lowest(Z, 3)
    assert list(le) == [0, 0, 0] and [oracle.rank_of_bits(v) for v in lx] == [0, 1, 2]


def test_small_problems_run_the_int32_pass_alone(q):
    # below 30 variables only the int32 minimum pass is launched (launch-bound sizes)
    p = q.plan(24)
    assert p["packed"] == 0 and p["biased"] == 0
    check_int(q, qi.random_upper_int(24, -5, 5, 2480))


def test_n40_narrow_slices_against_oracle(q):
    Q = qi.workload_n40_narrow()
    assert q.plan(40)["pruned"] == 1
    k = 16
    ids = qi.Stream(4041).integers(0, (1 << k) - 1, 4).astype(np.uint64)
    e, x, t = q.solve_slices(Q, k, ids)
    for i, sid in enumerate(ids):
        want = O.solve_slice(Q, k, int(sid))
        assert (int(e[i]), int(t[i])) == (want[0], want[2]) and (x[i] == want[1]).all()


# ---------------------------------------------------------------- configs

def test_n20_config(q):
    Q = qi.workload_n20()
    e, x, t = check_int(q, Q)
    assert O.direct_i64(O.fold_i32(Q)) == (e, oracle.rank_of_bits(x), t)


def test_n24_random_and_ties(q):
    check_int(q, qi.random_upper_int(24, -1000, 1000, 5))
    check_int(q, qi.random_upper_int(24, -1, 1, 6))


def test_n32_config(q):
    check_int(q, qi.workload_n32())


def test_n32_mattis_planted(q):
    Q, s_star, w, offset = qi.workload_n32_mattis()
    differ = np.not_equal.outer(s_star, s_star)
    e_want = -2 * int(np.triu(w * differ, 1).sum())
    xs = ((1 + s_star) // 2).astype(np.uint8)
    x_want = xs if xs[0] == 0 else 1 - xs
    e, x, t = q.solve(Q)
    assert e == e_want and t == 2 and (x == x_want).all()


def test_n40_slices_against_oracle(q):
    Q = qi.workload_n40()
    k = 12
    ids = qi.Stream(4040).integers(0, (1 << k) - 1, 6).astype(np.uint64)
    e, x, t = q.solve_slices(Q, k, ids)
    for s, sid in enumerate(ids):
        want = O.solve_slice(Q, k, int(sid))
        assert (int(e[s]), int(t[s])) == (want[0], want[2])
        assert (x[s] == want[1]).all()


def test_maximum_size_n62_slices_against_oracle(q):
    # n = 62, the largest size the ABI takes: slices of 2^24 states (int32) and 2^22 (fp32)
    n = 62
    Q = qi.random_upper_int(n, -100, 100, 6262)
    k = 38
    ids = qi.Stream(6263).integers(0, (1 << k) - 1, 3).astype(np.uint64)
    e, x, t = q.solve_slices(Q, k, ids)
    for s, sid in enumerate(ids):
        want = O.solve_slice(Q, k, int(sid))
        assert (int(e[s]), int(t[s])) == (want[0], want[2]) and (x[s] == want[1]).all()
    Qf = qi.random_symmetric_normal_f32(n, 6264)
    k = 40
    ids = qi.Stream(6265).integers(0, (1 << k) - 1, 2).astype(np.uint64)
    e, x, t = q.solve_slices(Qf, k, ids)
    U = O.fold_f32(Qf)
    for s, sid in enumerate(ids):
        want = O.solve_slice(Qf, k, int(sid))
        assert O.eval64(U, x[s]) == e[s] and abs(e[s] - want[0]) <= fp32_tol(Qf)
        assert (x[s] == want[1]).all()


def test_n40_full_solve_consistent_with_sampled_slices(q):
    Q = qi.workload_n40()
    e, x, t = q.solve(Q)
    assert t >= 1
    U = O.fold_i32(Q)
    assert O.energy_i64(U, x) == e  # the reported state has the reported energy
    k = 12
    sid = oracle.rank_of_bits(x[:k])
    want = O.solve_slice(Q, k, sid)  # the slice holding the argmin has the same optimum
    assert want[0] == e and (want[1] == x).all() and 1 <= want[2] <= t
    for sid2 in qi.Stream(41).integers(0, (1 << k) - 1, 3):
        assert O.solve_slice(Q, k, int(sid2))[0] >= e


def test_slice_range_shards_combine_to_whole(q):
    Q = qi.random_upper_int(26, -300, 300, 9)
    whole = q.solve(Q)
    k = 6
    parts = [q.solve_slice_range(Q, k, a, 16) for a in range(0, 64, 16)]
    best = min(p[0] for p in parts)
    ties = sum(p[2] for p in parts if p[0] == best)
    first = min(oracle.rank_of_bits(p[1]) for p in parts if p[0] == best)
    assert (best, first, ties) == (whole[0], oracle.rank_of_bits(whole[1]), whole[2])


# ---------------------------------------------------------------- fp32

@pytest.mark.parametrize("n,seed", [(1, 0), (5, 1), (12, 2), (18, 3), (22, 4), (26, 5)])
def test_fp32_against_oracle(q, n, seed):
    Q = qi.random_symmetric_normal_f32(n, seed)
    e, x, t = q.solve(Q)
    want = O.solve(Q)
    U = O.fold_f32(Q)
    assert O.eval64(U, x) == e
    assert abs(e - want[0]) <= fp32_tol(Q)
    assert (x == want[1]).all() and t == want[2]


def test_fp32_degenerate_inputs(q):
    e, x, t = q.solve(np.zeros((10, 10), np.float32))
    assert e == 0.0 and t == 1024 and not x.any()
    d = np.array([0.5, -1.25, 0.0, -3.0, 2.0, -0.125], np.float32)
    e, x, t = q.solve(np.diag(d))
    assert e == float(np.minimum(d, 0).astype(np.float64).sum()) and t == 2 and (x == (d < 0)).all()
    tiny = (qi.random_symmetric_normal_f32(9, 3) * np.float32(1e-30)).astype(np.float32)
    e, x, t = q.solve(tiny)
    want = O.solve(tiny)
    assert e == want[0] and (x == want[1]).all()


def test_fp32_nonfinite_rejected(q):
    Q = qi.random_symmetric_normal_f32(6, 1)
    Q[2, 3] = np.nan
    with pytest.raises(q.QuboError) as ei:
        q.solve(Q)
    assert ei.value.status == -3
    Q[2, 3] = np.inf
    with pytest.raises(q.QuboError):
        q.solve(Q)


def test_n36_fp32_config_on_slices(q):
    Q = qi.workload_n36_f32()
    e, x, t = q.solve(Q)
    U = O.fold_f32(Q)
    assert O.eval64(U, x) == e
    k = 14
    sid = oracle.rank_of_bits(x[:k])
    want = O.solve_slice(Q, k, sid)
    assert abs(want[0] - e) <= fp32_tol(Q) and (want[1] == x).all()
    ids = qi.Stream(3636).integers(0, (1 << k) - 1, 4).astype(np.uint64)
    es, xs, ts = q.solve_slices(Q, k, ids)
    for s, sid2 in enumerate(ids):
        w2 = O.solve_slice(Q, k, int(sid2))
        assert abs(es[s] - w2[0]) <= fp32_tol(Q) and (xs[s] == w2[1]).all()
        assert w2[0] >= e - fp32_tol(Q)


# ---------------------------------------------------------------- errors and edges

def test_int32_range_error(q):
    Q = np.full((8, 8), 1 << 26, np.int32)
    with pytest.raises(q.QuboError) as ei:
        q.solve(Q)
    assert ei.value.status == -2


def test_range_limit_is_exact(q):
    # sum |U| = 2^30 - 1 passes, one more fails
    n = 4
    Q = np.zeros((n, n), np.int32)
    Q[0, 0] = -((1 << 30) - 1)
    e, x, t = q.solve(Q)
    assert e == -((1 << 30) - 1) and x[0] == 1 and t == 1 << (n - 1)
    Q[1, 1] = 1
    with pytest.raises(q.QuboError):
        q.solve(Q)


def test_slices_argument_checks(q):
    Q = qi.random_upper_int(20, -9, 9, 1)
    with pytest.raises(q.QuboError):
        q.solve_slices(Q, 4, [16])  # id out of range
    with pytest.raises(q.QuboError):
        q.solve_slices(Q, 0, [0])


# ---------------------------------------------------------------- batched

def test_batched_against_oracle(q):
    Qs = qi.batched_upper_int(64, 24, -50, 50, 99)
    e, x, t = q.solve_batched(Qs)
    for b in range(0, 64, 4):
        want = O.solve(Qs[b])
        assert (int(e[b]), int(t[b])) == (want[0], want[2]) and (x[b] == want[1]).all()
    for b in range(64):
        assert O.energy_i64(O.fold_i32(Qs[b]), x[b]) == e[b] and t[b] >= 1


def test_batched_ties_and_other_sizes(q):
    Qs = np.stack([qi.random_upper_int(20, -1, 1, s) for s in range(6)] + [np.zeros((20, 20), np.int32)])
    e, x, t = q.solve_batched(Qs)
    for b in range(Qs.shape[0]):
        want = O.solve(Qs[b])
        assert (int(e[b]), int(t[b])) == (want[0], want[2]) and (x[b] == want[1]).all()
    Qs = qi.batched_upper_int(5, 9, -20, 20, 5)  # below the block kernel's size: per-instance path
    e, x, t = q.solve_batched(Qs)
    for b in range(5):
        want = O.solve(Qs[b])
        assert (int(e[b]), int(t[b])) == (want[0], want[2]) and (x[b] == want[1]).all()


@pytest.mark.parametrize("bounds", [True, False])
def test_batched_mixed_passes_against_oracle(q, bounds):
    # one batch whose instances take the packed (with and without block bounds), biased and int32
    # minimum passes, plus all-ties and many-ties instances
    n = 24
    Qs = np.stack([qi.random_upper_int(n, -20, 20, 510), qi.random_upper_int(n, -1000, 1000, 511),
                   qi.random_upper_int(n, -(1 << 20), 1 << 20, 512), np.zeros((n, n), np.int32),
                   qi.random_upper_int(n, -1, 1, 513), qi.random_upper_int(n, -30, 30, 514),
                   qi.random_upper_int(n, -5000, 5000, 515)])
    sums = np.abs(Qs.astype(np.int64)).sum(axis=(1, 2))
    assert sums[0] <= (1 << 14) - 1 < sums[1] <= (1 << 22) - 1 < sums[2]
    q.enable_block_bounds(bounds)
    try:
        e, x, t = q.solve_batched(Qs)
    finally:
        q.enable_block_bounds(True)
    for b in range(Qs.shape[0]):
        want = O.solve(Qs[b])
        assert (int(e[b]), int(t[b])) == (want[0], want[2]) and (x[b] == want[1]).all(), b


@pytest.mark.parametrize("bounds", [True, False])
def test_batched_packed_ties_across_steps_halves_and_columns(q, bounds):
    # n = 24 instances of the packed pass (12 cached bits, 1 prefix bit, 11 walked bits) with
    # variables whose couplings are all zero: each doubles the minimum's multiplicity, and the
    # tied states then differ in a register-row bit (x_7..x_11 in the minimum pass, x_8..x_11 in
    # the re-walk), a shared row flipped mid-iteration (x_6, or x_7 in the re-walk), a row
    # flipped between iterations (x_1..x_5), a cached bit (x_12..x_23) or the prefix bit (x_0)
    n = 24
    free_sets = [(1, 6, 9, 20), (4, 11), (7,), (0, 3, 5, 8, 10, 12, 23), ()]
    Qs = []
    for k, free in enumerate(free_sets):
        Q = qi.random_upper_int(n, -20, 20, 540 + k)
        for v in free:
            Q[v, :] = 0
            Q[:, v] = 0
        Qs.append(Q)
    Qs = np.stack(Qs)
    assert np.abs(Qs.astype(np.int64)).sum(axis=(1, 2)).max() <= (1 << 14) - 1
    q.enable_block_bounds(bounds)
    try:
        e, x, t = q.solve_batched(Qs)
    finally:
        q.enable_block_bounds(True)
    for b, free in enumerate(free_sets):
        want = O.solve(Qs[b])
        assert (int(e[b]), int(t[b])) == (want[0], want[2]) and (x[b] == want[1]).all(), b
        assert want[2] % (1 << len(free)) == 0


@pytest.mark.parametrize("n,batch", [(18, 40), (21, 12), (28, 2)])
def test_batched_sizes_and_unit_splits(q, n, batch):
    # n = 18, 21: one unit per instance; n = 28: 2^5 units per instance
    Qs = qi.batched_upper_int(batch, n, -60, 60, 520 + n)
    e, x, t = q.solve_batched(Qs)
    for b in range(batch):
        want = O.solve(Qs[b])
        assert (int(e[b]), int(t[b])) == (want[0], want[2]) and (x[b] == want[1]).all()


def test_batched_device_reports_per_instance_status(q):
    import torch
    n, batch = 20, 3
    Qs = qi.batched_upper_int(batch, n, -50, 50, 530)
    Qs[1, 0, 0] = (1 << 30)  # beyond the int32 range: only this instance fails
    dq = torch.from_numpy(Qs).cuda()
    nb = q.batched_workspace_bytes(batch, n)
    ws = torch.empty(max(nb, 256), dtype=torch.uint8, device="cuda")
    res = torch.zeros(batch * 32, dtype=torch.uint8, device="cuda")
    q.solve_batched_device(batch, n, dq, ws, nb, torch.cuda.current_stream().cuda_stream, res)
    torch.cuda.synchronize()
    r = np.frombuffer(res.cpu().numpy().tobytes(), dtype=q.RESULT_DTYPE)
    assert list(r["status"]) == [0, -2, 0]
    for b in (0, 2):
        want = O.solve(Qs[b])
        assert (int(r["min_energy"][b]), int(r["tie_count"][b]), int(r["argmin_rank"][b])) == \
            (want[0], want[2], oracle.rank_of_bits(want[1]))
    with pytest.raises(q.QuboError) as ei:
        q.solve_batched(Qs)
    assert ei.value.status == -2


# ---------------------------------------------------------------- device-resident entry point

def test_device_entry_point(q):
    import torch
    Q = qi.random_upper_int(28, -500, 500, 12)
    n = 28
    dq = torch.from_numpy(Q).cuda()
    nbytes = q.workspace_bytes(n)
    ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    res = torch.zeros(32, dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream()
    q.solve_device(n, dq, q.INT32, ws, nbytes, stream.cuda_stream, res)
    torch.cuda.synchronize()
    r = np.frombuffer(res.cpu().numpy().tobytes(), dtype=q.RESULT_DTYPE)[0]
    want = O.solve(Q)
    assert r["status"] == 0
    assert (int(r["min_energy"]), int(r["tie_count"])) == (want[0], want[2])
    assert int(r["argmin_rank"]) == oracle.rank_of_bits(want[1])
    assert q.last_launch_count() >= 5


def test_single_slice_and_single_range_use_their_own_prefix(q):
    Q = qi.random_upper_int(24, -200, 200, 31)
    for sid in (0, 5, 63):
        e, x, t = q.solve_slices(Q, 6, [sid])
        want = O.solve_slice(Q, 6, sid)
        assert (int(e[0]), int(t[0])) == (want[0], want[2]) and (x[0] == want[1]).all()
        e1, x1, t1 = q.solve_slice_range(Q, 6, sid, 1)
        assert (e1, t1) == (want[0], want[2]) and (x1 == want[1]).all()
