"""The block-bounded minimum passes against the oracle where the bound is tightest.

The biased (fp32-binade) and int32 minimum passes skip the per-step minima of a block of 2^6 or
2^7 Gray steps when a lower bound of every state in it lies above the group's best energy found
so far (the states are still added, eq. 9). A block holding a state at the minimum (or inside the fp32
band) always has its bound at or below the threshold, so it is walked exactly. These cases put
minimisers in many work units and many blocks at once: the results must still be bit-exact.
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


def with_free_prefix(Q_sub, free: int):
    """Q over free + m variables: the first `free` variables have no coupling and no diagonal, so
    every minimiser of Q_sub appears once for each of their 2^free assignments."""
    m = Q_sub.shape[0]
    Q = np.zeros((free + m, free + m), dtype=Q_sub.dtype)
    Q[free:, free:] = Q_sub
    return Q


def test_plans_use_the_bounded_passes(q):
    assert q.plan(40)["pruned"] == 1 and q.plan(32)["pruned"] == 1
    assert q.plan(36, q.FP32)["pruned"] == 1
    assert q.plan(8)["pruned"] == 0  # generic kernel


@pytest.mark.parametrize("lo,hi,seed", [(-1000, 1000, 901), (-(1 << 17), 1 << 17, 902), (-2, 2, 903)])
def test_minimisers_repeated_in_every_unit(q, lo, hi, seed):
    # 2^7 copies of the 27-variable landscape: one minimiser set per assignment of x_0..x_6, in
    # many units; bounded biased pass (entries to 1000), packed pass (narrow ones) and int32 pass
    # (entries to 2^17), all with block bounds
    sub = qi.random_upper_int(27, lo, hi, seed)
    e, x, t = O.solve(sub)
    Q = with_free_prefix(sub, 7)
    ge, gx, gt = q.solve(Q)
    assert (ge, gt) == (e, t << 7)
    assert not gx[:7].any() and (gx[7:] == x).all()


def test_minimisers_repeated_fp32(q):
    sub = qi.random_symmetric_normal_f32(26, 904)
    e, x, t = O.solve(sub)
    Q = with_free_prefix(sub, 6)
    ge, gx, gt = q.solve(Q)
    tol = 1e-3 * float(np.abs(Q.astype(np.float64)).sum()) * 2.0 ** -20
    assert abs(ge - e) <= tol and gt == t << 6
    assert not gx[:6].any() and (gx[6:] == x).all()


def test_many_near_minimum_states(q):
    # entries in {-1, 0, 1}: huge numbers of states within a few units of the minimum, so many
    # blocks are walked exactly and the threshold meets the bounds often
    Q = qi.random_upper_int(32, -1, 1, 905)
    want = O.solve(Q)
    e, x, t = q.solve(Q)
    assert (e, t) == (want[0], want[2]) and (x == want[1]).all()


def test_small_units_and_explicit_splits(q):
    # many small units (most of them report only an upper bound of their minimum)
    Q = qi.random_upper_int(31, -1000, 1000, 906)
    want = O.solve(Q)
    for k, c in ((14, 12), (10, 9), (16, 10)):
        e, x, t = q.solve(Q, k_prefix=k, cache_bits=c)
        assert (e, t) == (want[0], want[2]) and (x == want[1]).all(), (k, c)


def test_slices_keep_their_own_thresholds(q):
    # slices whose minima differ by a lot: each group's threshold must come from its own units
    n, k = 30, 3
    Q = qi.random_upper_int(n, -500, 500, 907)
    Q[0, 0] = -200000  # slices with x_0 = 1 lie far below those with x_0 = 0
    ids = np.arange(1 << k, dtype=np.uint64)
    e, x, t = q.solve_slices(Q, k, ids)
    for s in range(1 << k):
        want = O.solve_slice(Q, k, s)
        assert (int(e[s]), int(t[s])) == (want[0], want[2]) and (x[s] == want[1]).all(), s


def test_slice_range_starting_above_zero(q):
    # a range that does not hold the zero state: no threshold below its own minimum is used
    n, k = 30, 4
    Q = qi.random_upper_int(n, 0, 9, 908)  # non-negative: every minimum is 0 ... except the range's
    Q[np.diag_indices(n)] += 1               # all diagonals >= 1: E(x) > 0 for every x != 0
    e, x, t = q.solve_slice_range(Q, k, 5, 7)
    recs = [O.solve_slice(Q, k, s) for s in range(5, 12)]
    best = min(r[0] for r in recs)
    ties = sum(r[2] for r in recs if r[0] == best)
    first = min(oracle.rank_of_bits(r[1]) for r in recs if r[0] == best)
    assert (e, t, oracle.rank_of_bits(x)) == (best, ties, first) and best > 0


@pytest.mark.parametrize("d", [1e-9, 3e-7])
def test_fp32_near_ties_inside_the_band(q, d):
    # Three decoupled variables around a 27-variable fp32 landscape: x_0 with diagonal +d (in the
    # prefix: another work unit), x_15 with diagonal 0 and x_29 with -d (cached: the same unit).
    # In the fixed-point image the +-d round to 0, so the states x*, x* + e_0 and x* + e_29 tie
    # inside the band; the fp64 re-evaluation decides: x_0 = 0, x_29 = 1, and x_15 either way
    # (an exact fp64 tie: twice the landscape's minimisers, the lower rank has x_15 = 0).
    sub = qi.random_symmetric_normal_f32(27, 909)
    e, x, t = O.solve(sub)
    n = 30
    rest = [i for i in range(n) if i not in (0, 15, 29)]
    Q = np.zeros((n, n), np.float32)
    Q[np.ix_(rest, rest)] = sub
    Q[0, 0], Q[29, 29] = np.float32(d), np.float32(-d)
    assert q.plan(n, q.FP32)["pruned"] == 1
    ge, gx, gt = q.solve(Q)
    tol = 1e-3 * float(np.abs(Q.astype(np.float64)).sum()) * 2.0 ** -20
    want = np.zeros(n, np.uint8)
    want[rest] = x
    want[29] = 1
    assert (gx == want).all() and gt == 2 * t
    U = O.fold_f32(Q)
    assert ge == O.eval64(U, gx) and abs(ge - (e - float(np.float32(d)))) <= tol
    # the states one flip away in x_0 or x_29 lie inside the fp32 band but above in fp64
    for v in (0, 29):
        y = gx.copy()
        y[v] ^= 1
        assert O.eval64(U, y) > ge


@pytest.mark.parametrize("sign", ["mixed", "negative", "positive"])
def test_int32_bounded_pass_at_the_range_limit(q, sign):
    # sum |U| = 2^30 - 1, the largest int32 input: running values reach +-S, the bound with the
    # walked energy and D_par reaches -3S (formed in 64 bits); all-negative entries give
    # E = -S at x = 1, all-positive ones the zero state alone
    n = 30
    lo, hi = {"mixed": (-(1 << 21), 1 << 21), "negative": (-(1 << 21), -1), "positive": (1, 1 << 21)}[sign]
    total = (1 << 30) - 1
    Q = np.triu(qi.random_upper_int(n, lo, hi, 910)).astype(np.int64)
    Q[0, 0] = 0
    rest = int(np.abs(Q).sum())
    assert rest < total
    Q[0, 0] = (total - rest) if sign == "positive" else -(total - rest)
    Q = Q.astype(np.int32)
    assert int(np.abs(Q.astype(np.int64)).sum()) == total
    assert q.plan(n)["pruned"] == 1
    want = O.solve(Q)
    e, x, t = q.solve(Q)
    assert (e, t) == (want[0], want[2]) and (x == want[1]).all()
    if sign == "negative":
        assert e == -total and x.all()
    if sign == "positive":
        assert e == 0 and t == 1 and not x.any()


def test_int32_bounded_pass_ties_in_many_units(q):
    # wide entries, 2^6 copies of every minimiser (free prefix variables), and slices of it
    sub = qi.random_upper_int(26, -(1 << 19), 1 << 19, 911)
    e, x, t = O.solve(sub)
    Q = with_free_prefix(sub, 6)
    assert int(np.abs(Q.astype(np.int64)).sum()) >= 1 << 22
    ge, gx, gt = q.solve(Q)
    assert (ge, gt) == (e, t << 6) and not gx[:6].any() and (gx[6:] == x).all()
    ids = np.array([0, 5, 63], dtype=np.uint64)
    se, sx, st = q.solve_slices(Q, 6, ids)
    for i, sid in enumerate(ids):
        assert (int(se[i]), int(st[i])) == (e, t)
        assert (sx[i][6:] == x).all() and oracle.rank_of_bits(sx[i][:6]) == int(sid)


@pytest.mark.parametrize("first,count", [(0, 8), (8, 8), (3, 1)])
def test_slice_ranges_seed_inside_their_range(q, first, count):
    # x_0 = 1 lowers every energy by 200000, so every state of slices 8..15 (k = 4) lies below
    # every state of slices 0..7: a starting best taken from outside the range would be below
    # the range's minimum. Each range's answer must be its own.
    n, k = 31, 4
    Q = qi.random_upper_int(n, -500, 500, 912)
    Q[0, 0] = -200000
    e, x, t = q.solve_slice_range(Q, k, first, count)
    recs = [O.solve_slice(Q, k, s) for s in range(first, first + count)]
    best = min(r[0] for r in recs)
    ties = sum(r[2] for r in recs if r[0] == best)
    rank = min(oracle.rank_of_bits(r[1]) for r in recs if r[0] == best)
    assert (e, t, oracle.rank_of_bits(x)) == (best, ties, rank)


@pytest.mark.parametrize("first,count", [(0, 8), (8, 8)])
def test_device_slice_ranges_seed_inside_their_range(q, first, count):
    # the device entry of the sharded search (one range per rank): the same instance, a range
    # from slice 0 that is not the whole problem, and one above it
    torch = pytest.importorskip("torch")
    n, k = 31, 4
    Q = qi.random_upper_int(n, -500, 500, 912)
    Q[0, 0] = -200000
    dq = torch.from_numpy(Q).cuda()
    nb = max(q.slice_range_workspace_bytes(n, q.INT32, k, count), 256)
    ws = torch.empty(nb, dtype=torch.uint8, device="cuda")
    res = torch.zeros(32, dtype=torch.uint8, device="cuda")
    s = torch.cuda.current_stream()
    q.solve_slice_range_device(n, dq, q.INT32, k, first, count, ws, nb, s.cuda_stream, res)
    torch.cuda.synchronize()
    r = np.frombuffer(res.cpu().numpy().tobytes(), dtype=q.RESULT_DTYPE)[0]
    recs = [O.solve_slice(Q, k, s_) for s_ in range(first, first + count)]
    best = min(rr[0] for rr in recs)
    ties = sum(rr[2] for rr in recs if rr[0] == best)
    rank = min(oracle.rank_of_bits(rr[1]) for rr in recs if rr[0] == best)
    assert (int(r["status"]), float(r["min_energy"]), int(r["tie_count"]), int(r["argmin_rank"])) == (0, best, ties, rank)
