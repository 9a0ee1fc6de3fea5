"""Host-side Ising -> QUBO conversion of the library (qubo_ising_to_qubo; no GPU needed), against
the oracle's direct evaluation of the Ising energy H(s) = sum_ij J_ij s_i s_j + sum_i h_i s_i."""
import itertools

import numpy as np
import pytest

import oracle
import qubo_instances as qi

O = oracle.get()


@pytest.fixture(scope="module")
def q():
    import exact_qubo_exhaustive_gb300 as lib
    return lib


def ising_at(J, h, x):
    """H at one state via the oracle (a one-state direct search)."""
    n = len(x)
    r = int("".join(str(int(b)) for b in x), 2)
    if J.dtype.kind == "f":
        import ctypes
        Jd = np.ascontiguousarray(J, np.float64)
        hd = None if h is None else np.ascontiguousarray(h, np.float64)
        e, a, t = ctypes.c_double(), ctypes.c_uint64(), ctypes.c_uint64()
        O.lib.oracle_ising_direct_f64(n, Jd.ctypes.data, None if hd is None else hd.ctypes.data, r, r + 1,
                                      ctypes.byref(e), ctypes.byref(a), ctypes.byref(t))
        return e.value
    import ctypes
    Jd = np.ascontiguousarray(J, np.int64)
    hd = None if h is None else np.ascontiguousarray(h, np.int64)
    e, a, t = ctypes.c_int64(), ctypes.c_uint64(), ctypes.c_uint64()
    O.lib.oracle_ising_direct_i64(n, Jd.ctypes.data, None if hd is None else hd.ctypes.data, r, r + 1,
                                  ctypes.byref(e), ctypes.byref(a), ctypes.byref(t))
    return e.value


@pytest.mark.parametrize("seed", [1, 2])
def test_int_conversion_is_exact_on_every_state(q, seed):
    st = qi.Stream(800 + seed)
    n = 8
    J = st.integers(-50, 50, n * n).reshape(n, n).astype(np.int32)  # full matrix incl. diagonal
    h = st.integers(-50, 50, n).astype(np.int32)
    Q, off = q.ising_to_qubo(J, h)
    assert Q.dtype == np.int32 and not np.tril(Q, -1).any()
    for x in itertools.product((0, 1), repeat=n):
        x = np.array(x, np.uint8)
        assert O.energy_raw_i32(Q, x) + off == ising_at(J, h, x)


def test_fp_conversion_matches_on_every_state(q):
    st = qi.Stream(803)
    n = 8
    J = st.normals(n * n).reshape(n, n).astype(np.float32)
    h = st.normals(n).astype(np.float32)
    Q, off = q.ising_to_qubo(J, h)
    assert Q.dtype == np.float64
    scale = float(np.abs(J.astype(np.float64)).sum() + np.abs(h.astype(np.float64)).sum())
    U = O.fold_f64(Q)
    for x in itertools.product((0, 1), repeat=n):
        x = np.array(x, np.uint8)
        assert abs(O.eval64(U, x) + off - ising_at(J.astype(np.float64), h.astype(np.float64), x)) <= 1e-12 * scale


def test_mattis_conversion_matches_the_generator(q):
    s_star, w, J = qi.mattis_couplings(12, 1, 100, 9)
    Q, off = q.ising_to_qubo(J.astype(np.int32))
    Qg, offg = qi.ising_to_qubo(J, np.zeros(12, np.int64))  # independent restatement
    assert (Q == Qg).all() and off == offg


def test_conversion_errors(q):
    big = np.zeros((3, 3), np.int32)
    big[0, 1] = 1 << 30  # 4 * (J_01 + J_10) leaves int32
    with pytest.raises(q.QuboError) as ei:
        q.ising_to_qubo(big)
    assert ei.value.status == -2
    bad = np.zeros((3, 3), np.float32)
    bad[1, 2] = np.nan
    with pytest.raises(q.QuboError) as ei:
        q.ising_to_qubo(bad)
    assert ei.value.status == -3
    with pytest.raises(ValueError):
        q.ising_to_qubo(np.zeros((3, 3), np.int32), np.zeros(4, np.int32))
