"""GPU parity of the Ising entry point and of fp64 QUBO input (through the C ABI) against the
oracle: the Ising oracle evaluates H(s) from its definition, with no QUBO conversion."""
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


@pytest.mark.parametrize("n,seed", [(3, 1), (11, 2), (17, 3), (21, 4)])
def test_ising_int_against_oracle(q, n, seed):
    st = qi.Stream(900 + seed)
    J = st.integers(-40, 40, n * n).reshape(n, n).astype(np.int32)
    h = st.integers(-40, 40, n).astype(np.int32)
    H, s, t = q.solve_ising(J, h)
    wH, ws, wt = O.ising_direct(J, h)
    assert (H, t) == (wH, wt) and (s == ws).all()


@pytest.mark.parametrize("n,seed", [(16, 5), (22, 6)])
def test_ising_mattis_planted(q, n, seed):
    s_star, w, J = qi.mattis_couplings(n, 1, 100, seed)
    H, s, t = q.solve_ising(J.astype(np.int32))
    assert H == -int(np.triu(w, 1).sum()) and t == 2
    assert (s == (s_star if s_star[0] == -1 else -s_star)).all()


def test_ising_zero_field_default_and_ties(q):
    # J = 0, h = 0: every one of the 2^10 spin states is a ground state, H = 0, s = all -1
    H, s, t = q.solve_ising(np.zeros((10, 10), np.int32))
    assert (H, t) == (0, 1 << 10) and (s == -1).all()


@pytest.mark.parametrize("dt", [np.float32, np.float64])
def test_ising_fp_against_oracle(q, dt):
    st = qi.Stream(950)
    n = 18
    J = st.normals(n * n).reshape(n, n).astype(dt)
    h = st.normals(n).astype(dt)
    H, s, t = q.solve_ising(J, h)
    wH, ws, wt = O.ising_direct(J.astype(np.float64), h.astype(np.float64))
    Q, off = q.ising_to_qubo(J, h)
    tol = 1e-3 * float(np.abs(O.fold_f64(Q)).sum()) * 2.0 ** -20
    assert abs(H - wH) <= tol
    x = ((s + 1) // 2).astype(np.uint8)
    r = int("".join(str(int(b)) for b in x), 2)
    import ctypes
    Jd = np.ascontiguousarray(J, np.float64)  # kept alive across the call
    hd = np.ascontiguousarray(h, np.float64)
    e, a, c = ctypes.c_double(), ctypes.c_uint64(), ctypes.c_uint64()
    O.lib.oracle_ising_direct_f64(n, Jd.ctypes.data, hd.ctypes.data, r, r + 1,
                                  ctypes.byref(e), ctypes.byref(a), ctypes.byref(c))
    assert abs(e.value - H) <= tol  # the returned spins reach the returned energy


@pytest.mark.parametrize("n,seed", [(7, 1), (19, 2), (25, 3)])
def test_fp64_qubo_input_against_oracle(q, n, seed):
    Q = qi.random_symmetric_normal_f32(n, 960 + seed).astype(np.float64) * 3.0 + 1e-9
    e, x, t = q.solve(Q)
    want = O.solve(Q)
    U = O.fold_f64(Q)
    assert O.eval64(U, x) == e
    assert abs(e - want[0]) <= 1e-3 * float(np.abs(U).sum()) * 2.0 ** -20
    assert (x == want[1]).all() and t == want[2]
