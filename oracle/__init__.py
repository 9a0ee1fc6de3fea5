"""CPU oracle for exhaustive QUBO minimisation -- TEST INFRASTRUCTURE ONLY.

Only tests/, __graft_entry__.smoke() and bench.py's cpu_baseline / reference leg may import
this package. The product (exact_qubo_exhaustive_gb300) never imports it and shares no code
with it. The arithmetic lives in qubo_oracle.c (plain C, OpenMP over slices); this module
only compiles it with gcc and marshals arguments.

Definitions followed (Terastate-per-second QUBO Brute-Force on a Single GPU, §I objective and
§II-B lexicographic state order):
  E(x) = sum_{i,j} Q_ij x_i x_j,  x in {0,1}^n, rank(x) = sum_i x_i 2^(n-1-i)
  result = (E_min, lowest-rank argmin, number of states with E = E_min)
For fp32 Q the energy is the fixed-order fp64 sum (eval64) of the fp64-folded triangle.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "qubo_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_lock = threading.Lock()
_libs: dict[int, ctypes.CDLL] = {}

_i64p = ctypes.POINTER(ctypes.c_int64)
_u64p = ctypes.POINTER(ctypes.c_uint64)
_f64p = ctypes.POINTER(ctypes.c_double)


def lib_path(mutant: int = 0) -> str:
    name = "liboracle.so" if mutant == 0 else f"liboracle_mutant{mutant}.so"
    return os.path.join(_BUILD, name)


def build(mutant: int = 0, force: bool = False) -> str:
    """Compile qubo_oracle.c with gcc (-O2, OpenMP, no FP contraction). Returns the .so path."""
    out = lib_path(mutant)
    os.makedirs(_BUILD, exist_ok=True)
    if not force and os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(_SRC):
        return out
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off",
           f"-DORACLE_MUTANT={mutant}", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def _load(mutant: int = 0) -> ctypes.CDLL:
    with _lock:
        if mutant in _libs:
            return _libs[mutant]
        lib = ctypes.CDLL(build(mutant))
        lib.oracle_gray_code.restype = ctypes.c_uint64
        lib.oracle_gray_code.argtypes = [ctypes.c_uint64]
        lib.oracle_gray_flip_bit.restype = ctypes.c_int
        lib.oracle_gray_flip_bit.argtypes = [ctypes.c_uint64]
        lib.oracle_num_threads.restype = ctypes.c_int
        lib.oracle_fold_i32.argtypes = [ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p]
        lib.oracle_fold_f32.argtypes = [ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p]
        lib.oracle_fold_f64.argtypes = [ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p]
        lib.oracle_set_threads.argtypes = [ctypes.c_int]
        lib.oracle_lowest_i64.restype = ctypes.c_int
        lib.oracle_lowest_i64.argtypes = [ctypes.c_int, ctypes.c_void_p, ctypes.c_int, ctypes.c_uint64, ctypes.c_uint64,
                                          ctypes.c_void_p, ctypes.c_void_p]
        lib.oracle_ising_direct_i64.argtypes = [ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_uint64,
                                                ctypes.c_uint64, _i64p, _u64p, _u64p]
        lib.oracle_ising_direct_f64.argtypes = [ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_uint64,
                                                ctypes.c_uint64, _f64p, _u64p, _u64p]
        lib.oracle_energy_i64.restype = ctypes.c_int64
        lib.oracle_energy_i64.argtypes = [ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p]
        lib.oracle_eval64.restype = ctypes.c_double
        lib.oracle_eval64.argtypes = [ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p]
        lib.oracle_energy_raw_i32.restype = ctypes.c_int64
        lib.oracle_energy_raw_i32.argtypes = [ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p]
        lib.oracle_direct_i64.argtypes = [ctypes.c_int, ctypes.c_void_p, ctypes.c_uint64, ctypes.c_uint64,
                                          _i64p, _u64p, _u64p]
        lib.oracle_gray_i64.argtypes = [ctypes.c_int, ctypes.c_void_p, ctypes.c_int, ctypes.c_uint64,
                                        _i64p, _u64p, _u64p]
        lib.oracle_gray_trace_i64.argtypes = [ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]
        lib.oracle_gray_f64.argtypes = [ctypes.c_int, ctypes.c_void_p, ctypes.c_int, ctypes.c_uint64,
                                        _f64p, _u64p, _u64p]
        lib.oracle_direct_f64.argtypes = [ctypes.c_int, ctypes.c_void_p, ctypes.c_uint64, ctypes.c_uint64,
                                          _f64p, _u64p, _u64p]
        lib.oracle_walk_bound_f64.restype = ctypes.c_double
        lib.oracle_walk_bound_f64.argtypes = [ctypes.c_int, ctypes.c_void_p, ctypes.c_int]
        lib.oracle_subproblem_i64.restype = ctypes.c_int64
        lib.oracle_subproblem_i64.argtypes = [ctypes.c_int, ctypes.c_void_p, ctypes.c_int, ctypes.c_uint64,
                                              ctypes.c_void_p]
        _libs[mutant] = lib
        return lib


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


class Oracle:
    """Bound oracle functions (mutant != 0 loads a build with one step broken on purpose)."""

    def __init__(self, mutant: int = 0):
        self.lib = _load(mutant)

    # -- helpers
    def gray_code(self, i: int) -> int:
        return int(self.lib.oracle_gray_code(i))

    def gray_flip_bit(self, i: int) -> int:
        return int(self.lib.oracle_gray_flip_bit(i))

    def num_threads(self) -> int:
        return int(self.lib.oracle_num_threads())

    def set_threads(self, t: int) -> None:
        self.lib.oracle_set_threads(int(t))

    # -- folding and energies
    def fold_i32(self, Q) -> np.ndarray:
        Q = np.ascontiguousarray(Q, dtype=np.int32)
        n = Q.shape[0]
        U = np.zeros((n, n), dtype=np.int64)
        self.lib.oracle_fold_i32(n, _ptr(Q), _ptr(U))
        return U

    def fold_f32(self, Q) -> np.ndarray:
        Q = np.ascontiguousarray(Q, dtype=np.float32)
        n = Q.shape[0]
        U = np.zeros((n, n), dtype=np.float64)
        self.lib.oracle_fold_f32(n, _ptr(Q), _ptr(U))
        return U

    def fold_f64(self, Q) -> np.ndarray:
        Q = np.ascontiguousarray(Q, dtype=np.float64)
        n = Q.shape[0]
        U = np.zeros((n, n), dtype=np.float64)
        self.lib.oracle_fold_f64(n, _ptr(Q), _ptr(U))
        return U

    def energy_i64(self, U, x) -> int:
        U = np.ascontiguousarray(U, dtype=np.int64)
        x = np.ascontiguousarray(x, dtype=np.uint8)
        return int(self.lib.oracle_energy_i64(U.shape[0], _ptr(U), _ptr(x)))

    def eval64(self, U, x) -> float:
        U = np.ascontiguousarray(U, dtype=np.float64)
        x = np.ascontiguousarray(x, dtype=np.uint8)
        return float(self.lib.oracle_eval64(U.shape[0], _ptr(U), _ptr(x)))

    def energy_raw_i32(self, Q, x) -> int:
        Q = np.ascontiguousarray(Q, dtype=np.int32)
        x = np.ascontiguousarray(x, dtype=np.uint8)
        return int(self.lib.oracle_energy_raw_i32(Q.shape[0], _ptr(Q), _ptr(x)))

    # -- searches on folded matrices
    def direct_i64(self, U, lo: int = 0, hi: int | None = None):
        U = np.ascontiguousarray(U, dtype=np.int64)
        n = U.shape[0]
        hi = (1 << n) if hi is None else hi
        e, r, t = ctypes.c_int64(), ctypes.c_uint64(), ctypes.c_uint64()
        self.lib.oracle_direct_i64(n, _ptr(U), lo, hi, ctypes.byref(e), ctypes.byref(r), ctypes.byref(t))
        return int(e.value), int(r.value), int(t.value)

    def lowest(self, Q, k: int, lo: int = 0, hi: int | None = None):
        """The k smallest keys (E, rank) of the int32 matrix Q among ranks [lo, hi), ascending:
        (energies int64[m], states uint8[m, n])."""
        U = self.fold_i32(Q)
        n = U.shape[0]
        hi = (1 << n) if hi is None else hi
        e = np.zeros(k, np.int64)
        r = np.zeros(k, np.uint64)
        m = self.lib.oracle_lowest_i64(n, _ptr(U), k, lo, hi, _ptr(e), _ptr(r))
        return e[:m], np.array([bits_of_rank(n, int(v)) for v in r[:m]], dtype=np.uint8).reshape(m, n)

    def ising_direct(self, J, h=None):
        """Ising ground state by direct evaluation of H(s) = sum_ij J_ij s_i s_j + sum_i h_i s_i over
        all 2^n spin states: (H_min, spins of the lowest-rank ground state as int8, ground states)."""
        J = np.asarray(J)
        n = J.shape[0]
        if J.dtype.kind == "f":
            Jd = np.ascontiguousarray(J, dtype=np.float64)
            hd = None if h is None else np.ascontiguousarray(h, dtype=np.float64)
            e, r, t = ctypes.c_double(), ctypes.c_uint64(), ctypes.c_uint64()
            self.lib.oracle_ising_direct_f64(n, _ptr(Jd), None if hd is None else _ptr(hd), 0, 1 << n,
                                             ctypes.byref(e), ctypes.byref(r), ctypes.byref(t))
            H = float(e.value)
        else:
            Jd = np.ascontiguousarray(J, dtype=np.int64)
            hd = None if h is None else np.ascontiguousarray(h, dtype=np.int64)
            e, r, t = ctypes.c_int64(), ctypes.c_uint64(), ctypes.c_uint64()
            self.lib.oracle_ising_direct_i64(n, _ptr(Jd), None if hd is None else _ptr(hd), 0, 1 << n,
                                             ctypes.byref(e), ctypes.byref(r), ctypes.byref(t))
            H = int(e.value)
        s = 2 * bits_of_rank(n, int(r.value)).astype(np.int8) - 1
        return H, s, int(t.value)

    def gray_i64(self, U, k: int = 0, prefix: int = 0):
        U = np.ascontiguousarray(U, dtype=np.int64)
        e, r, t = ctypes.c_int64(), ctypes.c_uint64(), ctypes.c_uint64()
        self.lib.oracle_gray_i64(U.shape[0], _ptr(U), k, prefix, ctypes.byref(e), ctypes.byref(r), ctypes.byref(t))
        return int(e.value), int(r.value), int(t.value)

    def gray_trace_i64(self, U):
        U = np.ascontiguousarray(U, dtype=np.int64)
        n = U.shape[0]
        assert n <= 24
        E = np.zeros(1 << n, dtype=np.int64)
        R = np.zeros(1 << n, dtype=np.uint64)
        self.lib.oracle_gray_trace_i64(n, _ptr(U), _ptr(E), _ptr(R))
        return E, R

    def gray_f64(self, U, k: int = 0, prefix: int = 0):
        U = np.ascontiguousarray(U, dtype=np.float64)
        e, r, t = ctypes.c_double(), ctypes.c_uint64(), ctypes.c_uint64()
        self.lib.oracle_gray_f64(U.shape[0], _ptr(U), k, prefix, ctypes.byref(e), ctypes.byref(r), ctypes.byref(t))
        return float(e.value), int(r.value), int(t.value)

    def direct_f64(self, U, lo: int = 0, hi: int | None = None):
        U = np.ascontiguousarray(U, dtype=np.float64)
        n = U.shape[0]
        hi = (1 << n) if hi is None else hi
        e, r, t = ctypes.c_double(), ctypes.c_uint64(), ctypes.c_uint64()
        self.lib.oracle_direct_f64(n, _ptr(U), lo, hi, ctypes.byref(e), ctypes.byref(r), ctypes.byref(t))
        return float(e.value), int(r.value), int(t.value)

    def walk_bound_f64(self, U, mb: int) -> float:
        U = np.ascontiguousarray(U, dtype=np.float64)
        return float(self.lib.oracle_walk_bound_f64(U.shape[0], _ptr(U), mb))

    def subproblem_i64(self, U, k: int, prefix: int):
        U = np.ascontiguousarray(U, dtype=np.int64)
        n = U.shape[0]
        Qr = np.zeros((n - k, n - k), dtype=np.int64)
        c = self.lib.oracle_subproblem_i64(n, _ptr(U), k, prefix, _ptr(Qr))
        return int(c), Qr

    # -- whole-problem entry points on the raw Q
    def solve(self, Q, method: str = "gray"):
        """(E_min, argmin bits, ties) of the raw matrix Q (int32, fp32 or fp64), whole state space."""
        return self.solve_slice(Q, 0, 0, method)

    def solve_slice(self, Q, k: int, prefix: int, method: str = "gray"):
        """Same, restricted to the states whose first k variables equal `prefix` (MSB first)."""
        Q = np.asarray(Q)
        n = Q.shape[0]
        if Q.dtype in (np.float32, np.float64):
            U = self.fold_f32(Q) if Q.dtype == np.float32 else self.fold_f64(Q)
            if method == "direct":
                e, r, t = self.direct_f64(U, prefix << (n - k), (prefix + 1) << (n - k))
            else:
                e, r, t = self.gray_f64(U, k, prefix)
        else:
            U = self.fold_i32(Q)
            if method == "direct":
                e, r, t = self.direct_i64(U, prefix << (n - k), (prefix + 1) << (n - k))
            else:
                e, r, t = self.gray_i64(U, k, prefix)
        return e, bits_of_rank(n, r), t


def bits_of_rank(n: int, rank: int) -> np.ndarray:
    """x with x_0 as the most significant bit of rank."""
    return np.array([(rank >> (n - 1 - i)) & 1 for i in range(n)], dtype=np.uint8)


def rank_of_bits(x) -> int:
    r = 0
    for b in x:
        r = (r << 1) | int(b)
    return r


_default: Oracle | None = None


def get() -> Oracle:
    global _default
    if _default is None:
        _default = Oracle(0)
    return _default
