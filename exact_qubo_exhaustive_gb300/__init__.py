"""exact_qubo_exhaustive_gb300 -- exhaustive QUBO minimisation on one GB300 (sm_103a).

Thin Python binding of the C ABI in include/qubo.h (argument marshalling only; every step of
the search runs in the CUDA kernels of libqubo_gb300.so). The library must have been built
(`python exact_qubo_exhaustive_gb300/build.py` or __graft_entry__.build()); there is no CPU
fallback, and importing the binding without the library raises ImportError.

    E(x) = sum_{i,j} Q_ij x_i x_j,  x in {0,1}^n   (Terastate-per-second QUBO Brute-Force, §I)

Results are (E_min, argmin x as uint8[n] with x_0 first, number of minimisers); the argmin is
the minimiser of lowest rank (x_0 the most significant bit).
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

__all__ = [
    "QuboError", "INT32", "FP32", "FP64", "RESULT_DTYPE", "library_path",
    # whole problems, slices, ranges, batches
    "solve", "solve_slices", "solve_slice_range", "solve_batched",
    "solve_device", "solve_slice_range_device", "solve_batched_device", "solve_device_no_alloc",
    "workspace_bytes", "slice_range_workspace_bytes", "batched_workspace_bytes", "NO_ALLOC_SCRATCH_BYTES",
    # the k lowest energies, Ising input, long runs
    "solve_lowest", "LOWEST_MAX_K", "solve_ising", "ising_to_qubo",
    "solve_checkpointed", "checkpoint_read", "fnv1a64", "INCOMPLETE",
    # planner, measurement, status, cancellation
    "plan", "probe_alu", "enable_kernel_timing", "enable_block_bounds", "kernel_time_ms", "last_launch_count",
    "status_string", "last_error", "request_abort", "clear_abort", "rank_to_bits",
]

INT32 = 0
FP32 = 1
FP64 = 2

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "libqubo_gb300.so")


def library_path() -> str:
    return _LIB_PATH


if not os.path.exists(_LIB_PATH):
    raise ImportError(f"{_LIB_PATH} is missing: build it with `python exact_qubo_exhaustive_gb300/build.py` "
                      "(the CUDA library is required; there is no CPU path)")

_lib = ctypes.CDLL(_LIB_PATH)

_u8p = ctypes.POINTER(ctypes.c_uint8)
_u64p = ctypes.POINTER(ctypes.c_uint64)
_f64p = ctypes.POINTER(ctypes.c_double)


class _PlanDesc(ctypes.Structure):
    _fields_ = [("n", ctypes.c_int), ("dtype", ctypes.c_int), ("k_prefix", ctypes.c_int),
                ("cache_bits", ctypes.c_int), ("walked_bits", ctypes.c_int), ("register_bits", ctypes.c_int),
                ("columns_per_thread", ctypes.c_int), ("threads_per_block", ctypes.c_int), ("blocks", ctypes.c_int),
                ("variant", ctypes.c_int), ("units", ctypes.c_uint64), ("workspace_bytes", ctypes.c_size_t),
                ("smem_bytes", ctypes.c_size_t), ("packed", ctypes.c_int), ("biased", ctypes.c_int),
                ("pruned", ctypes.c_int)]


# qubo_result record as a numpy dtype (status, reserved, min_energy, argmin_rank, tie_count)
RESULT_DTYPE = np.dtype([("status", np.int32), ("reserved", np.int32), ("min_energy", np.float64),
                         ("argmin_rank", np.uint64), ("tie_count", np.uint64)])

_sig = {
    "qubo_solve": (ctypes.c_int, [ctypes.c_int, ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_int, _f64p,
                                  _u8p, _u64p]),
    "qubo_solve_slices": (ctypes.c_int, [ctypes.c_int, ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                         _u64p, ctypes.c_int, _f64p, _u8p, _u64p]),
    "qubo_solve_slice_range": (ctypes.c_int, [ctypes.c_int, ctypes.c_void_p, ctypes.c_int, ctypes.c_int,
                                              ctypes.c_int, ctypes.c_uint64, ctypes.c_uint64, _f64p, _u8p, _u64p]),
    "qubo_solve_batched": (ctypes.c_int, [ctypes.c_int, ctypes.c_int, ctypes.c_void_p, ctypes.c_int, _f64p, _u8p,
                                          _u64p]),
    "qubo_workspace_bytes": (ctypes.c_size_t, [ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int]),
    "qubo_solve_device": (ctypes.c_int, [ctypes.c_int, ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                         ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p, ctypes.c_void_p]),
    "qubo_batched_workspace_bytes": (ctypes.c_size_t, [ctypes.c_int, ctypes.c_int, ctypes.c_int]),
    "qubo_slice_range_workspace_bytes": (ctypes.c_size_t, [ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                                           ctypes.c_uint64]),
    "qubo_solve_slice_range_device": (ctypes.c_int, [ctypes.c_int, ctypes.c_void_p, ctypes.c_int, ctypes.c_int,
                                                     ctypes.c_int, ctypes.c_uint64, ctypes.c_uint64, ctypes.c_void_p,
                                                     ctypes.c_size_t, ctypes.c_void_p, ctypes.c_void_p]),
    "qubo_solve_device_no_alloc": (ctypes.c_int, [ctypes.c_int, ctypes.c_void_p, ctypes.c_int, ctypes.c_int,
                                                  ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p]),
    "qubo_enable_kernel_timing": (None, [ctypes.c_int]),
    "qubo_kernel_time_ms": (ctypes.c_double, []),
    "qubo_enable_block_bounds": (None, [ctypes.c_int]),
    "qubo_solve_batched_device": (ctypes.c_int, [ctypes.c_int, ctypes.c_int, ctypes.c_void_p, ctypes.c_int,
                                                 ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p,
                                                 ctypes.c_void_p]),
    "qubo_plan": (ctypes.c_int, [ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.POINTER(_PlanDesc)]),
    "qubo_last_launch_count": (ctypes.c_int, []),
    "qubo_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "qubo_last_error": (ctypes.c_char_p, []),
    "qubo_request_abort": (None, []),
    "qubo_clear_abort": (None, []),
    "qubo_probe_alu": (ctypes.c_int, [ctypes.c_int, ctypes.c_int, _f64p, _f64p]),
    "qubo_solve_lowest": (ctypes.c_int, [ctypes.c_int, ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                         ctypes.c_int, _f64p, _u8p, ctypes.POINTER(ctypes.c_int)]),
    "qubo_solve_checkpointed": (ctypes.c_int, [ctypes.c_int, ctypes.c_void_p, ctypes.c_int, ctypes.c_int,
                                               ctypes.c_int, ctypes.c_uint64, ctypes.c_char_p, ctypes.c_double,
                                               _f64p, _u8p, _u64p, _u64p]),
    "qubo_checkpoint_read": (ctypes.c_int, [ctypes.c_char_p, ctypes.POINTER(ctypes.c_int), ctypes.POINTER(ctypes.c_int),
                                            ctypes.POINTER(ctypes.c_int), _u64p, _u64p, _u64p,
                                            ctypes.POINTER(ctypes.c_int), _f64p, _u64p, _u64p]),
    "qubo_fnv1a64": (ctypes.c_uint64, [ctypes.c_void_p, ctypes.c_size_t]),
    "qubo_ising_to_qubo": (ctypes.c_int, [ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int,
                                          ctypes.c_void_p, _f64p]),
    "qubo_solve_ising": (ctypes.c_int, [ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int, ctypes.c_int,
                                        ctypes.c_int, _f64p, ctypes.c_void_p, _u64p]),
}
for _name, (_res, _args) in _sig.items():
    _f = getattr(_lib, _name)
    _f.restype = _res
    _f.argtypes = _args


class QuboError(RuntimeError):
    def __init__(self, status: int):
        msg = _lib.qubo_status_string(status).decode()
        if status == -5:
            msg += ": " + _lib.qubo_last_error().decode()
        super().__init__(f"qubo status {status}: {msg}")
        self.status = status


def _check(st: int):
    if st != 0:
        raise QuboError(st)


def _matrix(Q):
    Q = np.asarray(Q)
    if Q.ndim != 2 or Q.shape[0] != Q.shape[1]:
        raise ValueError("Q must be a square matrix")
    if Q.dtype == np.float32:
        return np.ascontiguousarray(Q), FP32
    if Q.dtype == np.float64:
        return np.ascontiguousarray(Q), FP64
    if Q.dtype.kind in "iu" and Q.dtype.itemsize <= 4:
        return np.ascontiguousarray(Q, dtype=np.int32), INT32
    if Q.dtype.kind in "iu":
        if Q.size and (Q.min() < -(1 << 31) or Q.max() >= (1 << 31)):
            raise ValueError("integer Q must fit int32")
        return np.ascontiguousarray(Q, dtype=np.int32), INT32
    raise TypeError("Q must be int32, float32 or float64")


def solve(Q, k_prefix: int = 0, cache_bits: int = 0):
    """Exhaustive minimum of E(x) = x^T Q x over {0,1}^n: (E_min, argmin x, tie count)."""
    Q, dt = _matrix(Q)
    n = Q.shape[0]
    e = ctypes.c_double()
    x = np.zeros(n, np.uint8)
    t = ctypes.c_uint64()
    _check(_lib.qubo_solve(n, Q.ctypes.data, dt, k_prefix, cache_bits, ctypes.byref(e),
                           x.ctypes.data_as(_u8p), ctypes.byref(t)))
    return (int(e.value) if dt == INT32 else float(e.value)), x, int(t.value)


def solve_slices(Q, k_prefix: int, slice_ids, cache_bits: int = 0):
    """Per-slice results for the slices whose first k_prefix variables equal slice_ids (MSB first)."""
    Q, dt = _matrix(Q)
    n = Q.shape[0]
    ids = np.ascontiguousarray(slice_ids, dtype=np.uint64)
    m = ids.size
    e = np.zeros(m, np.float64)
    x = np.zeros((m, n), np.uint8)
    t = np.zeros(m, np.uint64)
    _check(_lib.qubo_solve_slices(n, Q.ctypes.data, dt, k_prefix, cache_bits, ids.ctypes.data_as(_u64p), m,
                                  e.ctypes.data_as(_f64p), x.ctypes.data_as(_u8p), t.ctypes.data_as(_u64p)))
    if dt == INT32:
        e = e.astype(np.int64)
    return e, x, t


def solve_slice_range(Q, k_prefix: int, first_slice: int, num_slices: int, cache_bits: int = 0):
    """One result over the slices [first_slice, first_slice + num_slices) of k_prefix bits."""
    Q, dt = _matrix(Q)
    n = Q.shape[0]
    e = ctypes.c_double()
    x = np.zeros(n, np.uint8)
    t = ctypes.c_uint64()
    _check(_lib.qubo_solve_slice_range(n, Q.ctypes.data, dt, k_prefix, cache_bits, first_slice, num_slices,
                                       ctypes.byref(e), x.ctypes.data_as(_u8p), ctypes.byref(t)))
    return (int(e.value) if dt == INT32 else float(e.value)), x, int(t.value)


LOWEST_MAX_K = 1 << 20


def solve_lowest(Q, k: int, k_prefix: int = 0, cache_bits: int = 0):
    """The min(k, 2^n) lowest states of x^T Q x (int32 Q): (energies int64[m], states uint8[m, n]),
    ordered by energy, then by rank."""
    Q, dt = _matrix(Q)
    n = Q.shape[0]
    e = np.zeros(k, np.float64)
    x = np.zeros((k, n), np.uint8)
    m = ctypes.c_int()
    _check(_lib.qubo_solve_lowest(n, Q.ctypes.data, dt, k_prefix, cache_bits, k, e.ctypes.data_as(_f64p),
                                  x.ctypes.data_as(_u8p), ctypes.byref(m)))
    return e[:m.value].astype(np.int64), x[:m.value]


INCOMPLETE = 1


def solve_checkpointed(Q, k_prefix: int, checkpoint_path: str, slices_per_chunk: int = 0,
                       time_budget_s: float = 0.0, cache_bits: int = 0):
    """Slice-chunked search that saves its progress after every chunk and resumes from the file.

    Returns (complete, E, x, ties, slices_done): complete is False when the time budget ended the
    call (E, x, ties then cover the slices done so far)."""
    Q, dt = _matrix(Q)
    n = Q.shape[0]
    e = ctypes.c_double()
    x = np.zeros(n, np.uint8)
    t = ctypes.c_uint64()
    done = ctypes.c_uint64()
    st = _lib.qubo_solve_checkpointed(n, Q.ctypes.data, dt, k_prefix, cache_bits, slices_per_chunk,
                                      os.fsencode(checkpoint_path), time_budget_s, ctypes.byref(e),
                                      x.ctypes.data_as(_u8p), ctypes.byref(t), ctypes.byref(done))
    if st not in (0, INCOMPLETE):
        raise QuboError(st)
    return st == 0, (int(e.value) if dt == INT32 else float(e.value)), x, int(t.value), int(done.value)


def checkpoint_read(checkpoint_path: str) -> dict:
    """Contents of a checkpoint file written by solve_checkpointed."""
    ints = [ctypes.c_int() for _ in range(4)]
    u64 = [ctypes.c_uint64() for _ in range(5)]
    e = ctypes.c_double()
    _check(_lib.qubo_checkpoint_read(os.fsencode(checkpoint_path), ctypes.byref(ints[0]), ctypes.byref(ints[1]),
                                     ctypes.byref(ints[2]), ctypes.byref(u64[0]), ctypes.byref(u64[1]),
                                     ctypes.byref(u64[2]), ctypes.byref(ints[3]), ctypes.byref(e),
                                     ctypes.byref(u64[3]), ctypes.byref(u64[4])))
    return {"n": ints[0].value, "dtype": ints[1].value, "k_prefix": ints[2].value, "q_hash": u64[0].value,
            "next_slice": u64[1].value, "total_slices": u64[2].value, "have": ints[3].value,
            "min_energy": e.value, "argmin_rank": u64[3].value, "tie_count": u64[4].value}


def fnv1a64(data) -> int:
    """The 64-bit FNV-1a hash the checkpoint files use to identify a problem."""
    b = bytes(data)
    buf = ctypes.create_string_buffer(b, len(b))
    return int(_lib.qubo_fnv1a64(buf, len(b)))


def _ising_inputs(J, h):
    J = np.asarray(J)
    if J.ndim != 2 or J.shape[0] != J.shape[1]:
        raise ValueError("J must be a square matrix")
    n = J.shape[0]
    if J.dtype in (np.float32, np.float64):
        dt = FP32 if J.dtype == np.float32 else FP64
        J = np.ascontiguousarray(J)
        h = None if h is None else np.ascontiguousarray(h, dtype=J.dtype)
    else:
        dt = INT32
        J, _ = _matrix(J)
        h = None if h is None else np.ascontiguousarray(h, dtype=np.int32)
    if h is not None and h.shape != (n,):
        raise ValueError("h must have n entries")
    return J, h, dt, n


def ising_to_qubo(J, h=None):
    """Exact QUBO of H(s) = sum_ij J_ij s_i s_j + sum_i h_i s_i: (Q, offset), H = E_Q(x) + offset."""
    J, h, dt, n = _ising_inputs(J, h)
    Q = np.zeros((n, n), np.int32 if dt == INT32 else np.float64)
    off = ctypes.c_double()
    _check(_lib.qubo_ising_to_qubo(n, J.ctypes.data, None if h is None else h.ctypes.data, dt, Q.ctypes.data,
                                   ctypes.byref(off)))
    return Q, (int(off.value) if dt == INT32 else float(off.value))


def solve_ising(J, h=None, k_prefix: int = 0, cache_bits: int = 0):
    """Exhaustive Ising ground state: (H_min, spins s in {-1,+1} as int8, number of ground states)."""
    J, h, dt, n = _ising_inputs(J, h)
    e = ctypes.c_double()
    s = np.zeros(n, np.int8)
    t = ctypes.c_uint64()
    _check(_lib.qubo_solve_ising(n, J.ctypes.data, None if h is None else h.ctypes.data, dt, k_prefix, cache_bits,
                                 ctypes.byref(e), s.ctypes.data, ctypes.byref(t)))
    return (int(e.value) if dt == INT32 else float(e.value)), s, int(t.value)


def solve_batched(Qs):
    """Independent problems Qs[b] (batch x n x n, int32): arrays of E_min, argmin x, ties."""
    Qs = np.ascontiguousarray(Qs, dtype=np.int32)
    if Qs.ndim != 3 or Qs.shape[1] != Qs.shape[2]:
        raise ValueError("Qs must be batch x n x n")
    b, n = Qs.shape[0], Qs.shape[1]
    e = np.zeros(b, np.float64)
    x = np.zeros((b, n), np.uint8)
    t = np.zeros(b, np.uint64)
    _check(_lib.qubo_solve_batched(b, n, Qs.ctypes.data, INT32, e.ctypes.data_as(_f64p), x.ctypes.data_as(_u8p),
                                   t.ctypes.data_as(_u64p)))
    return e.astype(np.int64), x, t


def _ptr(a) -> int:
    if a is None:
        return 0
    if isinstance(a, int):
        return a
    return int(a.data_ptr())


def workspace_bytes(n: int, dtype: int = INT32, k_prefix: int = 0, cache_bits: int = 0) -> int:
    return int(_lib.qubo_workspace_bytes(n, dtype, k_prefix, cache_bits))


def batched_workspace_bytes(batch: int, n: int, dtype: int = INT32) -> int:
    return int(_lib.qubo_batched_workspace_bytes(batch, n, dtype))


def solve_device(n: int, d_Q, dtype: int, workspace, workspace_nbytes: int, stream, d_result,
                 k_prefix: int = 0, cache_bits: int = 0) -> None:
    """Enqueue a search on device memory: d_Q, workspace and d_result are device pointers (ints or
    tensors with data_ptr()); stream is a cudaStream_t handle (int) or None. Asynchronous."""
    _check(_lib.qubo_solve_device(n, _ptr(d_Q), dtype, k_prefix, cache_bits, _ptr(workspace), workspace_nbytes,
                                  _ptr(stream) if stream is not None else 0, _ptr(d_result)))


NO_ALLOC_SCRATCH_BYTES = 8 << 20


def solve_device_no_alloc(n: int, d_Q, dtype: int, stream, d_result, k_prefix: int = 0, cache_bits: int = 0) -> None:
    """Like solve_device, but with no workspace argument and no allocation: for callers that cannot
    call cudaMalloc (a latency-critical loop, or a plug-in whose host owns all device memory).
    Scratch is one fixed device array of NO_ALLOC_SCRATCH_BYTES shared by all calls; larger
    problems raise QuboError(-1). Calls that overlap on the GPU race: keep them on one stream."""
    _check(_lib.qubo_solve_device_no_alloc(n, _ptr(d_Q), dtype, k_prefix, cache_bits,
                                           _ptr(stream) if stream is not None else 0, _ptr(d_result)))


def slice_range_workspace_bytes(n: int, dtype: int, k_prefix: int, num_slices: int, cache_bits: int = 0) -> int:
    return int(_lib.qubo_slice_range_workspace_bytes(n, dtype, k_prefix, cache_bits, num_slices))


def solve_slice_range_device(n: int, d_Q, dtype: int, k_prefix: int, first_slice: int, num_slices: int, workspace,
                             workspace_nbytes: int, stream, d_result, cache_bits: int = 0) -> None:
    """Enqueue the search of slices [first_slice, first_slice + num_slices) on device memory."""
    _check(_lib.qubo_solve_slice_range_device(n, _ptr(d_Q), dtype, k_prefix, cache_bits, first_slice, num_slices,
                                              _ptr(workspace), workspace_nbytes,
                                              _ptr(stream) if stream is not None else 0, _ptr(d_result)))


def enable_kernel_timing(enable: bool = True) -> None:
    _lib.qubo_enable_kernel_timing(1 if enable else 0)


def enable_block_bounds(enable: bool = True) -> None:
    """Block bounds in the single-problem minimum pass (on by default). Off, calls planned from
    then on form every step's minimum (the packed pass for narrow int32 input, the biased pass
    without bounds otherwise); results are identical either way."""
    _lib.qubo_enable_block_bounds(1 if enable else 0)


def kernel_time_ms() -> float:
    """Elapsed ms of the enumeration launches of the most recent call (events on its stream)."""
    return float(_lib.qubo_kernel_time_ms())


def solve_batched_device(batch: int, n: int, d_Q, workspace, workspace_nbytes: int, stream, d_results) -> None:
    _check(_lib.qubo_solve_batched_device(batch, n, _ptr(d_Q), INT32, _ptr(workspace), workspace_nbytes,
                                          _ptr(stream) if stream is not None else 0, _ptr(d_results)))


def plan(n: int, dtype: int = INT32, k_prefix: int = 0, cache_bits: int = 0) -> dict:
    d = _PlanDesc()
    _check(_lib.qubo_plan(n, dtype, k_prefix, cache_bits, ctypes.byref(d)))
    return {f: getattr(d, f) for f, _ in _PlanDesc._fields_}


def probe_alu(kind: int, iters: int = 20000):
    """(lane-operations per second, SM MHz) of one ALU operation kind on the current device."""
    ops, mhz = ctypes.c_double(), ctypes.c_double()
    _check(_lib.qubo_probe_alu(kind, iters, ctypes.byref(ops), ctypes.byref(mhz)))
    return ops.value, mhz.value


def last_launch_count() -> int:
    return int(_lib.qubo_last_launch_count())


def status_string(status: int) -> str:
    return _lib.qubo_status_string(status).decode()


def last_error() -> str:
    return _lib.qubo_last_error().decode()


def request_abort() -> None:
    _lib.qubo_request_abort()


def clear_abort() -> None:
    _lib.qubo_clear_abort()


def rank_to_bits(n: int, rank: int) -> np.ndarray:
    return np.array([(int(rank) >> (n - 1 - i)) & 1 for i in range(n)], dtype=np.uint8)
