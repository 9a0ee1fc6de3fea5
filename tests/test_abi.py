"""The C-ABI library loads and exports every function include/qubo.h declares; host-side argument
checks answer without touching a GPU (CPU-only tests)."""
import ctypes
import os
import re

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    text = open(os.path.join(ROOT, "include", "qubo.h")).read()
    return re.findall(r"^QUBO_API\s+[\w\s\*]+?\b(qubo_\w+)\s*\(", text, flags=re.M)


def test_header_declares_the_entry_points():
    names = set(declared_functions())
    for must in ("qubo_solve", "qubo_solve_slices", "qubo_solve_batched", "qubo_solve_device",
                 "qubo_workspace_bytes", "qubo_status_string"):
        assert must in names


def test_library_exports_every_declared_symbol():
    import exact_qubo_exhaustive_gb300 as q
    lib = ctypes.CDLL(q.library_path())
    names = declared_functions()
    assert len(names) >= 15
    for name in names:
        assert hasattr(lib, name), name


def test_status_strings():
    import exact_qubo_exhaustive_gb300 as q
    for st in range(0, -8, -1):
        assert q.status_string(st) and q.status_string(st) != "unknown status"


def test_argument_errors_need_no_device():
    import exact_qubo_exhaustive_gb300 as q
    lib = ctypes.CDLL(q.library_path())
    e = ctypes.c_double()
    t = ctypes.c_uint64()
    x = (ctypes.c_uint8 * 64)()
    Q = np.zeros((4, 4), np.int32)
    for n in (0, -1, 63):
        assert lib.qubo_solve(n, Q.ctypes.data_as(ctypes.c_void_p), 0, 0, 0, ctypes.byref(e), x, ctypes.byref(t)) == -1
    assert lib.qubo_solve(4, None, 0, 0, 0, ctypes.byref(e), x, ctypes.byref(t)) == -1
    assert lib.qubo_solve(4, Q.ctypes.data_as(ctypes.c_void_p), 7, 0, 0, ctypes.byref(e), x, ctypes.byref(t)) == -1
    assert lib.qubo_solve(4, Q.ctypes.data_as(ctypes.c_void_p), 0, 0, 0, None, x, ctypes.byref(t)) == -1
    # k_prefix beyond n is a plan error, caught on the host
    assert lib.qubo_solve(4, Q.ctypes.data_as(ctypes.c_void_p), 0, 9, 0, ctypes.byref(e), x, ctypes.byref(t)) == -4


def test_no_device_is_reported_not_hidden():
    torch = pytest.importorskip("torch")
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    import exact_qubo_exhaustive_gb300 as q
    with pytest.raises(q.QuboError) as ei:
        q.solve(np.eye(3, dtype=np.int32))
    assert ei.value.status == -6
