"""The whole n=36 fp32 and n=40 int32 workloads against a full exhaustive oracle search.

tests/golden/make_full_oracle.py ran the CPU oracle over all 2^36 and 2^40 states and stored the
minimum, the lowest-rank minimiser and the number of minimisers. The CPU tests pin the stored
minimiser to the stored energy with the oracle's direct energy evaluation; the GPU tests compare
the CUDA path's whole-problem answer with the stored one.
"""
import os

import numpy as np
import pytest

import oracle
import qubo_instances as qi
from conftest import ROOT, read_golden

O = oracle.get()


def _golden(name):
    path = os.path.join(ROOT, "tests", "golden", f"full_oracle_{name}.txt")
    if not os.path.exists(path):
        pytest.skip(f"{path} not generated")
    (row,) = read_golden(f"full_oracle_{name}.txt")
    return float(row[0]) if "." in row[0] or "e" in row[0] else int(row[0]), int(row[1]), int(row[2])


def test_stored_n40_minimiser_has_the_stored_energy():
    e, rank, ties = _golden("n40_int32")
    Q = qi.workload_n40()
    x = oracle.bits_of_rank(40, rank)
    assert O.energy_i64(O.fold_i32(Q), x) == e and ties >= 1
    # the minimiser is a local minimum: no single flip lowers the energy
    U = O.fold_i32(Q)
    for v in range(40):
        y = x.copy()
        y[v] ^= 1
        assert O.energy_i64(U, y) >= e


def test_stored_n36_fp32_minimiser_has_the_stored_energy():
    e, rank, ties = _golden("n36_fp32")
    Q = qi.workload_n36_f32()
    U = O.fold_f32(Q)
    x = oracle.bits_of_rank(36, rank)
    assert O.eval64(U, x) == e and ties >= 1
    for v in range(36):
        y = x.copy()
        y[v] ^= 1
        assert O.eval64(U, y) >= e


@pytest.fixture(scope="module")
def q():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import exact_qubo_exhaustive_gb300 as lib
    return lib


@pytest.mark.gpu
def test_n40_workload_whole_problem_against_full_oracle(q):
    e, rank, ties = _golden("n40_int32")
    ge, gx, gt = q.solve(qi.workload_n40())
    assert (ge, oracle.rank_of_bits(gx), gt) == (e, rank, ties)


@pytest.mark.gpu
def test_n36_fp32_workload_whole_problem_against_full_oracle(q):
    e, rank, ties = _golden("n36_fp32")
    Q = qi.workload_n36_f32()
    ge, gx, gt = q.solve(Q)
    tol = 1e-3 * float(np.abs(Q.astype(np.float64)).sum()) * 2.0 ** -20
    assert abs(ge - e) <= tol
    assert oracle.rank_of_bits(gx) == rank and gt == ties
