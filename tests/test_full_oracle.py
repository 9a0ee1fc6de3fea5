"""The whole n=36 and n=40 workloads against a full exhaustive oracle search.

tests/golden/make_full_oracle.py ran the CPU oracle over all 2^36 or 2^40 states and stored the
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


@pytest.mark.parametrize("name,n,make", [("n36_wide_int32", 36, qi.workload_n36_wide),
                                         ("n40_narrow_int32", 40, qi.workload_n40_narrow)])
def test_stored_int32_minimisers_have_the_stored_energy(name, n, make):
    e, rank, ties = _golden(name)
    U = O.fold_i32(make())
    x = oracle.bits_of_rank(n, rank)
    assert O.energy_i64(U, x) == e and ties >= 1
    for v in range(n):
        y = x.copy()
        y[v] ^= 1
        assert O.energy_i64(U, y) >= e


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


@pytest.mark.gpu
@pytest.mark.parametrize("name,n,make", [("n36_wide_int32", 36, qi.workload_n36_wide),
                                         ("n40_narrow_int32", 40, qi.workload_n40_narrow)])
def test_int32_workloads_with_and_without_bounds_against_full_oracle(q, name, n, make):
    # wide entries take the int32 pass; narrow ones the bounded biased pass, and without bounds
    # the packed 16x2 pass
    e, rank, ties = _golden(name)
    Q = make()
    ge, gx, gt = q.solve(Q)
    assert (ge, oracle.rank_of_bits(gx), gt) == (e, rank, ties)
    q.enable_block_bounds(False)
    try:
        ge, gx, gt = q.solve(Q)
    finally:
        q.enable_block_bounds(True)
    assert (ge, oracle.rank_of_bits(gx), gt) == (e, rank, ties)


@pytest.mark.gpu
def test_n40_workload_without_bounds_against_full_oracle(q):
    e, rank, ties = _golden("n40_int32")
    q.enable_block_bounds(False)
    try:
        ge, gx, gt = q.solve(qi.workload_n40())
    finally:
        q.enable_block_bounds(True)
    assert (ge, oracle.rank_of_bits(gx), gt) == (e, rank, ties)
