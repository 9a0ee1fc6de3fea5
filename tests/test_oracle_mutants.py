"""The pins must be able to fail: oracle builds with one step broken on purpose are rejected.

Mutants (compiled from qubo_oracle.c with -DORACLE_MUTANT=k, CPU only):
  1 -- the diagonal term U_ii is dropped from the energy,
  2 -- the Gray walker ignores the flip direction (always adds),
  3 -- the walker's field update reads the (zero) lower triangle: a transposed operand.
"""
import itertools

import numpy as np
import pytest

import oracle
import qubo_instances as qi


def pins_hold(o: oracle.Oracle) -> bool:
    n = 7
    Q = qi.random_full_int(n, -20, 20, 3)
    U = o.fold_i32(Q)
    for i in range(n):  # E(e_i) = Q_ii
        e = np.zeros(n, np.uint8)
        e[i] = 1
        if o.energy_i64(U, e) != Q[i, i]:
            return False
    E, R = o.gray_trace_i64(U)  # walker equals direct evaluation
    for e, r in zip(E, R):
        if e != o.energy_i64(U, oracle.bits_of_rank(n, int(r))):
            return False
    best = None  # search equals Python brute force
    for r, x in enumerate(itertools.product((0, 1), repeat=n)):
        v = sum(int(Q[i][j]) for i in range(n) for j in range(n) if x[i] and x[j])
        if best is None or v < best[0]:
            best = (v, r, 1)
        elif v == best[0]:
            best = (v, best[1], best[2] + 1)
    return o.gray_i64(U) == best and o.direct_i64(U) == best


def test_correct_oracle_passes_pins():
    assert pins_hold(oracle.get())


@pytest.mark.parametrize("mutant", [1, 2, 3])
def test_mutant_oracle_fails_pins(mutant):
    assert not pins_hold(oracle.Oracle(mutant))
