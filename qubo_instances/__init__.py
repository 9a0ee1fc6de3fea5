"""Seeded synthetic QUBO instances shared by the oracle tests, the GPU tests and the bench.

This module only draws numbers and lays them out as matrices. It holds none of the
search arithmetic (no energies, no folding, no minimisation), so the oracle and the
CUDA path stay independent of each other while solving identical inputs.

Random source: SplitMix64 (Steele, Lea and Flood, "Fast splittable pseudorandom number
generators", OOPSLA 2014; constants as published by Vigna for java.util.SplittableRandom).
It is counter based: draw k (k = 1, 2, ...) of seed s is mix(s + k * GAMMA) mod 2^64,
so the stream can be produced in vectorised blocks.

* integers in [lo, hi]: rejection sampling on the full 64-bit draw, then lo + u mod m;
* N(0,1): Box-Muller in fp64 on two consecutive draws (only the cosine branch is used),
  rounded to fp32 afterwards;
* matrices are filled row-major over the upper triangle i <= j, one draw per entry.

The pages benchmark on uniformly random matrices without stating a range or a seed
(Terastate-per-second QUBO Brute-Force, §V-C); the ranges and the master seed below are
the workload definition used throughout this repository.
"""
from __future__ import annotations

import numpy as np

MASTER_SEED = 20260702

_GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_MASK64 = (1 << 64) - 1


def splitmix64_block(seed: int, start: int, count: int) -> np.ndarray:
    """Draws start+1 .. start+count of the SplitMix64 stream of `seed` (uint64 array)."""
    k = np.arange(start + 1, start + count + 1, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = np.uint64(seed & _MASK64) + k * _GAMMA
        z = (z ^ (z >> np.uint64(30))) * _M1
        z = (z ^ (z >> np.uint64(27))) * _M2
        z = z ^ (z >> np.uint64(31))
    return z


def splitmix64_scalar(seed: int, k: int) -> int:
    """Draw k (1-based) of the stream, in plain Python integers (reference for the block form)."""
    z = (seed + k * 0x9E3779B97F4A7C15) & _MASK64
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & _MASK64
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & _MASK64
    return z ^ (z >> 31)


class Stream:
    """Sequential reader over one SplitMix64 stream."""

    def __init__(self, seed: int):
        self.seed = int(seed)
        self.pos = 0

    def raw(self, count: int) -> np.ndarray:
        out = splitmix64_block(self.seed, self.pos, count)
        self.pos += count
        return out

    def integers(self, lo: int, hi: int, count: int) -> np.ndarray:
        """`count` integers uniform in [lo, hi] by rejection sampling (int64 array)."""
        m = hi - lo + 1
        assert m >= 1
        limit = ((1 << 64) // m) * m  # accept u < limit
        out = np.empty(count, dtype=np.int64)
        filled = 0
        while filled < count:
            need = count - filled
            u = self.raw(need)
            if limit < (1 << 64):
                u = u[u < np.uint64(limit)]
            take = u[:need]
            out[filled:filled + take.size] = (take % np.uint64(m)).astype(np.int64) + lo
            filled += take.size
            # Rejected draws were consumed; keep reading the stream in order.
        return out

    def normals(self, count: int) -> np.ndarray:
        """`count` N(0,1) samples (fp64) by Box-Muller on consecutive draw pairs."""
        u = self.raw(2 * count).reshape(count, 2)
        scale = 2.0 ** -53
        u1 = 1.0 - (u[:, 0] >> np.uint64(11)).astype(np.float64) * scale  # (0, 1]
        u2 = (u[:, 1] >> np.uint64(11)).astype(np.float64) * scale  # [0, 1)
        return np.sqrt(-2.0 * np.log(u1)) * np.cos(2.0 * np.pi * u2)

    def signs(self, count: int) -> np.ndarray:
        """`count` values in {-1, +1} from the top bit of each draw."""
        return 1 - 2 * (self.raw(count) >> np.uint64(63)).astype(np.int64)


def _upper_fill(n: int, values: np.ndarray, dtype) -> np.ndarray:
    q = np.zeros((n, n), dtype=dtype)
    iu = np.triu_indices(n)  # row-major order over i <= j
    q[iu] = values
    return q


def random_upper_int(n: int, lo: int, hi: int, seed: int) -> np.ndarray:
    """n x n int32 matrix, upper triangle (diagonal included) uniform in [lo, hi], zero below."""
    s = Stream(seed)
    return _upper_fill(n, s.integers(lo, hi, n * (n + 1) // 2), np.int32)


def random_full_int(n: int, lo: int, hi: int, seed: int) -> np.ndarray:
    """n x n int32 matrix with every entry uniform in [lo, hi] (not triangular), row-major."""
    s = Stream(seed)
    return s.integers(lo, hi, n * n).reshape(n, n).astype(np.int32)


def random_symmetric_normal_f32(n: int, seed: int) -> np.ndarray:
    """n x n fp32 matrix with Q_ij = Q_ji ~ N(0,1), drawn for i <= j and mirrored."""
    s = Stream(seed)
    q = _upper_fill(n, s.normals(n * (n + 1) // 2), np.float64)
    q = q + np.triu(q, 1).T
    return q.astype(np.float32)


def mattis_couplings(n: int, wlo: int, whi: int, seed: int):
    """Planted Mattis-type Ising instance on the complete graph.

    Returns (s_star, w, J): s_star in {-1,+1}^n, integer weights w_ij in [wlo, whi] for i < j
    (upper triangle, zero elsewhere), and couplings J_ij = -w_ij s*_i s*_j for i < j, h = 0.
    """
    s = Stream(seed)
    s_star = s.signs(n)
    w = np.zeros((n, n), dtype=np.int64)
    iu = np.triu_indices(n, 1)
    w[iu] = s.integers(wlo, whi, n * (n - 1) // 2)
    J = -w * np.outer(s_star, s_star)
    J = np.triu(J, 1)
    return s_star, w, J


def ising_to_qubo(J: np.ndarray, h: np.ndarray):
    """Ising (J upper triangular, h) to an upper-triangular integer QUBO matrix and offset.

    With s = 2x - 1 and H(s) = sum_{i<j} J_ij s_i s_j + sum_i h_i s_i:
    Q_ij = 4 J_ij (i < j), Q_ii = -2 sum_{j != i} J_ij + 2 h_i, offset = sum_{i<j} J_ij - sum_i h_i,
    so that H(s) = x^T Q x + offset. This is instance construction (a change of variables),
    not part of the search.
    """
    J = np.triu(np.asarray(J, dtype=np.int64), 1)
    h = np.asarray(h, dtype=np.int64)
    n = J.shape[0]
    Jsym = J + J.T
    Q = 4 * J
    Q[np.diag_indices(n)] = -2 * Jsym.sum(axis=1) + 2 * h
    offset = int(J.sum() - h.sum())
    return Q, offset


def mattis_planted(n: int, seed: int, wlo: int = 1, whi: int = 100):
    """Mattis planted QUBO (int32 upper-triangular) with its couplings; see mattis_couplings."""
    s_star, w, J = mattis_couplings(n, wlo, whi, seed)
    Q, offset = ising_to_qubo(J, np.zeros(n, dtype=np.int64))
    return Q.astype(np.int32), s_star, w, offset


def batched_upper_int(batch: int, n: int, lo: int, hi: int, seed: int) -> np.ndarray:
    """batch x n x n int32: instance i is random_upper_int(n, lo, hi, seed + i)."""
    out = np.empty((batch, n, n), dtype=np.int32)
    for i in range(batch):
        out[i] = random_upper_int(n, lo, hi, seed + i)
    return out


# The workloads (sizes, ranges, seeds) measured and checked by this repository.
def workload_n20():
    return random_upper_int(20, -100, 100, MASTER_SEED + 0)


def workload_n32():
    return random_upper_int(32, -1000, 1000, MASTER_SEED + 1)


def workload_n32_mattis():
    return mattis_planted(32, MASTER_SEED + 101)


def workload_n40():
    return random_upper_int(40, -1000, 1000, MASTER_SEED + 2)


def workload_n40_narrow():
    """n=40 dense, entries uniform in [-4, 4]: sum |U| ~ 1.8e3, inside the 16-bit packed range."""
    return random_upper_int(40, -4, 4, MASTER_SEED + 5)


def workload_n36_wide():
    """n=36 dense, entries uniform in [-2^20, 2^20]: sum |U| ~ 3.5e8, beyond the fp32 binade
    (2^22), so the minimum pass adds in int32."""
    return random_upper_int(36, -(1 << 20), 1 << 20, MASTER_SEED + 7)


def workload_n36_f32():
    return random_symmetric_normal_f32(36, MASTER_SEED + 3)


def workload_batched(batch: int = 4096, n: int = 24):
    return batched_upper_int(batch, n, -50, 50, MASTER_SEED + 4 * 1000000)
