"""Multi-GPU sharding of one exhaustive search: one process per GPU, contiguous slice ranges.

Terastate-per-second QUBO Brute-Force on a Single GPU, §III-C1 and §IV-C: fixing the first
k_prefix variables splits the search into 2^k_prefix independent subproblems, and every node
builds its own caches, so ranks exchange nothing until the end. The single exchange step
gathers one (minimum energy, lowest argmin rank, tie count) record per rank and reduces them:
the lowest energy wins; among equal energies the lowest rank wins and the tie counts add.

The per-rank search is `solve_slice_range` of this package (the CUDA path); `solver` exists so
that the host logic can be exercised by CPU processes.
"""
from __future__ import annotations

import numpy as np

from . import rank_to_bits, solve_slice_range


def shard_range(num_slices: int, rank: int, world: int) -> tuple[int, int]:
    """Contiguous share of `num_slices` slices for `rank` of `world`: (first slice, count).

    The first num_slices % world ranks take one slice more; a rank may get none when
    world > num_slices.
    """
    if world < 1 or not 0 <= rank < world:
        raise ValueError("need 0 <= rank < world")
    if num_slices < 0:
        raise ValueError("num_slices must be >= 0")
    base, extra = divmod(num_slices, world)
    first = rank * base + min(rank, extra)
    return first, base + (1 if rank < extra else 0)


def _rank_of_bits(x) -> int:
    r = 0
    for b in np.asarray(x, dtype=np.uint8):
        r = (r << 1) | int(b)
    return r


def combine(records):
    """Reduce (energy, argmin rank, ties) records of disjoint shards; None marks an empty shard."""
    best = None
    for rec in records:
        if rec is None:
            continue
        e, r, t = rec
        if best is None or e < best[0]:
            best = (e, r, t)
        elif e == best[0]:
            best = (e, min(r, best[1]), best[2] + t)
    if best is None:
        raise ValueError("no shard held any slice")
    return best


def _pack(rec, device):
    import torch
    if rec is None:
        return torch.tensor([0, 0, 0, 0], dtype=torch.int64, device=device)
    e, r, t = rec
    eb = np.array([e], dtype=np.float64).view(np.int64)[0]
    return torch.tensor([1, int(eb), int(r), int(t)], dtype=torch.int64, device=device)


def _unpack(v, integer: bool):
    v = [int(a) for a in v.tolist()]
    if v[0] == 0:
        return None
    e = float(np.array([v[1]], dtype=np.int64).view(np.float64)[0])
    return (int(e) if integer else e), v[2], v[3]


def solve_distributed(Q, k_prefix: int, group=None, cache_bits: int = 0, solver=None):
    """Exhaustive minimum of x^T Q x over all 2^n states, sharded over the ranks of `group`.

    Every rank must call this with the same Q and k_prefix. Rank i searches its contiguous share
    of the 2^k_prefix slices (`shard_range`), then one all-gather of 4 int64 per rank exchanges
    the shard results and every rank returns the same (E_min, argmin x, tie count).
    `solver(Q, k_prefix, first, count) -> (E, x, ties)` defaults to `solve_slice_range`.
    """
    import torch
    import torch.distributed as dist

    Q = np.asarray(Q)
    n = Q.shape[0]
    if not 0 <= k_prefix <= n:
        raise ValueError("need 0 <= k_prefix <= n")
    rank, world = dist.get_rank(group), dist.get_world_size(group)
    first, count = shard_range(1 << k_prefix, rank, world)
    rec = None
    if count > 0:
        run = solver or (lambda Qm, k, f, c: solve_slice_range(Qm, k, f, c, cache_bits))
        e, x, t = run(Q, k_prefix, first, count)
        rec = (e, _rank_of_bits(x), int(t))
    device = "cuda" if dist.get_backend(group) == "nccl" else "cpu"
    mine = _pack(rec, device)
    gathered = [torch.empty_like(mine) for _ in range(world)]
    dist.all_gather(gathered, mine, group=group)
    # integer input is searched as int32 and its energies are exact integers; float32 and float64
    # input give fp64 energies, which must not be truncated
    integer = Q.dtype.kind in "iu"
    e, r, t = combine(_unpack(g.cpu(), integer) for g in gathered)
    return e, rank_to_bits(n, r), t
