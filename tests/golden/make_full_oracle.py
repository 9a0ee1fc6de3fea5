"""Writes the full-search oracle results of the n=36 and n=40 workloads that the bench checks.

Every state of each workload is evaluated by the CPU oracle (oracle_gray: the O(n)-per-step Gray
walk over all 2^n states, OpenMP over leading-bit slices); nothing here touches the CUDA path.
The n=40 run takes hours on a few cores, so its result is stored and the GPU tests compare
against the stored value.

    python tests/golden/make_full_oracle.py [n36_fp32] [n40_int32] [n36_wide_int32] [n40_narrow_int32]
"""
import os
import sys
import time

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
import qubo_instances as qi  # noqa: E402

CASES = {
    "n36_fp32": ("n=36 fp32, entries N(0,1), symmetric (qubo_instances.workload_n36_f32)", qi.workload_n36_f32),
    "n40_int32": ("n=40 int32, upper-triangular, entries uniform in [-1000, 1000] (qubo_instances.workload_n40)",
                  qi.workload_n40),
    "n36_wide_int32": ("n=36 int32, upper-triangular, entries uniform in [-2^20, 2^20] "
                       "(qubo_instances.workload_n36_wide)", qi.workload_n36_wide),
    "n40_narrow_int32": ("n=40 int32, upper-triangular, entries uniform in [-4, 4] "
                         "(qubo_instances.workload_n40_narrow)", qi.workload_n40_narrow),
}


def main(names):
    O = oracle.get()
    for name in names:
        desc, make = CASES[name]
        Q = make()
        t0 = time.time()
        e, x, ties = O.solve(Q)
        dt = time.time() - t0
        rank = oracle.rank_of_bits(x)
        path = os.path.join(ROOT, "tests", "golden", f"full_oracle_{name}.txt")
        with open(path, "w") as f:
            f.write(f"# Full exhaustive search by the CPU oracle (oracle_gray) of the workload {desc}.\n")
            f.write(f"# Written by tests/golden/make_full_oracle.py ({O.num_threads()} threads, {dt:.0f} s).\n")
            f.write("# Columns: minimum energy (exact integer for int32, repr of the fp64 value for fp32), "
                    "rank of the lowest-rank minimiser (x_0 most significant), number of minimisers.\n")
            f.write(f"{e!r} {rank} {ties}\n")
        print(name, e, rank, ties, f"{dt:.0f} s", flush=True)


if __name__ == "__main__":
    main(sys.argv[1:] or list(CASES))
