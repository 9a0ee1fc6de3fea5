#!/usr/bin/env python
"""Benchmark: QUBO states evaluated per second at n=40 (int32) on GB300.

One step = one complete exhaustive search of the n=40 dense int32 workload (2^40 states:
fold/validate, cache construction, enumeration, group minimum, tie list, resolution, result
record) through the library's C ABI.

  value : device-resident input (qubo_solve_device), CUDA events on the launching stream around
          each step, L2 flushed (256 MB write) between steps outside the events.
  e2e   : the host API (qubo_solve) from pinned host memory: H2D of Q and D2H of the result are
          inside the timed region (wall clock, synchronised).
  roofline: the enumeration kernel's own duration (CUDA events the library records around its
          launches), one add per state (an exact fp32 add), against the issue roofline of the part:
          152 SMs x 128 lanes/clk x 2.07 GHz; also against the measured fp32-add and int32-add rates.
  cpu_baseline / --impl reference: the CPU oracle (test infrastructure, plain C + OpenMP) on a
          bounded sample of the same workload, on the host's cores.

Multi-GPU (torchrun, one process per GPU): ONE n=40 search sharded over the ranks (§III-C1 and
§IV-C of the paper: the 2^12 slices of the first 12 variables are independent subproblems, and each
GPU builds its own caches). Rank i searches its contiguous share of the slices
(qubo_solve_slice_range_device), then one all-gather of the 32-byte result records is the only
exchange; value = 2^40 / the slowest rank's step time (strong scaling: the total work is fixed).

Every run checks the answer it timed against the stored full oracle search of the workload
(tests/golden/full_oracle_n40_int32.txt) and exits non-zero on a mismatch.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import qubo_instances as qi  # noqa: E402

METRIC = "QUBO states evaluated/sec at n=40 int32 on 1 GB300; % of INT32-add roofline"
UNIT = "states/s"
N = 40
STATES = 1 << N
WORKLOAD = "n=40 dense QUBO, int32 Q upper-triangular incl. diagonal, entries iid uniform integers in [-1000,1000]"
SMS = 152
LANES_PER_CLK = 128          # issue-limited int32 lanes per SM per clock (ALU + FMA-heavy pipes)
MAX_SM_MHZ = 2070.0
PROFILE = os.path.join(ROOT, "profiles", "search_kernel_n40.md")
KERNEL_SOURCES = ["qubo_walk.cuh", "qubo_search_kernel.cuh", "qubo_search_pruned.cu", "qubo_internal.h", "qubo_search.cu"]


SHARD_K = 12                 # slices of the multi-GPU split: 2^12, divisible by 1, 2, 4 and 8 ranks


def log(*a):
    print(*a, file=sys.stderr, flush=True)


def golden(name: str):
    """(E_min, rank of the lowest-rank minimiser, ties) stored by the full oracle search of a workload."""
    path = os.path.join(ROOT, "tests", "golden", f"full_oracle_{name}.txt")
    with open(path) as f:
        row = [ln.split() for ln in f if ln.strip() and not ln.startswith("#")][0]
    e = float(row[0]) if ("." in row[0] or "e" in row[0]) else int(row[0])
    return e, int(row[1]), int(row[2])


class ResultMismatch(RuntimeError):
    pass


def check_result(name: str, e, rank: int, ties: int, tol: float = 0.0) -> str:
    """Compares a timed search's answer with the stored full oracle search; raises on a mismatch."""
    ge, grank, gties = golden(name)
    if abs(float(e) - float(ge)) > tol or int(rank) != grank or int(ties) != gties:
        raise ResultMismatch(f"{name}: got ({e}, {rank}, {ties}), full oracle search gave ({ge}, {grank}, {gties})")
    return "matches the full oracle search"


def combine_gathered(raw: bytes, world: int, result_dtype):
    """Reduces the per-rank result records of one sharded step (the bytes of an all-gather of
    `world` qubo_result records): lowest energy; among equal energies the lowest rank and the summed
    tie counts. Raises if a rank reports an error status."""
    from exact_qubo_exhaustive_gb300.distributed import combine
    recs = np.frombuffer(raw, dtype=result_dtype)
    assert recs.shape[0] == world, (recs.shape, world)
    if (recs["status"] != 0).any():
        raise RuntimeError(f"a shard failed: statuses {recs['status'].tolist()}")
    return combine((float(r["min_energy"]), int(r["argmin_rank"]), int(r["tie_count"])) for r in recs)


def dist_env():
    return int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")), int(os.environ.get("LOCAL_RANK", "0"))


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    for f in KERNEL_SOURCES:
        with open(os.path.join(ROOT, "exact_qubo_exhaustive_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def profiled_traffic():
    """DRAM bytes per enumeration launch from the committed ncu summary, if it describes this kernel."""
    try:
        text = open(PROFILE).read()
    except OSError:
        return None, "no ncu summary"
    kv = {}
    for line in text.splitlines():
        if ":" in line and line.strip().startswith("- "):
            k, v = line.strip()[2:].split(":", 1)
            kv[k.strip()] = v.strip().strip("`")
    if kv.get("kernel_source_sha256") != kernel_source_hash():
        return None, "kernel changed since the ncu capture"
    try:
        return float(kv["traffic_bytes_per_launch_n40"]), "ncu capture of a full n=40 launch (one-pass DRAM metrics)"
    except (KeyError, ValueError):
        return None, "ncu summary without traffic"


class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str):
        self.proc = None
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", gpu_id, f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        out, _ = self.proc.communicate(timeout=10)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for nm, val in zip(names, parts[3:7]):
                if val.lower() == "active":
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def oracle_sample(seconds: float):
    """States/s of the CPU oracle on n=40 slices of 2^24 states (k=16), stopping after `seconds`."""
    import oracle
    O = oracle.get()
    Q = qi.workload_n40()
    U = O.fold_i32(Q)
    k = 16
    ids = qi.Stream(2026).integers(0, (1 << k) - 1, 4096)
    t0 = time.perf_counter()
    done = 0
    for sid in ids:
        O.gray_i64(U, k, int(sid))
        done += 1
        if time.perf_counter() - t0 >= seconds:
            break
    dt = time.perf_counter() - t0
    states = done << (N - k)
    return {"value": states / dt, "unit": UNIT, "cores": O.num_threads(), "kind": "oracle",
            "sample": f"{done} slices x 2^{N - k} states of the n=40 workload (first {k} variables fixed), "
                      f"{dt:.1f} s, Gray-walk oracle (O(n) per state) on all host threads"}


def oracle_configs(seconds_each: float):
    """States/s of the CPU oracle on every workload, on one core and on all host cores: a bounded
    sample of each (whole search for small n, leading slices otherwise)."""
    import oracle
    O = oracle.get()
    all_cores = O.num_threads()
    cases = [
        ("n20_int32", qi.workload_n20(), 0),
        ("n32_int32", qi.workload_n32(), 12),
        ("n32_mattis_int32", qi.workload_n32_mattis()[0], 12),
        ("n40_int32", qi.workload_n40(), 18),
        ("n36_fp32", qi.workload_n36_f32(), 14),
        ("batched_n24_int32", qi.workload_batched(64)[0], 0),
    ]
    out = {"cores_all": all_cores}
    for name, Q, k in cases:
        n = Q.shape[0]
        row = {}
        for label, threads in (("one_core", 1), ("all_cores", all_cores)):
            O.set_threads(threads)
            t0 = time.perf_counter()
            done = 0
            states = 0
            while True:
                O.solve_slice(Q, k, done % (1 << k)) if k else O.solve(Q)
                done += 1
                states += 1 << (n - k)
                if time.perf_counter() - t0 >= seconds_each or (k == 0 and done >= 3):
                    break
            row[label] = states / (time.perf_counter() - t0)
        out[name] = row
    O.set_threads(all_cores)
    return out


def config_dict(plan=None):
    cfg = {"workload": WORKLOAD, "n": N, "states_per_step": STATES, "seed": qi.MASTER_SEED + 2,
           "l2": "flushed between steps (256 MB device write outside the timed events)"}
    if plan:
        cfg.update({"k_prefix": plan["k_prefix"], "cache_bits": plan["cache_bits"],
                    "walked_bits": plan["walked_bits"], "blocks": plan["blocks"],
                    "threads_per_block": plan["threads_per_block"]})
    return cfg


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    import oracle
    O = oracle.get()
    Q = qi.workload_n40()
    U = O.fold_i32(Q)
    k = 18  # each step: a bounded sample of 8 slices of 2^22 states
    ids = qi.Stream(777).integers(0, (1 << k) - 1, 8 * (args.steps + args.warmup))
    per_step = 8
    for s in range(args.warmup):
        for sid in ids[s * per_step:(s + 1) * per_step]:
            O.gray_i64(U, k, int(sid))
    t0 = time.perf_counter()
    for s in range(args.warmup, args.warmup + args.steps):
        for sid in ids[s * per_step:(s + 1) * per_step]:
            O.gray_i64(U, k, int(sid))
    dt = time.perf_counter() - t0
    states = args.steps * per_step * (1 << (N - k))
    value = states / dt
    sample = f"each step: {per_step} slices x 2^{N - k} states of the n=40 workload; CPU oracle, all host threads"
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3 / args.steps,
            "higher_is_better": True, "scaling": "strong", "vs_baseline": None, "dtype": "int64",
            "data": "synthetic", "config": config_dict(),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": O.num_threads(), "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "gpu_launches": 0}
    print(json.dumps(line), flush=True)
    return 0


def max_over_ranks(values, device):
    """Element-wise maximum of per-rank floats over the default process group (the slowest rank
    sets the whole job's step time)."""
    import torch
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return [float(v) for v in t.tolist()]


def run_gb300(args):
    import torch
    rank, world, local = dist_env()
    if world > 1 or args.sharded:
        return run_gb300_sharded(args)
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    import exact_qubo_exhaustive_gb300 as q

    Q = qi.workload_n40()
    plan = q.plan(N)
    dq = torch.from_numpy(Q).to(dev)
    nbytes = q.workspace_bytes(N)
    ws = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    res = torch.zeros(32, dtype=torch.uint8, device=dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    q.enable_kernel_timing(True)

    def step():
        q.solve_device(N, dq, q.INT32, ws, nbytes, stream.cuda_stream, res)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    launches_per_step = q.last_launch_count()

    def barrier():
        if world > 1:
            torch.distributed.barrier()

    props = torch.cuda.get_device_properties(dev)
    gpu_id = f"GPU-{props.uuid}" if getattr(props, "uuid", None) else str(local)
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    kernel_ms = []
    barrier()
    torch.cuda.synchronize()
    sampler = ClockSampler(gpu_id)
    time.sleep(0.3)
    for i in range(args.steps):
        flush.fill_(i & 0xFF)
        starts[i].record(stream)
        step()
        ends[i].record(stream)
        kernel_ms.append(q.kernel_time_ms())
    torch.cuda.synchronize()
    barrier()
    clocks = sampler.stop()
    step_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    ms = sum(step_ms) / args.steps
    kern = sum(kernel_ms) / len(kernel_ms)
    r = np.frombuffer(res.cpu().numpy().tobytes(), dtype=q.RESULT_DTYPE)[0]
    if int(r["status"]) != 0:
        raise RuntimeError(f"search failed: status {int(r['status'])}")
    checks = {"n40_int32": check_result("n40_int32", float(r["min_energy"]), int(r["argmin_rank"]),
                                        int(r["tie_count"]))}

    # end to end through the host API, from pinned host memory
    pinned = torch.empty((N, N), dtype=torch.int32, pin_memory=True)
    pinned.copy_(torch.from_numpy(Q))
    Qh = pinned.numpy()
    q.solve(Qh)
    e2e_ms = []
    for i in range(args.steps):
        flush.fill_(i & 0xFF)
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        he, hx, ht = q.solve(Qh)
        e2e_ms.append((time.perf_counter() - t0) * 1e3)
    e2e = sum(e2e_ms) / len(e2e_ms)
    checks["n40_int32_host_api"] = check_result("n40_int32", he, int("".join(map(str, hx)), 2), ht)

    value = STATES / (ms * 1e-3)
    e2e_value = STATES / (e2e * 1e-3)
    achieved = STATES / (kern * 1e-3) / 1e12  # int32 adds (one per state) per second, in T/s
    peak = SMS * LANES_PER_CLK * MAX_SM_MHZ * 1e6 / 1e12
    # the measured INT32-add roofline: the best int32 add throughput of the add microbenchmark
    # (kind 0: the compiler's own split of the adds; kind 8: half of them forced onto the FMA
    # pipe's multiply-add) times the SM count, at the clock the probe saw
    probes = [q.probe_alu(kind, 4000) for kind in (0, 8)]
    best_ops, probe_mhz = max(probes, key=lambda t: t[0])
    r_int = best_ops / 1e12
    # the add the kernel issues is an fp32 add (exact integers in the binade [2^23, 2^24)): its
    # measured rate is the roofline of the pipe the kernel runs on (the better of two patterns:
    # kind 4, chains that read a neighbour's sum; kind 16, loop-invariant addends as in the walk)
    fadd_ops, fadd_mhz = max((q.probe_alu(kind, 4000) for kind in (4, 16)), key=lambda t: t[0])
    r_fadd = fadd_ops / 1e12
    traffic, traffic_src = profiled_traffic()

    extra = {}
    if not args.no_extra:
        extra = other_configs(q, torch, dev, stream)
    cpu = None
    if not args.no_cpu:
        cpu = oracle_sample(args.cpu_seconds)

    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "strong",
        "vs_baseline": None, "dtype": "int32", "data": "synthetic (seeded uniform integers, no dataset)",
        "config": config_dict(plan),
        "result": {"min_energy": float(r["min_energy"]), "argmin_rank": int(r["argmin_rank"]),
                   "tie_count": int(r["tie_count"]), "checks": checks},
        "roofline": {"bound": "alu", "achieved": achieved, "peak": peak, "unit": "Tops/s (int32 lane-ops)",
                     "frac": achieved / peak, "traffic": traffic,
                     "kernel": ("search_kernel<16,R,min,biased,bounded> (enumeration, biased fp32-binade minimum pass "
                                "with block bounds; R = 7 register rows at n=40)"), "kernel_ms": kern,
                     "peak_basis": "152 SMs x 128 lanes/clk (4 schedulers x 32 lanes: the issue limit of one "
                                   "add per state) x 2.07 GHz max SM clock",
                     "traffic_source": traffic_src,
                     "measured_fp32_add_peak": r_fadd,
                     "frac_of_measured_fp32_add": achieved / r_fadd,
                     "measured_fp32_add_basis": (f"qubo_probe_alu fp32 add chains: {fadd_ops / (SMS * fadd_mhz * 1e6):.1f} "
                                                 f"lanes/clk/SM at {fadd_mhz:.0f} MHz x {SMS} SMs; the kernel's one add "
                                                 "per state is an fp32 add (ncu: 2^n fp32 add lane-ops per launch)"),
                     "measured_int32_add_peak": r_int,
                     "frac_of_measured_int32_add": achieved / r_int,
                     "measured_int32_add_basis": (f"qubo_probe_alu int32 add chains: {best_ops / (SMS * probe_mhz * 1e6):.1f} "
                                                  f"lanes/clk/SM at {probe_mhz:.0f} MHz x {SMS} SMs; above 1 because the "
                                                  "kernel's adds are fp32 adds, which this part issues faster than int32 adds"),
                     "frac_at_measured_clock": (achieved / (SMS * LANES_PER_CLK * clocks["sm_mhz"] * 1e-6)
                                                if clocks.get("sm_mhz") else None)},
        "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": N * N * 4,
                "d2h_bytes_per_step": 32, "ms_per_step": e2e},
        "cpu_baseline": cpu,
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clocks,
        "other_configs": extra,
    }
    print(json.dumps(line), flush=True)
    return 0


def run_gb300_sharded(args):
    """N > 1: one n=40 search sharded over the ranks by contiguous ranges of its 2^SHARD_K slices."""
    import torch
    import torch.distributed as dist
    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dist.init_process_group("nccl", device_id=dev)
    import exact_qubo_exhaustive_gb300 as q
    from exact_qubo_exhaustive_gb300 import distributed as qd

    Q = qi.workload_n40()
    first, count = qd.shard_range(1 << SHARD_K, rank, world)
    dq = torch.from_numpy(Q).to(dev)
    nbytes = max(q.slice_range_workspace_bytes(N, q.INT32, SHARD_K, count), 256)
    ws = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    res = torch.zeros(32, dtype=torch.uint8, device=dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    q.enable_kernel_timing(True)

    def step(out):
        q.solve_slice_range_device(N, dq, q.INT32, SHARD_K, first, count, ws, nbytes, stream.cuda_stream, res)
        dist.all_gather_into_tensor(out, res)  # the one exchange: 32 bytes per rank

    scratch = torch.empty(world * 32, dtype=torch.uint8, device=dev)
    for _ in range(args.warmup):
        step(scratch)
    torch.cuda.synchronize()
    launches_per_step = q.last_launch_count()
    gathered = [torch.empty(world * 32, dtype=torch.uint8, device=dev) for _ in range(args.steps)]
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    props = torch.cuda.get_device_properties(dev)
    gpu_id = f"GPU-{props.uuid}" if getattr(props, "uuid", None) else str(local)
    kernel_ms = []
    dist.barrier()
    torch.cuda.synchronize()
    sampler = ClockSampler(gpu_id)
    time.sleep(0.3)
    for i in range(args.steps):
        flush.fill_(i & 0xFF)
        starts[i].record(stream)
        step(gathered[i])
        ends[i].record(stream)
        kernel_ms.append(q.kernel_time_ms())
    torch.cuda.synchronize()
    dist.barrier()
    clocks = sampler.stop()
    ms = sum(s.elapsed_time(e) for s, e in zip(starts, ends)) / args.steps
    kern = sum(kernel_ms) / len(kernel_ms)
    checks = {}
    for i, g in enumerate(gathered):
        e, r, t = combine_gathered(g.cpu().numpy().tobytes(), world, q.RESULT_DTYPE)
        checks["sharded_step"] = check_result("n40_int32", e, r, t)

    # end to end through the public sharded API: host Q per rank, host result, one all-gather
    qd.solve_distributed(Q, SHARD_K)
    e2e_ms = []
    for i in range(args.steps):
        flush.fill_(i & 0xFF)
        torch.cuda.synchronize()
        dist.barrier()
        t0 = time.perf_counter()
        he, hx, ht = qd.solve_distributed(Q, SHARD_K)
        e2e_ms.append((time.perf_counter() - t0) * 1e3)
    e2e = sum(e2e_ms) / len(e2e_ms)
    checks["solve_distributed"] = check_result("n40_int32", he, int("".join(map(str, hx)), 2), ht)
    ms, e2e, kern_max = max_over_ranks([ms, e2e, kern], dev)
    rank_states = count << (N - SHARD_K)
    achieved = rank_states / (kern * 1e-3) / 1e12
    peak = SMS * LANES_PER_CLK * MAX_SM_MHZ * 1e6 / 1e12
    if rank == 0:
        cfg = config_dict()
        cfg.update({"parallelism": f"slice shards x{world}", "shard_k_prefix": SHARD_K,
                    "slices_per_rank": count})
        line = {
            "metric": METRIC, "value": STATES / (ms * 1e-3), "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "strong",
            "vs_baseline": None, "dtype": "int32", "data": "synthetic (seeded uniform integers, no dataset)",
            "config": cfg,
            "result": {"min_energy": float(he), "argmin_rank": int("".join(map(str, hx)), 2), "tie_count": int(ht),
                       "checks": checks},
            "roofline": {"bound": "alu", "achieved": achieved, "peak": peak, "unit": "Tops/s (int32 lane-ops)",
                         "frac": achieved / peak, "traffic": None,
                         "kernel": "search_kernel<16,R,min,biased,bounded> on rank 0's shard", "kernel_ms": kern,
                         "kernel_ms_max_over_ranks": kern_max,
                         "peak_basis": "152 SMs x 128 lanes/clk x 2.07 GHz max SM clock"},
            "e2e": {"value": STATES / (e2e * 1e-3), "unit": UNIT, "h2d_bytes_per_step": world * N * N * 4,
                    "d2h_bytes_per_step": world * 32, "ms_per_step": e2e,
                    "api": "exact_qubo_exhaustive_gb300.distributed.solve_distributed"},
            "cpu_baseline": None,
            "gpu_launches": launches_per_step * args.steps,
            "clocks": clocks,
        }
        print(json.dumps(line), flush=True)
    dist.destroy_process_group()
    return 0


def other_configs(q, torch, dev, stream):
    """Device-timed rates of the other workloads (one timed run each, for context)."""
    out = {}

    def timed(fn, reps=3):
        fn()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(reps):
            fn()
        e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / reps

    for name, n, Q, dt in (("n40_narrow_int32", 40, qi.workload_n40_narrow(), q.INT32),
                           ("n36_fp32", 36, qi.workload_n36_f32(), q.FP32),
                           ("n36_wide_int32", 36, qi.workload_n36_wide(), q.INT32),
                           ("n32_int32", 32, qi.workload_n32(), q.INT32),
                           ("n32_mattis_int32", 32, qi.workload_n32_mattis()[0], q.INT32),
                           ("n20_int32", 20, qi.workload_n20(), q.INT32)):
        dq = torch.from_numpy(Q).to(dev)
        nb = q.workspace_bytes(n, dt)
        ws = torch.empty(nb, dtype=torch.uint8, device=dev)
        res = torch.zeros(32, dtype=torch.uint8, device=dev)
        ms = timed(lambda: q.solve_device(n, dq, dt, ws, nb, stream.cuda_stream, res))
        kern = q.kernel_time_ms()
        out[name] = {"ms": ms, "states_per_s": (1 << n) / (ms * 1e-3), "min_pass_ms": kern,
                     "min_pass_states_per_s": (1 << n) / (kern * 1e-3) if kern > 0 else None}
        if name in ("n36_fp32", "n36_wide_int32", "n40_narrow_int32"):
            r = np.frombuffer(res.cpu().numpy().tobytes(), dtype=q.RESULT_DTYPE)[0]
            tol = 1e-3 * float(np.abs(Q.astype(np.float64)).sum()) * 2.0 ** -20 if dt == q.FP32 else 0.0
            out[name]["check"] = check_result(name, float(r["min_energy"]), int(r["argmin_rank"]),
                                              int(r["tie_count"]), tol)
        if name == "n40_narrow_int32":
            out[name]["workload"] = ("n=40 dense QUBO, int32 upper-triangular, entries uniform in [-4,4] "
                                     "(sum |U| = 1822: the packed 16x2 pass with block bounds)")
        if name == "n36_wide_int32":
            out[name]["workload"] = ("n=36 dense QUBO, int32 upper-triangular, entries uniform in "
                                     "[-2^20, 2^20] (sum |U| ~ 3.5e8 > 2^22: the int32 minimum pass)")
    # the minimum passes without block bounds, on the n=40 workloads (same results)
    q.enable_block_bounds(False)
    try:
        for name, Q in (("n40_int32_without_bounds", qi.workload_n40()),
                        ("n40_narrow_int32_without_bounds", qi.workload_n40_narrow())):
            dq = torch.from_numpy(Q).to(dev)
            nb = q.workspace_bytes(40, q.INT32)
            ws = torch.empty(nb, dtype=torch.uint8, device=dev)
            res = torch.zeros(32, dtype=torch.uint8, device=dev)
            ms = timed(lambda: q.solve_device(40, dq, q.INT32, ws, nb, stream.cuda_stream, res), reps=2)
            kern = q.kernel_time_ms()
            out[name] = {"ms": ms, "states_per_s": (1 << 40) / (ms * 1e-3), "min_pass_ms": kern,
                         "pass": "biased fp32-binade pass" if "narrow" not in name else "packed 16x2 pass"}
            r = np.frombuffer(res.cpu().numpy().tobytes(), dtype=q.RESULT_DTYPE)[0]
            out[name]["check"] = check_result(name.replace("_without_bounds", ""), float(r["min_energy"]),
                                              int(r["argmin_rank"]), int(r["tie_count"]))
    finally:
        q.enable_block_bounds(True)
    # k lowest energies of the n=40 workload through the host entry point (wall clock)
    Q40 = qi.workload_n40()
    q.solve_lowest(Q40, 1024)
    t0 = time.perf_counter()
    reps = 2
    for _ in range(reps):
        e40, _ = q.solve_lowest(Q40, 1024)
    wall = (time.perf_counter() - t0) * 1e3 / reps
    out["n40_lowest_k1024_int32"] = {"ms": wall, "states_per_s": (1 << 40) / (wall * 1e-3),
                                     "e_first": int(e40[0]), "e_last": int(e40[-1]),
                                     "timing": "host call, wall clock (includes H2D, passes, D2H, host sort)"}
    # long-run driver: n=42 in 8 checkpointed chunks of 32 slices against one uninterrupted call
    import tempfile
    Q42 = qi.random_upper_int(42, -1000, 1000, qi.MASTER_SEED + 6)
    q.solve(Q42)
    t0 = time.perf_counter()
    one = q.solve(Q42)
    t_one = (time.perf_counter() - t0) * 1e3
    with tempfile.TemporaryDirectory() as td:
        t0 = time.perf_counter()
        ck = q.solve_checkpointed(Q42, 8, os.path.join(td, "n42.ckpt"), slices_per_chunk=32)
        t_ck = (time.perf_counter() - t0) * 1e3
    out["n42_checkpointed_8_chunks_int32"] = {"ms": t_ck, "states_per_s": (1 << 42) / (t_ck * 1e-3),
                                              "uninterrupted_ms": t_one, "same_result": ck[1] == one[0] and ck[3] == one[2],
                                              "timing": "host calls, wall clock"}
    Qs = qi.workload_batched()
    dq = torch.from_numpy(Qs).to(dev)
    nb = max(q.batched_workspace_bytes(4096, 24), 256)
    ws = torch.empty(nb, dtype=torch.uint8, device=dev)
    res = torch.zeros(4096 * 32, dtype=torch.uint8, device=dev)
    ms = timed(lambda: q.solve_batched_device(4096, 24, dq, ws, nb, stream.cuda_stream, res))
    out["batched_4096x_n24_int32"] = {"ms": ms, "states_per_s": 4096 * (1 << 24) / (ms * 1e-3)}
    return out


def profile_batched(batch: int):
    """Two batched searches of the 4096 x n=24 workload's shape (first `batch` instances), for ncu."""
    import torch
    import exact_qubo_exhaustive_gb300 as q
    Qs = qi.workload_batched()[:batch]
    dq = torch.from_numpy(np.ascontiguousarray(Qs)).cuda()
    nb = max(q.batched_workspace_bytes(batch, 24), 256)
    ws = torch.empty(nb, dtype=torch.uint8, device="cuda")
    res = torch.zeros(batch * 32, dtype=torch.uint8, device="cuda")
    s = torch.cuda.current_stream()
    for _ in range(2):
        q.solve_batched_device(batch, 24, dq, ws, nb, s.cuda_stream, res)
    torch.cuda.synchronize()
    r = np.frombuffer(res.cpu().numpy().tobytes(), dtype=q.RESULT_DTYPE)
    log(f"profile batched {batch} x n=24: statuses ok={int((r['status'] == 0).sum())} E0={r['min_energy'][0]}")
    return 0 if (r["status"] == 0).all() else 1


def profile_case(n: int, dtype_name: str):
    """Two searches of an n-variable instance shaped like the workload (for ncu captures)."""
    import torch
    import exact_qubo_exhaustive_gb300 as q
    if dtype_name == "fp32":
        Q, dt = qi.random_symmetric_normal_f32(n, qi.MASTER_SEED + 3), q.FP32
    elif dtype_name == "int32_narrow":
        Q, dt = qi.random_upper_int(n, -4, 4, qi.MASTER_SEED + 5), q.INT32
    elif dtype_name == "int32_wide":
        Q, dt = qi.random_upper_int(n, -(1 << 20), 1 << 20, qi.MASTER_SEED + 7), q.INT32
    else:
        Q, dt = qi.random_upper_int(n, -1000, 1000, qi.MASTER_SEED + 2), q.INT32
    dq = torch.from_numpy(Q).cuda()
    nb = q.workspace_bytes(n, dt)
    ws = torch.empty(nb, dtype=torch.uint8, device="cuda")
    res = torch.zeros(32, dtype=torch.uint8, device="cuda")
    s = torch.cuda.current_stream()
    for _ in range(2):
        q.solve_device(n, dq, dt, ws, nb, s.cuda_stream, res)
    torch.cuda.synchronize()
    r = np.frombuffer(res.cpu().numpy().tobytes(), dtype=q.RESULT_DTYPE)[0]
    log(f"profile case n={n} {dtype_name}: plan={q.plan(n, dt)} result={r}")
    return 0 if int(r["status"]) == 0 else 1


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["gb300", "reference"], default="gb300")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU oracle baseline")
    ap.add_argument("--no-extra", action="store_true", help="skip the other workloads")
    ap.add_argument("--sharded", action="store_true",
                    help="time the slice-sharded search (the N > 1 path) even with one rank (run under torchrun)")
    ap.add_argument("--profile-case", type=int, default=0, metavar="N",
                    help="only run two searches of an N-variable instance (for ncu), print no JSON")
    ap.add_argument("--profile-dtype", choices=["int32", "fp32", "int32_narrow", "int32_wide"], default="int32")
    ap.add_argument("--oracle-configs", type=float, default=0.0, metavar="SECONDS",
                    help="time the CPU oracle on every workload (one core and all cores) and exit")
    ap.add_argument("--profile-batched", type=int, default=0, metavar="B",
                    help="run two batched searches of the first B instances of the batched workload (for ncu)")
    args = ap.parse_args(argv)
    if args.profile_case:
        return profile_case(args.profile_case, args.profile_dtype)
    if args.profile_batched:
        return profile_batched(args.profile_batched)
    if args.oracle_configs:
        print(json.dumps(oracle_configs(args.oracle_configs)))
        return 0
    if args.warmup < 3:
        log("warmup raised to 3 (timing rule)")
        args.warmup = 3
    if args.impl == "reference":
        return run_reference(args)
    try:
        return run_gb300(args)
    except ResultMismatch as exc:
        log(f"RESULT MISMATCH: {exc}")
        return 1


if __name__ == "__main__":
    sys.exit(main())
