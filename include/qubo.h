/*
 * qubo.h -- C ABI of the GB300 exhaustive QUBO solver.
 *
 * The library finds, for a dense QUBO matrix Q (n x n, row-major),
 *     E_min = min over x in {0,1}^n of E(x) = sum_{i,j} Q_ij x_i x_j
 * (Terastate-per-second QUBO Brute-Force on a Single GPU, §I objective), the minimiser with the
 * lowest rank, rank(x) = sum_i x_i 2^(n-1-i) (x_0 is the most significant bit: the lexicographic
 * order of the state space U_N in §II-B, Fig. 2), and the number of states attaining E_min.
 * Every one of the 2^n states is visited: the search is the prefix-suffix decomposition of
 * §II-A..C (eq. 4 and 8) walked in Gray-code order (§III-B, Algorithm 2, eq. 9), split into
 * independent fixed-prefix subproblems (§III-C1) and cached column segments (§III-C2), and every
 * state's column energy gets its one add (eq. 9). The comparison of a state's energy with the
 * minimum is left out only for blocks of Gray steps whose lower bound proves that none of their
 * states reaches the best energy found so far (block bounds, see qubo_enable_block_bounds); the
 * results are exactly those of comparing every state.
 *
 * Conventions for every entry point:
 *  - Q is read only during the call; the caller owns all buffers; the library keeps no pointer.
 *  - Q need not be triangular: E sums over all i, j. Internally Q is folded to the upper
 *    triangle U_ii = Q_ii, U_ij = Q_ij + Q_ji (i < j), the form §II-A assumes.
 *  - dtype QUBO_INT32: results are exact. The call fails with QUBO_ERR_RANGE unless
 *    S = sum_{i<=j} |U_ij| <= 2^30 - 1 (every partial energy the kernels form is a sum of at
 *    most two sub-sums of U, so int32 arithmetic never overflows).
 *  - dtype QUBO_FP32: the energy of a state is the fp64 sum of the fp64-folded triangle in fixed
 *    order (i ascending, j >= i ascending). The search runs on an exact int32 fixed-point image
 *    of U with a proven error band, and every state inside the band is re-evaluated in fp64, so
 *    the returned minimiser is the exact fp64 minimiser (lowest rank among equal fp64 values).
 *    Non-finite entries fail with QUBO_ERR_NONFINITE.
 *  - dtype QUBO_FP64: as QUBO_FP32 with fp64 entries (8 bytes each); the fold and every energy
 *    are the same fp64 operations. The batched entry points take int32 only.
 *  - out_min_energy receives E_min (exact for int32), out_argmin_x[n] receives x in {0,1}
 *    (x_0 first), out_tie_count the number of minimisers (for fp32: states with fp64 energy
 *    equal to E_min). On error no output is written.
 *  - n must be in [1, 62]. k_prefix <= 0 and cache_bits <= 0 select the planner's choice;
 *    explicit values that the kernels cannot run return QUBO_ERR_PLAN.
 *  - Host entry points block until the result is on the host. Calls are serialised internally.
 */
#ifndef QUBO_GB300_H
#define QUBO_GB300_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define QUBO_API __attribute__((visibility("default")))
#else
#define QUBO_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* dtype codes */
#define QUBO_INT32 0
#define QUBO_FP32 1
#define QUBO_FP64 2 /* fp64 input: the same fp64 semantics as QUBO_FP32, without the input rounding */

/* status codes (0 or negative) */
#define QUBO_OK 0
#define QUBO_ERR_ARG (-1)       /* n out of range, null pointer, bad dtype, bad slice id */
#define QUBO_ERR_RANGE (-2)     /* int32: S = sum |U_ij| > 2^30 - 1. Why 2^30 and not 2^31: §IV-B.5 keeps
                                   every intermediate inside the integer type; besides sub-sums of U
                                   (|v| <= S) the kernels form the difference of the running best and
                                   a unit's offset, two sub-sums, so |v| <= 2S, and 2S < 2^31 needs
                                   S <= 2^30 - 1. */
#define QUBO_ERR_NONFINITE (-3) /* fp32/fp64: NaN or Inf in Q */
#define QUBO_ERR_PLAN (-4)      /* explicit k_prefix / cache_bits the kernels cannot run */
#define QUBO_ERR_CUDA (-5)      /* a CUDA call failed (message via qubo_last_error) */
#define QUBO_ERR_NODEV (-6)     /* no CUDA device */
#define QUBO_ERR_ABORTED (-7)   /* the call was cancelled by qubo_request_abort() */
#define QUBO_ERR_CHECKPOINT (-8) /* checkpoint file unreadable, corrupt, or of another problem */
#define QUBO_INCOMPLETE 1        /* not an error: a time budget ended the call, progress is saved */

/* Device-side result record: one per solved problem (or slice). */
typedef struct qubo_result {
  int32_t status;       /* QUBO_OK or an error code found on the device */
  int32_t reserved;
  double min_energy;    /* E_min (int32: exact integer; fp32: fp64 energy of argmin) */
  uint64_t argmin_rank; /* rank of the lowest-rank minimiser; bit n-1-i is x_i */
  uint64_t tie_count;   /* number of minimisers */
} qubo_result;

/* Planner decision, for inspection and tests. */
typedef struct qubo_plan_desc {
  int n, dtype;
  int k_prefix;        /* fixed variables per work unit (slice bits) */
  int cache_bits;      /* cached variables: 2^cache_bits columns held on chip */
  int walked_bits;     /* Gray-walked variables per unit: n - k_prefix - cache_bits */
  int register_bits;   /* walked variables whose rows live in registers */
  int columns_per_thread;
  int threads_per_block;
  int blocks;          /* persistent grid */
  int variant;         /* 0 = generic kernel, 1 = register-cached fast kernel */
  uint64_t units;      /* work units (fixed prefixes) per call */
  size_t workspace_bytes;
  size_t smem_bytes;
  int packed;          /* 1: int32 input whose sum |U_ij| <= 2^14 - 1 runs the minimum pass with two
                          16-bit energies per 32-bit word (§IV-B.5's narrow path); planned only
                          where block bounds are off (qubo_enable_block_bounds) */
  int biased;          /* 1: the minimum pass adds columns as fp32 numbers in the exact binade
                          [2^23, 2^24): int32 input whose sum |U_ij| <= 2^22 - 1, and fp32 input
                          (its fixed-point image is scaled into that range); n >= 30 */
  int pruned;          /* 1: the minimum pass (biased fp32 columns, or int32 columns where sum
                          |U_ij| is too large for them) forms its per-step minima only in blocks of
                          2^6 or 2^7 Gray steps (2^7 from 12 walked bits on) whose lower bound does
                          not clear the best energy found so far (every state is still added;
                          results are unchanged) */
} qubo_plan_desc;

/* Minimise one QUBO. Q is a HOST pointer to n*n int32, fp32 or fp64 values (row-major).
 * (Algorithm 2 of §III-B with the §III-C1 split; inputs Q, A/B sizes; outputs x_opt, E_min.) */
QUBO_API int qubo_solve(int n, const void* Q, int dtype, int k_prefix, int cache_bits, double* out_min_energy,
               uint8_t* out_argmin_x, uint64_t* out_tie_count);

/* Minimise over selected slices only: slice s fixes x_0..x_{k-1} to the bits of slice_ids[s]
 * (bit k-1-f is x_f), k = k_prefix >= 1 (§III-C1: each fixed prefix is an independent
 * subproblem). Writes one result per slice: out_min_energy[num_slices],
 * out_argmin_x[num_slices * n] (full-length states), out_tie_count[num_slices]. */
QUBO_API int qubo_solve_slices(int n, const void* Q, int dtype, int k_prefix, int cache_bits,
                      const uint64_t* slice_ids, int num_slices, double* out_min_energy,
                      uint8_t* out_argmin_x, uint64_t* out_tie_count);

/* Minimise over the contiguous slice range [first_slice, first_slice + num_slices) of k_prefix
 * bits as ONE problem (one result). This is the shard a process solves when the 2^k_prefix
 * slices are split across devices; the shard results combine by (min energy, then min rank,
 * summed ties). */
QUBO_API int qubo_solve_slice_range(int n, const void* Q, int dtype, int k_prefix, int cache_bits,
                           uint64_t first_slice, uint64_t num_slices, double* out_min_energy,
                           uint8_t* out_argmin_x, uint64_t* out_tie_count);

/* Batched mode: `batch` independent problems of equal size n, Q = batch consecutive n*n
 * matrices (host pointer). §III-C1: the search splits into independent subproblems, each solved
 * by Algorithm 2 (§III-B); here every instance is one such problem and instances share no state.
 * Small instances run one thread block per instance; 18 <= n <= 32 splits each instance into
 * work units of the same persistent passes as qubo_solve. Outputs are per problem:
 * out_min_energy[batch], out_argmin_x[batch * n], out_tie_count[batch]. int32 only; an instance
 * whose range check fails makes the call return its status (QUBO_ERR_RANGE). */
QUBO_API int qubo_solve_batched(int batch, int n, const void* Q, int dtype, double* out_min_energy,
                       uint8_t* out_argmin_x, uint64_t* out_tie_count);

/* ---- device-resident entry points (PyTorch or the caller owns memory and streams) ----
 * The same searches as the host entry points: Algorithm 2 of §III-B with the §III-C1 split
 * (inputs Q, A/B sizes; outputs x_opt, E_min, plus the tie count), with every buffer in device
 * memory owned by the caller.
 * d_Q: DEVICE pointer to the input; d_workspace: device buffer of at least the size the
 * matching *_workspace_bytes call returns (256-byte aligned); cuda_stream: a cudaStream_t
 * (NULL = legacy default stream). The call only enqueues work and returns; d_result is
 * written on the stream (status included: range and finiteness errors are found on the device
 * and reported there). Host-detectable errors (arguments, plan, abort) are returned directly,
 * before anything is enqueued. qubo_workspace_bytes returns 0 for arguments it cannot plan. */
QUBO_API size_t qubo_workspace_bytes(int n, int dtype, int k_prefix, int cache_bits);
QUBO_API int qubo_solve_device(int n, const void* d_Q, int dtype, int k_prefix, int cache_bits, void* d_workspace,
                      size_t workspace_bytes, void* cuda_stream, qubo_result* d_result);

/* Search without any allocation, for callers that cannot call cudaMalloc when they need a result
 * (a latency-critical loop that cannot afford cudaMalloc's device-wide synchronisation, or a
 * plug-in inside a framework that owns all device memory and gives out no workspace). The paper
 * has no counterpart: this is a deployment variant of qubo_solve_device with the same arguments
 * minus the workspace. Scratch memory is one file-scope device array of
 * QUBO_NO_ALLOC_SCRATCH_BYTES that every GPU loading the library keeps until exit; problems
 * whose workspace (qubo_workspace_bytes) exceeds it return QUBO_ERR_ARG. The first call in each
 * CUDA context looks the array's device address up (cudaGetSymbolAddress) and keeps it with the
 * context's unique id, so a call from another context (after cudaDeviceReset, or under a context
 * made with the driver API) looks it up again; make the first call in a context before any
 * stream capture. All calls share the array and it keeps the last call's contents; every call
 * rewrites everything it reads, so nothing needs clearing. Calls that overlap on the GPU race on
 * the array: order them on one stream. No cudaMalloc, cudaFree or allocating routine is called.
 * A pending qubo_request_abort() refuses the call (QUBO_ERR_ABORTED) before any device work.
 * d_Q, d_result: device pointers; cuda_stream: a cudaStream_t (NULL = legacy stream);
 * asynchronous like qubo_solve_device. */
#define QUBO_NO_ALLOC_SCRATCH_BYTES (8u << 20)
QUBO_API int qubo_solve_device_no_alloc(int n, const void* d_Q, int dtype, int k_prefix, int cache_bits,
                                        void* cuda_stream, qubo_result* d_result);

/* Device-resident form of qubo_solve_slice_range (one result over a contiguous slice range). */
QUBO_API size_t qubo_slice_range_workspace_bytes(int n, int dtype, int k_prefix, int cache_bits, uint64_t num_slices);
QUBO_API int qubo_solve_slice_range_device(int n, const void* d_Q, int dtype, int k_prefix, int cache_bits,
                                           uint64_t first_slice, uint64_t num_slices, void* d_workspace,
                                           size_t workspace_bytes, void* cuda_stream, qubo_result* d_result);

QUBO_API size_t qubo_batched_workspace_bytes(int batch, int n, int dtype);
QUBO_API int qubo_solve_batched_device(int batch, int n, const void* d_Q, int dtype, void* d_workspace,
                              size_t workspace_bytes, void* cuda_stream, qubo_result* d_results);

/* ---- long runs: checkpoint / resume ----
 * §III-C1 / §IV-C: the 2^k_prefix slices (fixed first k_prefix variables) are independent, so a
 * long search can stop between slices and continue later. qubo_solve_checkpointed processes the
 * slices in ascending order, `slices_per_chunk` at a time (0: about 2^44 states per chunk), each
 * chunk as one qubo_solve_slice_range call, and after every chunk rewrites the checkpoint file
 * at `checkpoint_path` (written to "<path>.tmp", then renamed over it). The file holds the
 * problem's identity (n, dtype, k_prefix, a 64-bit FNV-1a hash of Q's bytes), the next slice and
 * the combined record so far (lowest energy; among equal energies the lowest rank and the summed
 * tie count). If the file exists when the call starts, the call resumes from it; a file of
 * another problem, or a corrupt one, gives QUBO_ERR_CHECKPOINT and is left untouched.
 * time_budget_s > 0: no new chunk starts once that many seconds have passed since the call
 * began (at least one chunk runs per call). Returns QUBO_OK when every slice is done
 * (out_* hold the final result, exactly as qubo_solve would give), or QUBO_INCOMPLETE with the
 * record over the slices done so far in out_* and their number in *out_slices_done. A
 * qubo_request_abort() stops between chunks with QUBO_ERR_ABORTED (progress up to the last
 * chunk is saved). 1 <= k_prefix < n. Other arguments and errors as qubo_solve_slice_range. */
QUBO_API int qubo_solve_checkpointed(int n, const void* Q, int dtype, int k_prefix, int cache_bits,
                                     uint64_t slices_per_chunk, const char* checkpoint_path, double time_budget_s,
                                     double* out_min_energy, uint8_t* out_argmin_x, uint64_t* out_tie_count,
                                     uint64_t* out_slices_done);

/* Reads a checkpoint file (progress monitoring): problem identity, progress and the record so far
 * (*out_have = 0 before the first chunk finished). QUBO_ERR_CHECKPOINT if unreadable or corrupt;
 * QUBO_ERR_ARG for a null pointer. */
QUBO_API int qubo_checkpoint_read(const char* checkpoint_path, int* out_n, int* out_dtype, int* out_k_prefix,
                                  uint64_t* out_q_hash, uint64_t* out_next_slice, uint64_t* out_total_slices,
                                  int* out_have, double* out_min_energy, uint64_t* out_argmin_rank,
                                  uint64_t* out_tie_count);

/* 64-bit FNV-1a hash of `bytes` bytes (the problem identity stored in checkpoint files). */
QUBO_API uint64_t qubo_fnv1a64(const void* data, size_t bytes);

/* ---- low-energy spectrum ----
 * The k lowest energies (§I: the search sees every state, so it can return the low-energy
 * spectrum, not only the minimum). Result: the min(k, 2^n) states with the smallest keys
 * (E(x), rank(x)), in ascending order -- energies ascending, equal energies by rank -- so it is
 * unique whatever the decomposition. out_energies[k] receives the energies (exact), out_x[k * n]
 * the states (x_0 first), *out_count the number written. int32 input only (QUBO_ERR_ARG for other
 * dtypes); 1 <= k <= QUBO_LOWEST_MAX_K. Q is a host pointer as for qubo_solve. The call runs the
 * minimum pass, then re-walks only the units that can hold one of the k states (more passes
 * only for very degenerate spectra). It allocates its device memory per call. */
#define QUBO_LOWEST_MAX_K (1 << 20)
QUBO_API int qubo_solve_lowest(int n, const void* Q, int dtype, int k_prefix, int cache_bits, int k,
                               double* out_energies, uint8_t* out_x, int* out_count);

/* ---- Ising input ----
 * §I: the Ising form with spins s in {-1,+1} and the QUBO form are the same problem under
 * s = 2x - 1. Convention: H(s) = sum_{i,j} J_ij s_i s_j + sum_i h_i s_i over all i, j (only
 * J_ij + J_ji matters off the diagonal; J_ii adds the constant J_ii). J is n*n row-major, h has n
 * entries or is NULL (zero field); both have the element type of dtype.
 *
 * qubo_ising_to_qubo: the exact equivalent QUBO, upper triangular, and the offset C with
 * H(s) = E_Q(x) + C for x = (s + 1) / 2:
 *   Q_ij = 4 (J_ij + J_ji) (i < j),  Q_ii = 2 h_i - 2 sum_{j != i} (J_ij + J_ji),
 *   C = sum_{i<j} (J_ij + J_ji) - sum_i h_i + sum_i J_ii.
 * dtype QUBO_INT32: out_Q receives n*n int32 (computed in int64; QUBO_ERR_RANGE if an entry
 * leaves int32); C is exact. QUBO_FP32 / QUBO_FP64: out_Q receives n*n fp64 computed in fp64
 * (fixed order); non-finite input or output gives QUBO_ERR_NONFINITE. */
QUBO_API int qubo_ising_to_qubo(int n, const void* J, const void* h, int dtype, void* out_Q, double* out_offset);

/* Minimise H(s) over all 2^n spin states: converts as above and runs qubo_solve (int32 input
 * stays int32; fp32/fp64 input is searched as the fp64 QUBO). out_min_H = E_min + C (exact for
 * int32), out_argmin_s[n] in {-1,+1} is the ground state whose bit vector x = (s + 1) / 2 has the
 * lowest rank, out_tie_count the number of ground states. Errors as qubo_solve; outputs are
 * untouched on error. */
QUBO_API int qubo_solve_ising(int n, const void* J, const void* h, int dtype, int k_prefix, int cache_bits,
                              double* out_min_H, int8_t* out_argmin_s, uint64_t* out_tie_count);

/* Planner decision for qubo_solve(n, ., dtype, k_prefix, cache_bits) on the current device. */
QUBO_API int qubo_plan(int n, int dtype, int k_prefix, int cache_bits, qubo_plan_desc* out);

/* Kernel timing (measurement): while enabled, every search call records two CUDA events on its
 * stream, around its enumeration (minimum-pass) launches. qubo_kernel_time_ms() waits for the
 * second event and returns the elapsed milliseconds of the most recent call (-1 when disabled or
 * nothing was recorded). Not thread-safe with concurrent device-resident calls. */
QUBO_API void qubo_enable_kernel_timing(int enable);
QUBO_API double qubo_kernel_time_ms(void);

/* Block bounds in the single-problem minimum pass (on by default). They are this library's
 * addition to the paper's walk (Terastate-per-second QUBO Brute-Force on a Single GPU, Alg. 2 and
 * eq. 9), which is otherwise unchanged: every state is still added, and blocks of Gray steps whose
 * lower bound clears the best energy found so far skip their per-step minima. With 0, calls
 * planned from then on take minimum passes that form every step's minimum: the packed 16x2 pass
 * for int32 input with sum |U| < 2^14, the biased fp32-binade pass without bounds up to 2^22,
 * the int32 pass without bounds above.
 * Results are identical either way; the switch exists to test and measure each pass.
 * Process-wide, read when a call is planned (qubo_plan reports it in `pruned`); calls already
 * planned are not affected. In the batched calls it applies to the packed pass (instances with
 * sum |U| < 2^14); their other passes have no bounds. */
QUBO_API void qubo_enable_block_bounds(int enable);

/* Number of kernel launches the last host or device call enqueued. */
QUBO_API int qubo_last_launch_count(void);

/* Text for a status code; the last CUDA error text for QUBO_ERR_CUDA. The paper defines no status
 * codes: these are this library's own. The returned strings are static (never freed); the
 * last-error text is overwritten by the next failing call. */
QUBO_API const char* qubo_status_string(int status);
QUBO_API const char* qubo_last_error(void);

/* Cancellation: a host flag checked between kernel launches of the current and later calls
 * (never polled inside a kernel). qubo_clear_abort() re-arms. */
QUBO_API void qubo_request_abort(void);
QUBO_API void qubo_clear_abort(void);

/* ---- measurement ----
 * ALU throughput microbenchmark on the current device: runs `iters` iterations of 16
 * independent chains of one operation per thread on every SM and reports warp-lane
 * operations per second and the SM clock seen by the kernel (clock64 / globaltimer).
 * kind: 0 int32 add, 1 int32 min, 2 int32 3-input min, 3 int32 add-then-min (fused),
 *       4 fp32 add, 5 fp32 min, 6 packed 16x2 3-input min, 7 packed 16x2 add-then-min,
 *       8 int32 add with half of the adds issued as integer multiply-adds by one (FMA pipe),
 *       9 packed fp32x2 add (two adds per instruction; counted as two operations),
 *       10 int32 add as a fused add-min against an opaque INT_MAX (ALU; cannot be merged),
 *       11 int32 add as a multiply-add by an opaque one (FMA pipe; cannot be merged),
 *       12 / 14 / 15: 11 / 10 / 12 of the 16 chains fp32 adds, the rest kind-10 adds,
 *       13: 8 chains kind 11, 8 chains kind 10,
 *       16 fp32 add / subtract of loop-invariant addends into 16 accumulators (the column-update
 *          pattern of the enumeration walk),
 *       17 / 18: 12 / 10 of the 16 chains as fp32x2 adds (two adds per instruction), the rest
 *          kind-10 adds (counted per add). */
QUBO_API int qubo_probe_alu(int kind, int iters, double* out_ops_per_s, double* out_sm_mhz);

#ifdef __cplusplus
}
#endif

#endif /* QUBO_GB300_H */
