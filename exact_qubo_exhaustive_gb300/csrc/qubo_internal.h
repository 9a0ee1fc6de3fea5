// Internal declarations shared by the library's translation units (not part of the C ABI).
#pragma once

#include <cuda_runtime.h>

#include <mutex>

#include <cstddef>
#include <cstdint>

#include "../../include/qubo.h"

namespace qgb {

// Largest sum of |U_ij| the int32 search accepts: every value a kernel forms is a sub-sum of U
// or the difference of two sub-sums, so |value| <= 2 * S <= 2^31 - 2 stays in int32.
constexpr int64_t kMaxAbsSum = (int64_t(1) << 30) - 1;

// Kernel variants.
enum Variant : int {
  kGeneric = 0,  // one column per thread, every walked row in shared memory
  kFast = 1,     // 16 columns per thread, the lowest kFastR walked rows in registers
};
constexpr int kFastCPT = 16;
constexpr int kFastThreadsMax = 256;  // 2^C / kFastCPT for C <= 12
// static shared memory of the fast resolve passes: one scan slot of kFastCPT ints per thread
constexpr size_t kFastScanSlotBytes = (size_t)kFastThreadsMax * kFastCPT * 4;
constexpr int kFastR = 4;
constexpr int kBiasedR = 5;  // register rows of the biased-binade minimum pass
constexpr int kPackedR = 5;  // register rows of the packed 16x2 minimum pass
constexpr int kIntMinR = 5;  // register rows of the int32 minimum pass (the resolve passes keep kFastR)
// Register rows of the block-bounded minimum passes, which walk blocks of 2^R Gray steps: R = 7
// for units of at least kPruneLongW walked bits, R = 6 below (the longer block body pays off
// only when a unit has many blocks). Measured per minimum pass at 12 walked bits, R = 7 against
// R = 6: int32 columns 2.45 against 3.01 ms (n=36), fp32 columns 2.006 against 2.015 ms (n=36)
// and 0.568 against 0.554 ms (n=34); at 10 walked bits (n=32) R = 6 is the faster (0.223 against
// 0.271 ms, fp32 columns).
constexpr int kPruneRShort = 6;
constexpr int kPruneRLong = 7;
constexpr int kPruneLongW = 12;
constexpr int kGenericMaxC = 10;  // 2^C threads per block
constexpr int kMaxWalkedBits = 24;

// Biased fp32 minimum walk: every running column energy is a sum of distinct U entries, so
// |V| <= sum |U| < 2^22 keeps 1.5 * 2^23 + V inside the binade [2^23, 2^24).
constexpr int64_t kBiasedWalkMaxAbsSum = (int64_t(1) << 22) - 1;
// Packed 16x2 minimum walk: column energies within sum |U| and (best - offset) within 2 sum |U|
// stay inside (-2^15, 2^15) when sum |U| < 2^14.
constexpr int64_t kPackedMaxAbsSum = (int64_t(1) << 14) - 1;

// Per block of 2^R Gray steps (block-bounded minimum pass): the block's least walked
// energy and the shared-row flip that follows it, precomputed once per launch (the same for every
// unit): the row's float4 offset in shared memory, its sign (+1 sets the variable, -1 clears it,
// 0 after the last block: no flip) and the index of its signed linear term in the walker's
// table of +L, -L and a zero.
struct alignas(16) BlockCtl {
  int32_t tmin;
  int32_t row;
  float dsgn;
  int32_t lvx;
};

// Written by the device, read back by the host (lives at the start of the workspace).
struct DevHeader {
  int32_t status;      // QUBO_OK or an error code found on the device
  int32_t scale_exp;   // fp32 path: U32 = round(U64 * 2^scale_exp)
  int32_t band;        // candidates: energy <= group minimum + band (int32 units)
  uint32_t tied_count; // number of entries in the tied-unit list
  int64_t abs_sum;     // sum |U_ij| of the int32 image
  double abs_sum64;    // fp32 path: sum |U_ij| in fp64
  int32_t pad[8];
};

// One state found by the k-lowest passes: its energy and rank.
struct KeyCand {
  int32_t e;
  int32_t pad;
  uint64_t rank;
};

// Host-side plan (one call).
struct Plan {
  int n = 0, dtype = 0;
  int variant = kGeneric;
  int C = 0;       // cached bits
  int F = 0;       // fixed bits per work unit
  int w = 0;       // walked bits = n - F - C
  int R = 0;       // register-row bits of the variant
  int cpt = 1;     // columns per thread
  int threads = 32;
  int blocks = 1;
  int seg_bits = 0;        // resolve: segments per tied unit = 2^seg_bits
  int ngroups = 1;
  uint64_t upg = 1;        // units per group
  uint64_t total_units = 1;
  size_t smem_bytes = 0;   // dynamic shared memory of the enumeration kernels
  bool host_gbase = false; // group bases uploaded by the host (else one group, written on device)
  uint64_t gbase0 = 0;     // first unit prefix of the single group when !host_gbase
  bool prune = false;      // the biased minimum pass skips the per-step minima of blocks bounded above the threshold
  int prune_r = 0;         // its register rows: blocks of 2^prune_r steps
  int bound_margin = 0;    // extra margin of its bound test: unit minima up to E* + margin stay exact
  bool biased = false;     // biased-binade minimum pass (fast variant, int32, w >= kBiasedR + 1)
  bool packed = false;     // packed 16x2 minimum pass (fast variant, int32, C >= 10, w >= kPackedR + 1)
  bool packed_ok = false;  //   the packed pass fits this plan
  bool packed_pruned = false;  // the packed pass with block bounds runs (packed_ok and prune)
  int packed_pruned_blocks = 0;     // its persistent grid (2 blocks of 128 threads per SM)
  size_t packed_pruned_smem = 0;
  int packed_threads = 0;  // 2^C / 32
  int packed_blocks = 0;
  size_t packed_smem = 0;
};

// Device pointers into one workspace.
struct Work {
  DevHeader* hdr = nullptr;
  int32_t* U = nullptr;     // n x n int32 image of the folded triangle
  double* U64 = nullptr;    // n x n fp64 folded triangle (fp32 path)
  int32_t* M = nullptr;     // (n - C) x 2^C: interaction of each non-cached variable with each column
  int32_t* Ec = nullptr;    // 2^C: energy of the cached variables alone
  int32_t* T = nullptr;     // 2^w (padded): walked-variable energy, in Gray order
  uint32_t* T2 = nullptr;   // packed pass: T's low 16 bits in both halves
  BlockCtl* blk = nullptr;  // block-bounded minimum pass: one entry per block of 2^prune_r steps (+ 1)
  int32_t* gthr = nullptr;  // pruned minimum passes: best energy published so far, per group
  int32_t* unit_min = nullptr;
  uint32_t* tied = nullptr;
  uint64_t* gbase = nullptr;  // first unit prefix of each group
  int32_t* gmin = nullptr;
  uint64_t* grank = nullptr;
  uint64_t* gties = nullptr;
  uint64_t* gkey = nullptr;
  qubo_result* results = nullptr;  // one per group
  size_t bytes = 0;
};

// Byte layout of the workspace for a plan (offsets only; base may be null).
Work layout_workspace(const Plan& p, unsigned char* base);

// Kernel launch sequence for one plan on `stream`. d_Q is the device input, `res` receives
// one qubo_result per group. Returns cudaSuccess or the first launch error; `launches` counts.
// A set abort flag stops before the next min-pass launch and sets *aborted. When `timing` is
// non-null, its two events are recorded around the min-pass launches.
struct KernelTiming {
  cudaEvent_t start = nullptr, stop = nullptr;
};
cudaError_t run_search(const Plan& p, const void* d_Q, const Work& w, qubo_result* res, cudaStream_t stream,
                       int* launches, const volatile int* abort_flag, bool* aborted, const KernelTiming* timing);

// Batched mode (one block per instance).
struct BatchPlan {
  int batch = 0, n = 0, C = 0, w = 0, threads = 0;
  size_t smem_bytes = 0;
  // table-based pipeline (tabled = true): per-instance caches in the workspace, work units of
  // 2^(n - F) states shared by persistent minimum passes (packed / biased / int32), re-walk of
  // the units at each instance's minimum
  bool tabled = false;
  int F = 0;
  int blocks = 0;          // persistent grid of the 256-thread passes
  int packed_blocks = 0;   // persistent grid of the 128-thread packed pass
  size_t smem_int = 0, smem_biased = 0, smem_packed = 0;
  bool pruned = false;     // packed instances take the packed pass with block bounds
  int pruned_blocks = 0;   // its persistent grid
  size_t smem_pruned = 0;
};
bool plan_batched(int batch, int n, BatchPlan* bp);
size_t batched_workspace_bytes(const BatchPlan& bp);
cudaError_t run_batched(const BatchPlan& bp, const void* d_Q, void* d_ws, qubo_result* res, cudaStream_t stream,
                        int* launches);

// Whole-problem plan as qubo_solve_device makes it; launch-count bookkeeping of the C ABI.
bool valid_dtype(int dtype);
size_t dtype_bytes(int dtype);
int plan_whole_problem(int n, int dtype, int k_prefix, int cache_bits, Plan* p);
void plan_without_bounds(Plan* p);  // minimum passes that report every unit's exact minimum
bool block_bounds_enabled();        // qubo_enable_block_bounds (default on)
int record_launch_count(int launches);
int record_cuda_error(cudaError_t e, const char* where);  // returns QUBO_ERR_CUDA
std::mutex& api_mutex();      // serialises the host entry points
bool abort_requested();       // qubo_request_abort() was called and not cleared
int api_stream(cudaStream_t* s);  // the library's stream on the current device (QUBO_OK or an error)

// Measurement.
cudaError_t run_alu_probe(int kind, int iters, double* ops_per_s, double* sm_mhz);

// Device properties cached per device.
struct DevInfo {
  int device = -1;
  int sms = 0;
  size_t smem_optin = 0;
  int cc_major = 0, cc_minor = 0;
};
const DevInfo& device_info();

}  // namespace qgb
