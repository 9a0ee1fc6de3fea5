// C ABI of the solver: argument checks, the decomposition planner, workspace management and
// the host entry points. All arithmetic of the search runs in the kernels.
#include <algorithm>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <cmath>
#include <atomic>
#include <mutex>
#include <string>
#include <vector>

#include "qubo_search_kernel.cuh"

namespace qgb {

// ------------------------------------------------------------------------------------------------
// State
// ------------------------------------------------------------------------------------------------
namespace {
std::mutex g_mu;
std::string g_last_error;
int g_last_launches = 0;
volatile int g_abort = 0;
bool g_timing_enabled = false;
int g_timing_device = -1;
KernelTiming g_timing;
bool g_timing_recorded = false;
std::atomic<int> g_block_bounds{1};  // qubo_enable_block_bounds

// Events around the min-pass launches of the next calls, when kernel timing is enabled.
const KernelTiming* timing_for_call(int dev) {
  if (!g_timing_enabled) return nullptr;
  if (g_timing_device != dev) {
    if (g_timing.start) cudaEventDestroy(g_timing.start);
    if (g_timing.stop) cudaEventDestroy(g_timing.stop);
    g_timing = KernelTiming();
    if (cudaEventCreate(&g_timing.start) != cudaSuccess || cudaEventCreate(&g_timing.stop) != cudaSuccess)
      return nullptr;
    g_timing_device = dev;
  }
  g_timing_recorded = true;
  return &g_timing;
}

struct DeviceBuffers {
  int device = -1;
  cudaStream_t stream = nullptr;
  void* ws = nullptr;
  size_t ws_bytes = 0;
  void* dq = nullptr;
  size_t dq_bytes = 0;
  void* hres = nullptr;  // pinned
  size_t hres_bytes = 0;
  void* hgb = nullptr;  // pinned staging for group bases
  size_t hgb_bytes = 0;
};
DeviceBuffers g_buf;
DevInfo g_info[64];

int set_cuda_error(cudaError_t e, const char* where) {
  g_last_error = std::string(where) + ": " + cudaGetErrorString(e);
  return QUBO_ERR_CUDA;
}

int current_device(int* dev) {
  int count = 0;
  cudaError_t e = cudaGetDeviceCount(&count);
  if (e != cudaSuccess || count == 0) {
    g_last_error = "no CUDA device";
    return QUBO_ERR_NODEV;
  }
  if ((e = cudaGetDevice(dev)) != cudaSuccess) return set_cuda_error(e, "cudaGetDevice");
  return QUBO_OK;
}

int ceil_log2_u64(uint64_t x) {
  int b = 0;
  while (b < 63 && ((uint64_t)1 << b) < x) ++b;
  return b;
}

// Grow-only device buffer.
int ensure(void** ptr, size_t* have, size_t want, bool pinned, const char* what) {
  if (*have >= want && *ptr) return QUBO_OK;
  cudaError_t e;
  if (*ptr) {
    e = pinned ? cudaFreeHost(*ptr) : cudaFree(*ptr);
    *ptr = nullptr;
    *have = 0;
  }
  size_t sz = want < 256 ? 256 : want;
  e = pinned ? cudaMallocHost(ptr, sz) : cudaMalloc(ptr, sz);
  if (e != cudaSuccess) {
    *ptr = nullptr;
    return set_cuda_error(e, what);
  }
  *have = sz;
  return QUBO_OK;
}

int prepare_device_buffers() {
  int dev;
  int st = current_device(&dev);
  if (st) return st;
  if (g_buf.device != dev) {
    // a different device is current: start over (buffers of the old device are released)
    if (g_buf.device >= 0) {
      int old;
      cudaGetDevice(&old);
      cudaSetDevice(g_buf.device);
      if (g_buf.ws) cudaFree(g_buf.ws);
      if (g_buf.dq) cudaFree(g_buf.dq);
      if (g_buf.stream) cudaStreamDestroy(g_buf.stream);
      cudaSetDevice(old);
    }
    if (g_buf.hres) cudaFreeHost(g_buf.hres);
    if (g_buf.hgb) cudaFreeHost(g_buf.hgb);
    g_buf = DeviceBuffers();
    g_buf.device = dev;
    cudaError_t e = cudaStreamCreateWithFlags(&g_buf.stream, cudaStreamNonBlocking);
    if (e != cudaSuccess) return set_cuda_error(e, "cudaStreamCreate");
  }
  return QUBO_OK;
}
}  // namespace

const DevInfo& device_info() {
  int dev = 0;
  cudaGetDevice(&dev);
  DevInfo& d = g_info[dev & 63];
  if (d.device != dev) {
    cudaDeviceProp prop;
    if (cudaGetDeviceProperties(&prop, dev) == cudaSuccess) {
      d.sms = prop.multiProcessorCount;
      d.smem_optin = prop.sharedMemPerBlockOptin;
      d.cc_major = prop.major;
      d.cc_minor = prop.minor;
      d.device = dev;
    } else {
      d.sms = 1;
      d.smem_optin = 48 * 1024;
    }
  }
  return d;
}

// ------------------------------------------------------------------------------------------------
// The decomposition planner. n = F (fixed, per unit) + w (Gray-walked) + C (cached).
// ------------------------------------------------------------------------------------------------
namespace {

constexpr size_t kStaticSmemReserve = 2048;
// Work units of one call: unit indices are 32-bit (the tied-unit list), and every unit keeps an
// int32 minimum in the workspace.
constexpr double kMaxUnits = 2147483648.0;
// Problems with at least this many variables also launch the packed and biased minimum passes.
constexpr int kNarrowPassesMinN = 30;

bool fast_fits(int n, int C, int F, size_t smem_optin, size_t* smem) {
  const int w = n - F - C;
  if (C < 9 || C > 12 || F < 0 || w < kFastR + 1 || w > kMaxWalkedBits) return false;
  const size_t sm = (size_t)(w - kFastR) << (C + 2);
  if (sm + kStaticSmemReserve + kFastScanSlotBytes > smem_optin) return false;
  *smem = sm;
  return true;
}

bool generic_fits(int n, int C, int F, size_t smem_optin, size_t* smem) {
  const int w = n - F - C;
  if (C < 0 || C > kGenericMaxC || F < 0 || w < 0 || w > kMaxWalkedBits) return false;
  const size_t sm = (size_t)w << (C + 2);
  if (sm + kStaticSmemReserve > smem_optin) return false;
  *smem = sm < 16 ? 16 : sm;
  return true;
}

// The biased-binade minimum pass: fast variant, at least one iteration of 2^(kBiasedR+1) Gray
// steps; int32 input whose sum |U| turns out below 2^22 on the device, and every fp32/fp64 input
// (its fixed-point image is scaled to that range). Below 2^30 states a search takes tens of
// microseconds, mostly kernel launches: the alternative minimum passes (each launched, the ones
// that do not apply exiting at once) would cost more than they save, so small problems run the
// int32 pass alone.
bool biased_pass_applies(const Plan& p) {
  return p.n >= kNarrowPassesMinN && p.variant == kFast && p.w >= kBiasedR + 1;
}

// kind: 0 = whole problem (fixed_lo = 0), 1 = slices/range (fixed bits >= K).
// units_base: number of groups (slices) or range length; unit bits F = K + s.
int make_plan(int n, int dtype, int k_prefix, int cache_bits, int K, uint64_t units_base, bool explicit_F,
              Plan* out) {
  const DevInfo& di = device_info();
  const uint64_t target = (uint64_t)64 * (uint64_t)(di.sms > 0 ? di.sms : 1);
  Plan p;
  p.n = n;
  p.dtype = dtype;
  bool ok = false;
  size_t smem = 0;
  // candidate cache sizes
  std::vector<int> Cs;
  if (cache_bits > 0) Cs.push_back(cache_bits);
  else Cs = {12, 11, 10, 9};
  // choose F for a given C (fast variant)
  auto pick_F_fast = [&](int C, int* F) {
    if (explicit_F) {
      *F = k_prefix;
      if ((double)units_base * std::ldexp(1.0, k_prefix - K) > kMaxUnits) return false;
      return fast_fits(n, C, *F, di.smem_optin, &smem);
    }
    const int F_hi = n - C - (kFastR + 1);
    int F_lo = std::max(K, n - C - kMaxWalkedBits);
    if (F_hi < F_lo) return false;
    // Cost model of the persistent minimum pass: the units run in waves of one unit per block,
    // and every unit pays a fixed set-up (linear terms, register rows, block reduction) worth
    // about 2^18 states of walking on this part. Pick the F with the smallest
    // waves * (states per unit + set-up).
    const double sms = (double)(di.sms > 0 ? di.sms : 1);
    int best_F = -1;
    double best_cost = 0.0;
    size_t best_smem = 0;
    for (int Fv = F_lo; Fv <= F_hi; ++Fv) {
      size_t sm = 0;
      if (!fast_fits(n, C, Fv, di.smem_optin, &sm)) continue;
      const double units = (double)units_base * std::ldexp(1.0, Fv - K);
      if (units > kMaxUnits) continue;
      const double cost = std::ceil(units / sms) * (std::ldexp(1.0, n - Fv) + std::ldexp(1.0, 18));
      if (best_F < 0 || cost <= best_cost) {
        best_F = Fv;
        best_cost = cost;
        best_smem = sm;
      }
    }
    if (best_F < 0) return false;
    *F = best_F;
    smem = best_smem;
    return true;
  };
  for (int C : Cs) {
    int F;
    if (pick_F_fast(C, &F)) {
      p.variant = kFast;
      p.C = C;
      p.F = F;
      ok = true;
      break;
    }
  }
  if (!ok) {
    int C = cache_bits > 0 ? cache_bits : std::min(n - (explicit_F ? k_prefix : K), kGenericMaxC);
    int F = explicit_F ? k_prefix : std::max(K, n - C - kMaxWalkedBits);
    if (!explicit_F && cache_bits <= 0) {
      // spread small problems over a few blocks when possible
      while (F - K < 8 && n - C - F > 0 && ((units_base << (F - K)) < target)) ++F;
    }
    if ((double)units_base * std::ldexp(1.0, F - K) <= kMaxUnits && generic_fits(n, C, F, di.smem_optin, &smem)) {
      p.variant = kGeneric;
      p.C = C;
      p.F = F;
      ok = true;
    }
  }
  if (!ok) return QUBO_ERR_PLAN;
  p.w = n - p.F - p.C;
  p.R = (p.variant == kFast) ? kFastR : 0;
  p.cpt = (p.variant == kFast) ? kFastCPT : 1;
  p.threads = (p.variant == kFast) ? ((1 << p.C) / kFastCPT) : std::max(32, 1 << p.C);
  p.smem_bytes = smem;
  int occ = 1;
  cudaError_t e = (p.variant == kFast) ? occupancy_fast(p.threads, p.smem_bytes, &occ)
                                       : occupancy_generic(p.threads, p.smem_bytes, &occ);
  if (e != cudaSuccess || occ < 1) occ = 1;
  p.blocks = std::max(1, di.sms) * occ;
  const int64_t niter = (p.variant == kFast) ? walk_iterations<kFastR>(p.w) : walk_iterations<0>(p.w);
  int seg = 0;
  const int want_seg = ceil_log2_u64((uint64_t)p.blocks);
  while (seg < want_seg && (niter >> (seg + 1)) >= 1) ++seg;
  p.seg_bits = (niter > 0) ? seg : 0;
  // Small problems run the int32 pass alone (see biased_pass_applies).
  const bool narrow_passes = n >= kNarrowPassesMinN;
  p.biased = biased_pass_applies(p);
  // The biased pass with block bounds: 2^12 columns (256 threads of 16) and at least two blocks
  // of 2^prune_r steps per unit.
  p.prune_r = p.w >= kPruneLongW ? kPruneRLong : kPruneRShort;
  p.prune = g_block_bounds.load() && p.biased && p.C == 12 && p.threads == 256 && p.w >= p.prune_r + 1;
  // Packed 16x2 minimum pass: 32 columns per thread, so at least one warp needs C >= 10; its
  // shared rows are 2 bytes per column. It runs where the bounded biased pass does not: narrow
  // inputs (sum |U| < 2^14) fit the binade too, and there the bounded pass is the faster one
  // (n=40, entries in [-4, 4]: 29.0 ms against 30.3 ms).
  if (narrow_passes && p.variant == kFast && dtype == QUBO_INT32 && p.C >= 10 && p.w >= kPackedR + 1) {
    p.packed_threads = (1 << p.C) / 32;
    p.packed_smem = packed_smem_bytes(p.C, p.w);
    int pocc = 0;
    if (p.packed_smem + kStaticSmemReserve <= di.smem_optin &&
        occupancy_packed(p.packed_threads, p.packed_smem, &pocc) == cudaSuccess && pocc >= 1) {
      p.packed_ok = true;
      p.packed_blocks = std::max(1, di.sms) * pocc;
    }
  }
  p.packed = p.packed_ok && !p.prune;
  p.packed_pruned = p.packed_ok && p.prune;
  if (p.packed_pruned) {
    p.packed_pruned_smem = packed_pruned_smem_bytes(p.C, p.w, p.prune_r);
    int pocc = 0;
    if (occupancy_packed_pruned(p.prune_r, p.packed_pruned_smem, &pocc) != cudaSuccess || pocc < 1) pocc = 1;
    p.packed_pruned_blocks = std::max(1, di.sms) * pocc;
  }
  *out = p;
  return QUBO_OK;
}

int check_common(int n, const void* Q, int dtype) {
  if (n < 1 || n > 62 || Q == nullptr || !valid_dtype(dtype)) return QUBO_ERR_ARG;
  return QUBO_OK;
}

void rank_to_bits(int n, uint64_t rank, uint8_t* x) {
  for (int i = 0; i < n; ++i) x[i] = (uint8_t)((rank >> (n - 1 - i)) & 1u);
}

// Run a planned search on host input; copies results of all groups into hres.
int host_search(const Plan& p, const void* Q, const uint64_t* gbase_host, std::vector<qubo_result>* out) {
  int st = prepare_device_buffers();
  if (st) return st;
  Work lay = layout_workspace(p, nullptr);
  if ((st = ensure(&g_buf.ws, &g_buf.ws_bytes, lay.bytes, false, "cudaMalloc(workspace)"))) return st;
  const size_t qbytes = (size_t)p.n * p.n * dtype_bytes(p.dtype);
  if ((st = ensure(&g_buf.dq, &g_buf.dq_bytes, qbytes, false, "cudaMalloc(Q)"))) return st;
  const size_t rbytes = (size_t)p.ngroups * sizeof(qubo_result);
  if ((st = ensure(&g_buf.hres, &g_buf.hres_bytes, rbytes, true, "cudaMallocHost(results)"))) return st;
  Work w = layout_workspace(p, static_cast<unsigned char*>(g_buf.ws));
  cudaStream_t s = g_buf.stream;
  cudaError_t e = cudaMemcpyAsync(g_buf.dq, Q, qbytes, cudaMemcpyHostToDevice, s);
  if (e != cudaSuccess) return set_cuda_error(e, "cudaMemcpyAsync(Q)");
  if (gbase_host) {
    if (!p.host_gbase) return QUBO_ERR_ARG;
    const size_t gb = (size_t)p.ngroups * 8;
    if ((st = ensure(&g_buf.hgb, &g_buf.hgb_bytes, gb, true, "cudaMallocHost(groups)"))) return st;
    memcpy(g_buf.hgb, gbase_host, gb);
    e = cudaMemcpyAsync(w.gbase, g_buf.hgb, gb, cudaMemcpyHostToDevice, s);
    if (e != cudaSuccess) return set_cuda_error(e, "cudaMemcpyAsync(groups)");
  }
  int nl = 0;
  bool aborted = false;
  e = run_search(p, g_buf.dq, w, w.results, s, &nl, &g_abort, &aborted, timing_for_call(g_buf.device));
  g_last_launches = nl;
  if (aborted) {
    cudaStreamSynchronize(s);
    return QUBO_ERR_ABORTED;
  }
  if (e != cudaSuccess) return set_cuda_error(e, "kernel launch");
  e = cudaMemcpyAsync(g_buf.hres, w.results, rbytes, cudaMemcpyDeviceToHost, s);
  if (e != cudaSuccess) return set_cuda_error(e, "cudaMemcpyAsync(results)");
  e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return set_cuda_error(e, "cudaStreamSynchronize");
  if (g_abort) return QUBO_ERR_ABORTED;
  const qubo_result* r = static_cast<const qubo_result*>(g_buf.hres);
  out->assign(r, r + p.ngroups);
  for (const auto& x : *out)
    if (x.status != QUBO_OK) return x.status;
  return QUBO_OK;
}

}  // namespace

// Plan of a whole-problem search, exactly as qubo_solve_device makes it.
int plan_whole_problem(int n, int dtype, int k_prefix, int cache_bits, Plan* p) {
  int st = make_plan(n, dtype, k_prefix, cache_bits, 0, 1, k_prefix > 0, p);
  if (st) return st;
  p->ngroups = 1;
  p->upg = (uint64_t)1 << p->F;
  p->total_units = p->upg;
  return QUBO_OK;
}

bool block_bounds_enabled() { return g_block_bounds.load() != 0; }

void plan_without_bounds(Plan* p) {
  p->prune = false;
  p->packed = p->packed_ok;
  p->packed_pruned = false;
}

int record_launch_count(int launches) {
  g_last_launches = launches;
  return launches;
}

int record_cuda_error(cudaError_t e, const char* where) { return set_cuda_error(e, where); }

std::mutex& api_mutex() { return g_mu; }

bool abort_requested() { return g_abort != 0; }

int api_stream(cudaStream_t* s) {
  const int st = prepare_device_buffers();
  if (st) return st;
  *s = g_buf.stream;
  return QUBO_OK;
}
bool valid_dtype(int dtype) { return dtype == QUBO_INT32 || dtype == QUBO_FP32 || dtype == QUBO_FP64; }

size_t dtype_bytes(int dtype) { return dtype == QUBO_FP64 ? 8 : 4; }

}  // namespace qgb

using namespace qgb;

extern "C" {

int qubo_solve(int n, const void* Q, int dtype, int k_prefix, int cache_bits, double* out_min_energy,
               uint8_t* out_argmin_x, uint64_t* out_tie_count) {
  int st = check_common(n, Q, dtype);
  if (st) return st;
  if (!out_min_energy || !out_argmin_x || !out_tie_count) return QUBO_ERR_ARG;
  if (k_prefix > n || cache_bits > n) return QUBO_ERR_PLAN;
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_abort) return QUBO_ERR_ABORTED;
  int dev;
  if ((st = current_device(&dev))) return st;
  Plan p;
  if ((st = make_plan(n, dtype, k_prefix, cache_bits, 0, 1, k_prefix > 0, &p))) return st;
  p.ngroups = 1;
  p.upg = (uint64_t)1 << p.F;
  p.total_units = p.upg;
  std::vector<qubo_result> res;
  if ((st = host_search(p, Q, nullptr, &res))) return st;
  *out_min_energy = res[0].min_energy;
  rank_to_bits(n, res[0].argmin_rank, out_argmin_x);
  *out_tie_count = res[0].tie_count;
  return QUBO_OK;
}

int qubo_solve_slices(int n, const void* Q, int dtype, int k_prefix, int cache_bits, const uint64_t* slice_ids,
                      int num_slices, double* out_min_energy, uint8_t* out_argmin_x, uint64_t* out_tie_count) {
  int st = check_common(n, Q, dtype);
  if (st) return st;
  if (k_prefix < 1 || k_prefix >= n || num_slices < 1 || !slice_ids || !out_min_energy || !out_argmin_x ||
      !out_tie_count)
    return QUBO_ERR_ARG;
  for (int s = 0; s < num_slices; ++s)
    if (k_prefix < 64 && (slice_ids[s] >> k_prefix) != 0) return QUBO_ERR_ARG;
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_abort) return QUBO_ERR_ABORTED;
  int dev;
  if ((st = current_device(&dev))) return st;
  Plan p;
  if ((st = make_plan(n, dtype, k_prefix, cache_bits, k_prefix, (uint64_t)num_slices, false, &p))) return st;
  const int s_bits = p.F - k_prefix;
  p.ngroups = num_slices;
  p.upg = (uint64_t)1 << s_bits;
  p.total_units = p.upg * (uint64_t)num_slices;
  if (p.total_units >= ((uint64_t)1 << 32)) return QUBO_ERR_PLAN;
  std::vector<uint64_t> gb(num_slices);
  for (int s = 0; s < num_slices; ++s) gb[s] = slice_ids[s] << s_bits;
  p.host_gbase = true;
  std::vector<qubo_result> res;
  if ((st = host_search(p, Q, gb.data(), &res))) return st;
  for (int s = 0; s < num_slices; ++s) {
    out_min_energy[s] = res[s].min_energy;
    rank_to_bits(n, res[s].argmin_rank, out_argmin_x + (size_t)s * n);
    out_tie_count[s] = res[s].tie_count;
  }
  return QUBO_OK;
}

int qubo_solve_slice_range(int n, const void* Q, int dtype, int k_prefix, int cache_bits, uint64_t first_slice,
                           uint64_t num_slices, double* out_min_energy, uint8_t* out_argmin_x,
                           uint64_t* out_tie_count) {
  int st = check_common(n, Q, dtype);
  if (st) return st;
  if (k_prefix < 1 || k_prefix >= n || num_slices < 1 || !out_min_energy || !out_argmin_x || !out_tie_count)
    return QUBO_ERR_ARG;
  if (first_slice + num_slices > ((uint64_t)1 << k_prefix) || first_slice + num_slices < first_slice)
    return QUBO_ERR_ARG;
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_abort) return QUBO_ERR_ABORTED;
  int dev;
  if ((st = current_device(&dev))) return st;
  Plan p;
  if ((st = make_plan(n, dtype, k_prefix, cache_bits, k_prefix, num_slices, false, &p))) return st;
  const int s_bits = p.F - k_prefix;
  p.ngroups = 1;
  p.upg = num_slices << s_bits;
  p.total_units = p.upg;
  if (p.total_units >= ((uint64_t)1 << 32)) return QUBO_ERR_PLAN;
  uint64_t gb = first_slice << s_bits;
  p.host_gbase = true;
  std::vector<qubo_result> res;
  if ((st = host_search(p, Q, &gb, &res))) return st;
  *out_min_energy = res[0].min_energy;
  rank_to_bits(n, res[0].argmin_rank, out_argmin_x);
  *out_tie_count = res[0].tie_count;
  return QUBO_OK;
}

size_t qubo_workspace_bytes(int n, int dtype, int k_prefix, int cache_bits) {
  if (n < 1 || n > 62 || !valid_dtype(dtype)) return 0;
  int dev;
  if (current_device(&dev)) return 0;
  Plan p;
  if (make_plan(n, dtype, k_prefix, cache_bits, 0, 1, k_prefix > 0, &p)) return 0;
  p.ngroups = 1;
  p.upg = (uint64_t)1 << p.F;
  p.total_units = p.upg;
  return layout_workspace(p, nullptr).bytes;
}

int qubo_solve_device(int n, const void* d_Q, int dtype, int k_prefix, int cache_bits, void* d_workspace,
                      size_t workspace_bytes, void* cuda_stream, qubo_result* d_result) {
  int st = check_common(n, d_Q, dtype);
  if (st) return st;
  if (!d_workspace || !d_result || (reinterpret_cast<uintptr_t>(d_workspace) & 255)) return QUBO_ERR_ARG;
  if (k_prefix > n || cache_bits > n) return QUBO_ERR_PLAN;
  if (g_abort) return QUBO_ERR_ABORTED;
  int dev;
  if ((st = current_device(&dev))) return st;
  Plan p;
  if ((st = make_plan(n, dtype, k_prefix, cache_bits, 0, 1, k_prefix > 0, &p))) return st;
  p.ngroups = 1;
  p.upg = (uint64_t)1 << p.F;
  p.total_units = p.upg;
  Work w = layout_workspace(p, static_cast<unsigned char*>(d_workspace));
  if (w.bytes > workspace_bytes) return QUBO_ERR_ARG;
  int nl = 0;
  cudaError_t e = run_search(p, d_Q, w, d_result, static_cast<cudaStream_t>(cuda_stream), &nl, nullptr, nullptr,
                             timing_for_call(dev));
  g_last_launches = nl;
  if (e != cudaSuccess) return set_cuda_error(e, "kernel launch");
  return QUBO_OK;
}

int qubo_solve_batched(int batch, int n, const void* Q, int dtype, double* out_min_energy, uint8_t* out_argmin_x,
                       uint64_t* out_tie_count) {
  if (batch < 1 || n < 1 || n > 62 || !Q || dtype != QUBO_INT32 || !out_min_energy || !out_argmin_x ||
      !out_tie_count)
    return QUBO_ERR_ARG;
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_abort) return QUBO_ERR_ABORTED;
  int st = prepare_device_buffers();
  if (st) return st;
  const size_t per = (size_t)n * n;
  BatchPlan bp;
  if (plan_batched(batch, n, &bp)) {
    const size_t qbytes = per * 4 * (size_t)batch;
    if ((st = ensure(&g_buf.dq, &g_buf.dq_bytes, qbytes, false, "cudaMalloc(Q)"))) return st;
    const size_t rbytes = (size_t)batch * sizeof(qubo_result);
    const size_t wsb = (batched_workspace_bytes(bp) + 255) & ~(size_t)255;  // then the results
    if ((st = ensure(&g_buf.ws, &g_buf.ws_bytes, wsb + rbytes, false, "cudaMalloc(workspace)"))) return st;
    if ((st = ensure(&g_buf.hres, &g_buf.hres_bytes, rbytes, true, "cudaMallocHost(results)"))) return st;
    cudaStream_t s = g_buf.stream;
    cudaError_t e = cudaMemcpyAsync(g_buf.dq, Q, qbytes, cudaMemcpyHostToDevice, s);
    if (e != cudaSuccess) return set_cuda_error(e, "cudaMemcpyAsync(Q)");
    int nl = 0;
    qubo_result* d_res = reinterpret_cast<qubo_result*>(static_cast<unsigned char*>(g_buf.ws) + wsb);
    e = run_batched(bp, g_buf.dq, g_buf.ws, d_res, s, &nl);
    g_last_launches = nl;
    if (e != cudaSuccess) return set_cuda_error(e, "batched launch");
    e = cudaMemcpyAsync(g_buf.hres, d_res, rbytes, cudaMemcpyDeviceToHost, s);
    if (e != cudaSuccess) return set_cuda_error(e, "cudaMemcpyAsync(results)");
    if ((e = cudaStreamSynchronize(s)) != cudaSuccess) return set_cuda_error(e, "cudaStreamSynchronize");
    const qubo_result* r = static_cast<const qubo_result*>(g_buf.hres);
    for (int b = 0; b < batch; ++b)
      if (r[b].status != QUBO_OK) return r[b].status;
    for (int b = 0; b < batch; ++b) {
      out_min_energy[b] = r[b].min_energy;
      rank_to_bits(n, r[b].argmin_rank, out_argmin_x + (size_t)b * n);
      out_tie_count[b] = r[b].tie_count;
    }
    return QUBO_OK;
  }
  // Sizes the block-per-instance kernel does not take: one full search per instance.
  std::vector<qubo_result> all((size_t)batch);
  int launches = 0;
  for (int b = 0; b < batch; ++b) {
    Plan p;
    if ((st = make_plan(n, dtype, 0, 0, 0, 1, false, &p))) return st;
    p.ngroups = 1;
    p.upg = (uint64_t)1 << p.F;
    p.total_units = p.upg;
    std::vector<qubo_result> res;
    if ((st = host_search(p, static_cast<const int32_t*>(Q) + (size_t)b * per, nullptr, &res))) return st;
    all[b] = res[0];
    launches += g_last_launches;
  }
  g_last_launches = launches;
  for (int b = 0; b < batch; ++b) {
    out_min_energy[b] = all[b].min_energy;
    rank_to_bits(n, all[b].argmin_rank, out_argmin_x + (size_t)b * n);
    out_tie_count[b] = all[b].tie_count;
  }
  return QUBO_OK;
}

size_t qubo_batched_workspace_bytes(int batch, int n, int dtype) {
  BatchPlan bp;
  if (dtype != QUBO_INT32) return 0;
  int dev;
  if (current_device(&dev)) return 0;
  if (!plan_batched(batch, n, &bp)) return 0;
  return batched_workspace_bytes(bp);
}

int qubo_solve_batched_device(int batch, int n, const void* d_Q, int dtype, void* d_workspace,
                              size_t workspace_bytes, void* cuda_stream, qubo_result* d_results) {
  if (batch < 1 || n < 1 || n > 62 || !d_Q || dtype != QUBO_INT32 || !d_results) return QUBO_ERR_ARG;
  int dev, st;
  if ((st = current_device(&dev))) return st;
  BatchPlan bp;
  if (!plan_batched(batch, n, &bp)) return QUBO_ERR_PLAN;
  if (workspace_bytes < batched_workspace_bytes(bp) || !d_workspace) return QUBO_ERR_ARG;
  int nl = 0;
  cudaError_t e = run_batched(bp, d_Q, d_workspace, d_results, static_cast<cudaStream_t>(cuda_stream), &nl);
  g_last_launches = nl;
  if (e != cudaSuccess) return set_cuda_error(e, "batched launch");
  return QUBO_OK;
}

size_t qubo_slice_range_workspace_bytes(int n, int dtype, int k_prefix, int cache_bits, uint64_t num_slices) {
  if (n < 1 || n > 62 || !valid_dtype(dtype) || k_prefix < 1 || k_prefix >= n ||
      num_slices < 1)
    return 0;
  int dev;
  if (current_device(&dev)) return 0;
  Plan p;
  if (make_plan(n, dtype, k_prefix, cache_bits, k_prefix, num_slices, false, &p)) return 0;
  p.ngroups = 1;
  p.upg = num_slices << (p.F - k_prefix);
  p.total_units = p.upg;
  return layout_workspace(p, nullptr).bytes;
}

int qubo_solve_slice_range_device(int n, const void* d_Q, int dtype, int k_prefix, int cache_bits,
                                  uint64_t first_slice, uint64_t num_slices, void* d_workspace,
                                  size_t workspace_bytes, void* cuda_stream, qubo_result* d_result) {
  int st = check_common(n, d_Q, dtype);
  if (st) return st;
  if (k_prefix < 1 || k_prefix >= n || num_slices < 1 || !d_workspace || !d_result ||
      (reinterpret_cast<uintptr_t>(d_workspace) & 255))
    return QUBO_ERR_ARG;
  if (first_slice + num_slices > ((uint64_t)1 << k_prefix) || first_slice + num_slices < first_slice)
    return QUBO_ERR_ARG;
  if (g_abort) return QUBO_ERR_ABORTED;
  int dev;
  if ((st = current_device(&dev))) return st;
  Plan p;
  if ((st = make_plan(n, dtype, k_prefix, cache_bits, k_prefix, num_slices, false, &p))) return st;
  const int s_bits = p.F - k_prefix;
  p.ngroups = 1;
  p.upg = num_slices << s_bits;
  p.total_units = p.upg;
  if (p.total_units >= ((uint64_t)1 << 32)) return QUBO_ERR_PLAN;
  p.gbase0 = first_slice << s_bits;
  Work w = layout_workspace(p, static_cast<unsigned char*>(d_workspace));
  if (w.bytes > workspace_bytes) return QUBO_ERR_ARG;
  int nl = 0;
  cudaError_t e = run_search(p, d_Q, w, d_result, static_cast<cudaStream_t>(cuda_stream), &nl, nullptr, nullptr,
                             timing_for_call(dev));
  g_last_launches = nl;
  if (e != cudaSuccess) return set_cuda_error(e, "kernel launch");
  return QUBO_OK;
}

void qubo_enable_kernel_timing(int enable) {
  std::lock_guard<std::mutex> lk(g_mu);
  g_timing_enabled = enable != 0;
  g_timing_recorded = false;
}

void qubo_enable_block_bounds(int enable) { g_block_bounds.store(enable != 0 ? 1 : 0); }

double qubo_kernel_time_ms(void) {
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_timing_enabled || !g_timing_recorded || !g_timing.stop) return -1.0;
  if (cudaEventSynchronize(g_timing.stop) != cudaSuccess) return -1.0;
  float ms = 0.f;
  if (cudaEventElapsedTime(&ms, g_timing.start, g_timing.stop) != cudaSuccess) return -1.0;
  return (double)ms;
}

int qubo_plan(int n, int dtype, int k_prefix, int cache_bits, qubo_plan_desc* out) {
  if (n < 1 || n > 62 || !valid_dtype(dtype) || !out) return QUBO_ERR_ARG;
  if (k_prefix > n || cache_bits > n) return QUBO_ERR_PLAN;
  int dev, st;
  if ((st = current_device(&dev))) return st;
  Plan p;
  if ((st = make_plan(n, dtype, k_prefix, cache_bits, 0, 1, k_prefix > 0, &p))) return st;
  p.ngroups = 1;
  p.upg = (uint64_t)1 << p.F;
  p.total_units = p.upg;
  out->n = n;
  out->dtype = dtype;
  out->k_prefix = p.F;
  out->cache_bits = p.C;
  out->walked_bits = p.w;
  out->register_bits = p.R;
  out->columns_per_thread = p.cpt;
  out->threads_per_block = p.threads;
  out->blocks = p.blocks;
  out->variant = p.variant;
  out->units = p.total_units;
  out->workspace_bytes = layout_workspace(p, nullptr).bytes;
  out->smem_bytes = p.smem_bytes;
  out->packed = (p.packed || p.packed_pruned) ? 1 : 0;
  out->biased = p.biased ? 1 : 0;
  out->pruned = p.prune ? 1 : 0;
  return QUBO_OK;
}

int qubo_last_launch_count(void) { return g_last_launches; }

const char* qubo_status_string(int status) {
  switch (status) {
    case QUBO_OK: return "ok";
    case QUBO_ERR_ARG: return "invalid argument";
    case QUBO_ERR_RANGE: return "int32 range: sum of |U_ij| exceeds 2^30 - 1";
    case QUBO_ERR_NONFINITE: return "non-finite entry in floating-point input";
    case QUBO_ERR_PLAN: return "no kernel plan for the requested k_prefix / cache_bits";
    case QUBO_ERR_CUDA: return "CUDA error";
    case QUBO_ERR_NODEV: return "no CUDA device";
    case QUBO_ERR_ABORTED: return "aborted";
    case QUBO_ERR_CHECKPOINT: return "checkpoint file unreadable, corrupt, or of another problem";
    case QUBO_INCOMPLETE: return "incomplete: time budget reached, progress saved";
  }
  return "unknown status";
}

const char* qubo_last_error(void) { return g_last_error.c_str(); }

void qubo_request_abort(void) { g_abort = 1; }
void qubo_clear_abort(void) { g_abort = 0; }

int qubo_probe_alu(int kind, int iters, double* out_ops_per_s, double* out_sm_mhz) {
  if (!out_ops_per_s || !out_sm_mhz || iters < 1 || kind < 0 || kind > 18) return QUBO_ERR_ARG;
  std::lock_guard<std::mutex> lk(g_mu);
  int dev, st;
  if ((st = current_device(&dev))) return st;
  cudaError_t e = run_alu_probe(kind, iters, out_ops_per_s, out_sm_mhz);
  if (e != cudaSuccess) return set_cuda_error(e, "alu probe");
  return QUBO_OK;
}

}  // extern "C"
