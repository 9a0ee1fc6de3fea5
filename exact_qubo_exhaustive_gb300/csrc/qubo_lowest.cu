// The k lowest energies (low-energy spectrum) of a QUBO, exactly.
//
// Terastate-per-second QUBO Brute-Force on a Single GPU, §I and §VI-B: the exhaustive search
// sees every state, so besides the minimum it can return the lowest part of the spectrum. The
// result is the k states with the smallest keys (E(x), rank(x)) in ascending order: energies
// ascending, equal energies by rank, so the answer is unique whatever the decomposition.
//
// Driver (host), over the enumeration kernel's passes:
//  1. the usual fold, tables and minimum pass give every work unit's minimum (with block bounds
//     whose test keeps a margin: every unit whose minimum lies within E* + margin reports it
//     exactly, every other unit a value above E* + margin);
//  2. theta = the k-th smallest unit minimum (each of those units holds a state <= theta, so at
//     least k states have E <= theta) when it lies within the margin; otherwise theta =
//     E* + margin, whose collect pass counts the states at or below it exactly, and the margin
//     is widened fourfold (and the minimum pass rerun) while fewer than k states lie within it;
//     with fewer than k units (no bounds then), theta grows from the largest unit minimum until
//     the count reaches k;
//  3. one collect pass re-walks only the units whose minimum is <= theta and appends every state
//     with E <= theta; if they fit the candidate buffer, selecting the k smallest keys on the
//     host finishes;
//  4. otherwise (a very degenerate spectrum) count passes bisect theta down to the smallest value
//     with at least k states, then bisect the rank bound rho inside that energy level, and the
//     final collect pass returns exactly the k smallest keys.
#include <algorithm>
#include <cmath>
#include <cstring>
#include <vector>

#include "qubo_search_kernel.cuh"

using namespace qgb;

namespace {

struct Buffers {
  void* base = nullptr;
  ~Buffers() {
    if (base) cudaFree(base);
  }
};

}  // namespace

extern "C" int qubo_solve_lowest(int n, const void* Q, int dtype, int k_prefix, int cache_bits, int k,
                                 double* out_energies, uint8_t* out_x, int* out_count) {
  if (n < 1 || n > 62 || !Q || dtype != QUBO_INT32 || k < 1 || k > QUBO_LOWEST_MAX_K || !out_energies || !out_x ||
      !out_count)
    return QUBO_ERR_ARG;
  std::lock_guard<std::mutex> lk(api_mutex());
  if (abort_requested()) return QUBO_ERR_ABORTED;
  cudaStream_t s;
  int st = api_stream(&s);
  if (st) return st;
  Plan p;
  if ((st = plan_whole_problem(n, dtype, k_prefix, cache_bits, &p))) return st;

  const uint64_t total_states = (uint64_t)1 << n;
  const uint64_t want = (uint64_t)k < total_states ? (uint64_t)k : total_states;
  // The collect pass re-walks at least `want` whole units, so with the planner's default split
  // it could re-walk a large share of the states. Smaller units cost the minimum pass more unit
  // set-ups. Pick the split that minimises
  //   ceil(units / blocks) * (S_u + kSetup)  +  kCollectCost * want / blocks * (S_u + kSetup),
  // with S_u the states per unit. Measured at n=40: a unit set-up costs about 2^20 states of
  // walking when blocks run hundreds of units, and the collect pass costs about 1.5x the
  // minimum pass per state (its units hold the candidates, whose half-iterations are walked
  // twice).
  if (k_prefix <= 0) {
    constexpr double kSetup = 1048576.0, kCollectCost = 1.5;
    auto cost = [&](const Plan& q) {
      const double spu = std::ldexp(1.0, n - q.F), blocks = (double)std::max(1, q.blocks);
      return std::ceil((double)q.total_units / blocks) * (spu + kSetup) + kCollectCost * (double)want / blocks * (spu + kSetup);
    };
    double best = cost(p);
    for (int F = p.F + 1; F <= std::min(31, n); ++F) {
      Plan q;
      if (plan_whole_problem(n, dtype, F, cache_bits, &q) != QUBO_OK) continue;
      const double c = cost(q);
      if (c < best) {
        best = c;
        p = q;
      }
    }
  }
  // theta and the collect pass need the exact minimum of every unit at or below theta: the block
  // bounds keep a margin (below); without enough units for theta to be one of them, no bounds
  const bool bounded = p.prune && p.total_units >= want;
  if (!bounded) plan_without_bounds(&p);
  int64_t abs_sum = 0;  // sum |U_ij| of the folded triangle: every energy lies in [-S, S]
  {
    const int32_t* Qi = static_cast<const int32_t*>(Q);
    for (int i = 0; i < n; ++i)
      for (int j = i; j < n; ++j) {
        const int64_t u = (j == i) ? (int64_t)Qi[i * n + i] : (int64_t)Qi[i * n + j] + Qi[j * n + i];
        abs_sum += u < 0 ? -u : u;
      }
  }
  const uint64_t cap = std::max<uint64_t>(2 * want, (uint64_t)1 << 18);

  // one allocation: workspace | Q | candidates | counter
  const Work lay = layout_workspace(p, nullptr);
  const size_t qbytes = ((size_t)n * n * 4 + 255) & ~(size_t)255;
  const size_t cbytes = (size_t)cap * sizeof(KeyCand);
  Buffers buf;
  cudaError_t e = cudaMalloc(&buf.base, lay.bytes + qbytes + cbytes + 256);
  if (e != cudaSuccess) return record_cuda_error(e, "cudaMalloc(k lowest)");
  unsigned char* base = static_cast<unsigned char*>(buf.base);
  const Work w = layout_workspace(p, base);
  void* dQ = base + lay.bytes;
  KeyCand* cand = reinterpret_cast<KeyCand*>(base + lay.bytes + qbytes);
  unsigned long long* counter = reinterpret_cast<unsigned long long*>(base + lay.bytes + qbytes + cbytes);

  int launches = 0;
  if ((e = cudaMemcpyAsync(dQ, Q, (size_t)n * n * 4, cudaMemcpyHostToDevice, s)) != cudaSuccess)
    return record_cuda_error(e, "cudaMemcpyAsync(Q)");
  KParams kp;
  DevHeader hdr;
  std::vector<int32_t> um(p.total_units);
  // The margin starts at S / 64; from 2S on no block is skipped at all.
  int64_t margin = bounded ? std::max<int64_t>(64, abs_sum / 64) : 0;
  auto min_stage = [&]() -> int {
    if (abort_requested()) return QUBO_ERR_ABORTED;
    p.bound_margin = (int)std::min<int64_t>(margin, 2 * abs_sum);  // 2S < 2^31: S < 2^30 for int32
    int nl = 0;
    cudaError_t ee;
    if ((ee = run_min_stage(p, dQ, w, s, &nl, &kp)) != cudaSuccess) return record_cuda_error(ee, "kernel launch");
    launches += nl;
    if ((ee = cudaMemcpyAsync(&hdr, w.hdr, sizeof(hdr), cudaMemcpyDeviceToHost, s)) != cudaSuccess ||
        (ee = cudaMemcpyAsync(um.data(), w.unit_min, um.size() * 4, cudaMemcpyDeviceToHost, s)) != cudaSuccess ||
        (ee = cudaStreamSynchronize(s)) != cudaSuccess)
      return record_cuda_error(ee, "unit minima");
    return hdr.status;
  };
  if ((st = min_stage())) return st;

  int64_t E0 = *std::min_element(um.begin(), um.end());
  const int64_t Smax = hdr.abs_sum;  // every energy lies in [-S, S]

  // One pass: count (or collect) the states with key (E, rank) < (theta, rho) over the units
  // whose minimum is <= theta.
  std::vector<uint32_t> list;
  auto pass = [&](int mode, int64_t theta, uint64_t rho, uint64_t* count) -> int {
    if (abort_requested()) return QUBO_ERR_ABORTED;
    list.clear();
    for (uint64_t u = 0; u < p.total_units; ++u)
      if (um[u] <= theta) list.push_back((uint32_t)u);
    const uint32_t nt = (uint32_t)list.size();
    cudaError_t ee;
    if (nt && (ee = cudaMemcpyAsync(w.tied, list.data(), (size_t)nt * 4, cudaMemcpyHostToDevice, s)) != cudaSuccess)
      return record_cuda_error(ee, "cudaMemcpyAsync(units)");
    if ((ee = cudaMemcpyAsync(&w.hdr->tied_count, &nt, 4, cudaMemcpyHostToDevice, s)) != cudaSuccess ||
        (ee = cudaMemsetAsync(counter, 0, 8, s)) != cudaSuccess)
      return record_cuda_error(ee, "pass set-up");
    // split each listed unit into just enough segments to give every block a few items (the
    // plan's split is for a single tied unit; every segment pays a unit set-up)
    KParams kps = kp;
    int seg = 0;
    while (seg < p.seg_bits && ((uint64_t)nt << seg) < 4 * (uint64_t)p.blocks) ++seg;
    kps.seg_bits = seg;
    if ((ee = run_key_pass(p, kps, mode, (int)theta, rho, cand, (uint32_t)cap, counter, s)) != cudaSuccess)
      return record_cuda_error(ee, "kernel launch");
    ++launches;
    unsigned long long c = 0;
    if ((ee = cudaMemcpyAsync(&c, counter, 8, cudaMemcpyDeviceToHost, s)) != cudaSuccess ||
        (ee = cudaStreamSynchronize(s)) != cudaSuccess)
      return record_cuda_error(ee, "pass count");
    *count = c;
    return QUBO_OK;
  };
  const uint64_t kAllRanks = ~0ull;

  // 2. an upper threshold with at least `want` states at or below it
  int64_t theta;
  uint64_t c = 0;
  if (p.total_units >= want) {  // the want-th smallest unit minimum (linear-time selection)
    for (;;) {
      std::vector<int32_t> sel(um);
      std::nth_element(sel.begin(), sel.begin() + (want - 1), sel.end());
      theta = sel[want - 1];
      if (!bounded || margin >= 2 * abs_sum || theta <= E0 + margin) break;
      // beyond the margin: count the states within it exactly; enough of them make E0 + margin
      // the threshold, otherwise widen the margin and walk again
      theta = E0 + margin;
      if ((st = pass(kModeCollectKey, theta, kAllRanks, &c))) return st;
      if (c >= want) break;
      margin *= 4;
      if ((st = min_stage())) return st;
      E0 = *std::min_element(um.begin(), um.end());
    }
  } else {
    theta = *std::max_element(um.begin(), um.end());
  }
  if (c < want && (st = pass(kModeCollectKey, theta, kAllRanks, &c))) return st;
  int64_t lo = E0 - 1;  // count(E <= lo) = 0 < want
  while (c < want) {
    lo = theta;
    theta = std::min<int64_t>(Smax, E0 + 2 * (theta - E0) + 1);
    if ((st = pass(kModeCollectKey, theta, kAllRanks, &c))) return st;
  }
  uint64_t rho = kAllRanks;
  if (c > cap) {
    // 4. smallest theta with count >= want (collect as soon as a probe fits the buffer)
    int64_t hi = theta;
    bool done = false;
    while (hi - lo > 1) {
      const int64_t mid = lo + (hi - lo) / 2;
      uint64_t cm = 0;
      if ((st = pass(kModeCountKey, mid, kAllRanks, &cm))) return st;
      if (cm >= want) {
        hi = mid;
        if (cm <= cap) {
          if ((st = pass(kModeCollectKey, mid, kAllRanks, &c))) return st;
          theta = mid;
          done = true;
          break;
        }
      } else {
        lo = mid;
      }
    }
    if (!done) {
      theta = hi;
      // fewer than `want` states lie below theta: bisect the rank bound within the level
      uint64_t rlo = 0, rhi = total_states;  // count(key < (theta, rlo)) < want <= count(.., rhi)
      while (rhi - rlo > 1) {
        const uint64_t mid = rlo + (rhi - rlo) / 2;
        uint64_t cm = 0;
        if ((st = pass(kModeCountKey, theta, mid, &cm))) return st;
        if (cm >= want) rhi = mid;
        else rlo = mid;
      }
      rho = rhi;
      if ((st = pass(kModeCollectKey, theta, rho, &c))) return st;
    }
  }
  if (c > cap || c < want) {
    record_cuda_error(cudaErrorUnknown, "k lowest: inconsistent pass counts");
    return QUBO_ERR_CUDA;
  }
  std::vector<KeyCand> h(c);
  if ((e = cudaMemcpyAsync(h.data(), cand, (size_t)c * sizeof(KeyCand), cudaMemcpyDeviceToHost, s)) != cudaSuccess ||
      (e = cudaStreamSynchronize(s)) != cudaSuccess)
    return record_cuda_error(e, "candidates");
  // the `want` smallest keys first (linear-time selection), then only those sorted
  const auto key_less = [](const KeyCand& a, const KeyCand& b) { return a.e != b.e ? a.e < b.e : a.rank < b.rank; };
  std::nth_element(h.begin(), h.begin() + (want - 1), h.end(), key_less);
  std::sort(h.begin(), h.begin() + want, key_less);
  for (uint64_t i = 0; i < want; ++i) {
    out_energies[i] = (double)h[i].e;
    for (int v = 0; v < n; ++v) out_x[i * n + v] = (uint8_t)((h[i].rank >> (n - 1 - v)) & 1u);
  }
  *out_count = (int)want;
  record_launch_count(launches);
  return QUBO_OK;
}
