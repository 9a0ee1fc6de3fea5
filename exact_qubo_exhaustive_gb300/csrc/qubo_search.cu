// Fold/validate, cache construction, reductions and the launch sequence of one search.
#include <cstring>

#include "qubo_search_kernel.cuh"
#include "qubo_seed.cuh"

namespace qgb {

// ------------------------------------------------------------------------------------------------
// Fold Q to the upper triangle and validate (one block).
//   int32: U_ii = Q_ii, U_ij = Q_ij + Q_ji (i < j) in int64; S = sum |U_ij| must be <= 2^30 - 1.
//   fp32/fp64: every entry finite; U64 folded in fp64; the int32 image is round(U64 * 2^s) with the
//          largest s keeping sum |image| <= 2^22 - 1 (the range of the biased fp32 minimum pass).
//          A state's image energy then differs from 2^s times its energy by at most
//          (#selected terms)/2 <= n(n+1)/4, so every fp64 minimiser lies within
//          band = n(n+1)/2 image units of the image minimum.
// ------------------------------------------------------------------------------------------------
// gthr (optional, ngroups entries): the pruned minimum passes' per-group best, started at
// sum |U_ij| of the int32 image, which no energy exceeds.
__global__ void __launch_bounds__(256) prep_kernel(int n, int dtype, const void* __restrict__ Qv, DevHeader* hdr,
                                                   int32_t* U, double* U64, uint64_t* gbase0,
                                                   uint64_t gbase0_value, int32_t* gthr, int ngroups) {
  __shared__ unsigned long long s_sum;
  __shared__ int s_bad;
  __shared__ double s_part[256];
  const int tid = threadIdx.x, nt = blockDim.x;
  const int nn = n * n;
  if (tid == 0) {
    s_sum = 0;
    s_bad = 0;
    if (gbase0) *gbase0 = gbase0_value;
  }
  __syncthreads();
  if (dtype == QUBO_INT32) {
    const int32_t* Q = static_cast<const int32_t*>(Qv);
    unsigned long long local = 0;
    for (int idx = tid; idx < nn; idx += nt) {
      const int i = idx / n, j = idx - (idx / n) * n;
      long long u = 0;
      if (j == i) u = Q[idx];
      else if (j > i) u = (long long)Q[idx] + (long long)Q[j * n + i];
      local += (unsigned long long)(u < 0 ? -u : u);
      U[idx] = (int32_t)u;  // only used when the range check passes
    }
    atomicAdd(&s_sum, local);
    __syncthreads();
    if (tid == 0) {
      hdr->abs_sum = (int64_t)s_sum;
      hdr->abs_sum64 = (double)s_sum;
      hdr->scale_exp = 0;
      hdr->band = 0;
      hdr->tied_count = 0;
      hdr->status = (s_sum > (unsigned long long)kMaxAbsSum) ? QUBO_ERR_RANGE : QUBO_OK;
    }
    if (gthr) {
      const int32_t top = (int32_t)(s_sum < (unsigned long long)kMaxAbsSum ? s_sum : (unsigned long long)kMaxAbsSum);
      for (int g = tid; g < ngroups; g += nt) gthr[g] = top;
    }
    return;
  }
  // fp32 / fp64
  const float* Qf = static_cast<const float*>(Qv);
  const double* Qd = static_cast<const double*>(Qv);
  auto load = [&](int idx) -> double { return dtype == QUBO_FP64 ? Qd[idx] : (double)Qf[idx]; };
  double local = 0.0;
  int bad = 0;
  for (int idx = tid; idx < nn; idx += nt) {
    const int i = idx / n, j = idx - (idx / n) * n;
    const double a = load(idx);
    if (!isfinite(a)) bad = 1;
    double u = 0.0;
    if (j == i) u = a;
    else if (j > i) u = __dadd_rn(a, load(j * n + i));
    U64[idx] = u;
    local += fabs(u);
  }
  if (bad) atomicOr(&s_bad, 1);
  s_part[tid] = local;
  __syncthreads();
  for (int h = nt / 2; h > 0; h >>= 1) {  // fixed-order tree: deterministic
    if (tid < h) s_part[tid] += s_part[tid + h];
    __syncthreads();
  }
  const double S64 = s_part[0];
  __shared__ int s_scale;
  const int npairs = n * (n + 1) / 2;
  if (tid == 0) {
    int sc = 0;
    if (S64 > 0.0) {
      int e;
      frexp((double)(kBiasedWalkMaxAbsSum - npairs) / S64, &e);  // ratio = m * 2^e, m in [0.5, 1)
      sc = e - 1;
      sc = sc > 1074 ? 1074 : (sc < -1074 ? -1074 : sc);
    }
    s_scale = sc;
  }
  __syncthreads();
  // Exact check of the quantised sum; step the scale down until it fits (at most a few times).
  for (int attempt = 0; attempt < 4; ++attempt) {
    const int sc = s_scale;
    unsigned long long q = 0;
    for (int idx = tid; idx < nn; idx += nt) {
      const long long v = __double2ll_rn(ldexp(U64[idx], sc));
      q += (unsigned long long)(v < 0 ? -v : v);
    }
    if (tid == 0) s_sum = 0;
    __syncthreads();
    atomicAdd(&s_sum, q);
    __syncthreads();
    const bool fits = s_sum <= (unsigned long long)kBiasedWalkMaxAbsSum;
    __syncthreads();
    if (fits) break;
    if (tid == 0) s_scale = sc - 1;
    __syncthreads();
  }
  const int sc = s_scale;
  for (int idx = tid; idx < nn; idx += nt) U[idx] = (int32_t)__double2ll_rn(ldexp(U64[idx], sc));
  if (tid == 0) {
    hdr->abs_sum = (int64_t)s_sum;
    hdr->abs_sum64 = S64;
    hdr->scale_exp = sc;
    hdr->band = npairs;
    hdr->tied_count = 0;
    hdr->status = s_bad ? QUBO_ERR_NONFINITE
                        : (s_sum <= (unsigned long long)kBiasedWalkMaxAbsSum ? QUBO_OK : QUBO_ERR_RANGE);
  }
  if (gthr) {
    const int32_t top = (int32_t)(s_sum < (unsigned long long)kMaxAbsSum ? s_sum : (unsigned long long)kMaxAbsSum);
    for (int g = tid; g < ngroups; g += nt) gthr[g] = top;
  }
}

// ------------------------------------------------------------------------------------------------
// The energy-component cache (§II-C Table I, Alg. 2 preprocessing), computed directly:
//   M[v][j]  = sum_{cached b} U[v][b] x_b(j)        interaction rows M_int, v < n - C
//   Ec[j]    = sum_{cached a <= b} U[a][b] x_a x_b  E(U_B), the suffix energies
//   T[i]     = E of the walked variables at gray(i) (Gray-ordered prefix energies, §IV-B.3)
//   T2[i]    = (T[i] mod 2^16) in both 16-bit halves (packed pass; optional)

// ------------------------------------------------------------------------------------------------
__global__ void tables_kernel(int n, int C, int F, int w, const DevHeader* __restrict__ hdr,
                              const int32_t* __restrict__ U, int32_t* M, int32_t* Ec, int32_t* T, uint32_t* T2,
                              uint64_t nTpad) {
  if (hdr->status != QUBO_OK) return;
  const int ncols = 1 << C;
  const uint64_t nM = (uint64_t)(n - C) << C;
  const uint64_t nE = (uint64_t)ncols;
  const uint64_t total = nM + nE + nTpad;
  const int base_c = n - C;  // first cached variable
  for (uint64_t idx = blockIdx.x * (uint64_t)blockDim.x + threadIdx.x; idx < total;
       idx += (uint64_t)gridDim.x * blockDim.x) {
    if (idx < nM) {
      const int v = (int)(idx >> C);
      const int j = (int)(idx & (ncols - 1));
      int acc = 0;
      for (int b = 0; b < C; ++b)
        if ((j >> b) & 1) acc += U[v * n + (n - 1 - b)];
      M[idx] = acc;
    } else if (idx < nM + nE) {
      const int j = (int)(idx - nM);
      int acc = 0;
      for (int a = base_c; a < n; ++a) {
        if (!((j >> (n - 1 - a)) & 1)) continue;
        for (int b = a; b < n; ++b)
          if ((j >> (n - 1 - b)) & 1) acc += U[a * n + b];
      }
      Ec[j] = acc;
    } else {
      const uint64_t i = idx - nM - nE;
      if (i >= ((uint64_t)1 << w)) {
        T[i] = 0;
        if (T2) T2[i] = 0;
        continue;
      }
      const uint64_t g = i ^ (i >> 1);
      // Gray position a drives variable n - C - 1 - a; walked variables are F .. n - C - 1.
      int acc = 0;
      for (int a = 0; a < w; ++a) {
        if (!((g >> a) & 1u)) continue;
        const int va = n - C - 1 - a;
        for (int b = a; b < w; ++b)
          if ((g >> b) & 1u) acc += U[(n - C - 1 - b) * n + va];  // n-C-1-b <= va
      }
      T[i] = acc;
      if (T2) T2[i] = ((uint32_t)acc & 0xffffu) * 0x10001u;
    }
  }
}

// ------------------------------------------------------------------------------------------------
// Block table of the block-bounded minimum pass (one thread per block of 2^R Gray steps):
//   blk[m] = the least T of block m, and the flip that follows it: position R + ctz(m + 1),
//            which becomes set unless bit ctz(m + 1) + 1 of m + 1 is set (reflected Gray code);
//            its shared row's float4 offset, sign, and the index of +L or -L of its variable in
//            the walker's linear-term table. blk[nb - 1] and the padding entry blk[nb]: no flip.
// seed (optional): the best energy of a group that holds the unit with prefix 0; every T[i] is
// the energy of a state of that unit (prefix 0, cached variables 0), so min T may start it.
// ------------------------------------------------------------------------------------------------
__global__ void block_table_kernel(int n, int C, int w, int R, const DevHeader* __restrict__ hdr,
                                   const int32_t* __restrict__ T, BlockCtl* blk, int32_t* seed,
                                   int32_t* unit_min, uint64_t total_units) {
  if (hdr->status != QUBO_OK) return;
  // the bounded passes publish unit minima with atomics: they start at INT_MAX
  for (uint64_t u = blockIdx.x * (uint64_t)blockDim.x + threadIdx.x; u < total_units;
       u += (uint64_t)gridDim.x * blockDim.x)
    unit_min[u] = kIntInf;
  const uint32_t nb = 1u << (w - R);
  for (uint32_t m = blockIdx.x * blockDim.x + threadIdx.x; m <= nb; m += gridDim.x * blockDim.x) {
    const uint32_t mm = m < nb ? m : nb - 1;
    const int4* T4 = reinterpret_cast<const int4*>(T + ((size_t)mm << R));
    int tmin = kIntInf;
    for (int q = 0; q < (1 << R) / 4; ++q) {
      const int4 t = T4[q];
      tmin = min(tmin, __vimin3_s32(t.x, t.y, min(t.z, t.w)));
    }
    if (seed && m < nb) atomicMin(seed, tmin);
    BlockCtl b;
    b.tmin = tmin;
    if (m + 1 < nb) {
      const int rr = __ffs((int)(m + 1)) - 1;
      const bool up = !(((m + 1) >> (rr + 1)) & 1u);
      b.row = rr << (C - 2);
      b.dsgn = up ? 1.f : -1.f;
      b.lvx = (up ? 0 : 64) + (n - C - 1 - (R + rr));
    } else {
      b.row = 0;
      b.dsgn = 0.f;
      b.lvx = 128;
    }
    blk[m] = b;
  }
}

// Single-group searches (a whole problem or a slice range): greedy one-flip descents
// (warp_descent), one per warp; the least energy reached lowers the group's starting best of the
// bounded minimum pass (gthr), so that the first units already skip most blocks. With F > 0 the
// first F variables stay fixed to a unit prefix of the group, so that every state reached lies in
// the group; with F = 0 (a whole problem) every variable may flip.
constexpr int kSeedBlocks = 32, kSeedThreads = 128;  // 128 descents
__global__ void __launch_bounds__(kSeedThreads) descent_seed_kernel(int n, int F, uint64_t upg,
                                                                   const DevHeader* __restrict__ hdr,
                                                                   const int32_t* __restrict__ U,
                                                                   const uint64_t* __restrict__ gbase, int32_t* gthr) {
  __shared__ int32_t sU[kSeedMaxN * kSeedMaxN];
  if (hdr->status != QUBO_OK || n > kSeedMaxN || F >= n) return;
  for (int idx = threadIdx.x; idx < n * n; idx += blockDim.x) {
    const int i = idx / n, j = idx - i * n;
    sU[idx] = (j >= i) ? U[idx] : U[j * n + i];  // symmetric: sU[i][j] = U[min(i,j)][max(i,j)]
  }
  __syncthreads();
  const int32_t e = warp_descent(sU, n, F, gbase[0], upg, (blockIdx.x * blockDim.x + threadIdx.x) / 32);
  if ((threadIdx.x & 31) == 0) atomicMin(gthr, e);
}

// ------------------------------------------------------------------------------------------------
// Per-group minimum over its units (one block per group), and accumulator reset.
// ------------------------------------------------------------------------------------------------
__global__ void __launch_bounds__(256) group_min_kernel(KParams p) {
  __shared__ int s_red[8];
  if (p.hdr->status != QUBO_OK) return;
  for (int g = blockIdx.x; g < p.ngroups; g += gridDim.x) {
    int m = kIntInf;
    for (uint64_t x = threadIdx.x; x < p.upg; x += blockDim.x) m = min(m, p.unit_min[(uint64_t)g * p.upg + x]);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) m = min(m, __shfl_xor_sync(0xffffffffu, m, off));
    if ((threadIdx.x & 31) == 0) s_red[threadIdx.x >> 5] = m;
    __syncthreads();
    if (threadIdx.x == 0) {
      for (int k = 1; k < (int)(blockDim.x >> 5); ++k) m = min(m, s_red[k]);
      p.gmin[g] = m;
      p.grank[g] = ~0ull;
      p.gties[g] = 0;
      p.gkey[g] = ~0ull;
    }
    __syncthreads();
  }
  if (blockIdx.x == 0 && threadIdx.x == 0) p.hdr->tied_count = 0;
}

// Units whose minimum is within the band of their group's minimum (order does not matter:
// every later combination is commutative).
__global__ void tie_list_kernel(KParams p, uint64_t total_units) {
  if (p.hdr->status != QUBO_OK) return;
  const int band = p.hdr->band;
  for (uint64_t u = blockIdx.x * (uint64_t)blockDim.x + threadIdx.x; u < total_units;
       u += (uint64_t)gridDim.x * blockDim.x) {
    const uint64_t g = u / p.upg;
    if (p.unit_min[u] <= p.gmin[g] + band) {
      const unsigned idx = atomicAdd(&p.hdr->tied_count, 1u);
      p.tied[idx] = (uint32_t)u;
    }
  }
}

__global__ void finalize_kernel(KParams p, qubo_result* out) {
  const int g = blockIdx.x * blockDim.x + threadIdx.x;
  if (g >= p.ngroups) return;
  const int st = p.hdr->status;
  qubo_result r;
  r.status = st;
  r.reserved = 0;
  r.min_energy = 0.0;
  r.argmin_rank = 0;
  r.tie_count = 0;
  if (st == QUBO_OK) {
    r.min_energy = (p.dtype == QUBO_INT32) ? (double)p.gmin[g] : key_to_double(p.gkey[g]);
    r.argmin_rank = p.grank[g];
    r.tie_count = p.gties[g];
  }
  out[g] = r;
}

// ------------------------------------------------------------------------------------------------
// Workspace layout.
// ------------------------------------------------------------------------------------------------
static size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

Work layout_workspace(const Plan& p, unsigned char* base) {
  Work w;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    unsigned char* ptr = base ? base + off : nullptr;
    off += align256(bytes);
    return ptr;
  };
  const size_t nn = (size_t)p.n * p.n;
  const size_t ncols = (size_t)1 << p.C;
  const size_t nT = ((size_t)1 << p.w) < 4 ? 4 : ((size_t)1 << p.w);
  w.hdr = reinterpret_cast<DevHeader*>(take(sizeof(DevHeader)));
  w.U = reinterpret_cast<int32_t*>(take(nn * 4));
  w.U64 = reinterpret_cast<double*>(take(p.dtype != QUBO_INT32 ? nn * 8 : 8));
  w.M = reinterpret_cast<int32_t*>(take((size_t)(p.n - p.C > 0 ? p.n - p.C : 1) * ncols * 4));
  w.Ec = reinterpret_cast<int32_t*>(take(ncols * 4 < 16 ? 16 : ncols * 4));
  w.T = reinterpret_cast<int32_t*>(take(nT * 4));
  if (p.packed || p.packed_pruned) w.T2 = reinterpret_cast<uint32_t*>(take(nT * 4));
  if (p.prune) {
    w.blk = reinterpret_cast<BlockCtl*>(take(((nT >> p.prune_r) + 1) * sizeof(BlockCtl)));
    w.gthr = reinterpret_cast<int32_t*>(take((size_t)p.ngroups * 4));
  }
  w.unit_min = reinterpret_cast<int32_t*>(take(p.total_units * 4));
  w.tied = reinterpret_cast<uint32_t*>(take(p.total_units * 4));
  w.gbase = reinterpret_cast<uint64_t*>(take((size_t)p.ngroups * 8));
  w.gmin = reinterpret_cast<int32_t*>(take((size_t)p.ngroups * 4));
  w.grank = reinterpret_cast<uint64_t*>(take((size_t)p.ngroups * 8));
  w.gties = reinterpret_cast<uint64_t*>(take((size_t)p.ngroups * 8));
  w.gkey = reinterpret_cast<uint64_t*>(take((size_t)p.ngroups * 8));
  w.results = reinterpret_cast<qubo_result*>(take((size_t)p.ngroups * sizeof(qubo_result)));
  w.bytes = off;
  return w;
}

// ------------------------------------------------------------------------------------------------
// Launch sequence: prep -> tables -> min pass -> group minima -> tied units -> resolve -> results.
// ------------------------------------------------------------------------------------------------
static cudaError_t launch_search(const Plan& p, int mode, const KParams& kp, int blocks, cudaStream_t s) {
  if (p.variant == kFast) return launch_search_fast(mode, kp, blocks, p.threads, p.smem_bytes, s);
  return launch_search_generic(mode, kp, blocks, p.threads, p.smem_bytes, s);
}

// Fold, tables and the minimum pass (unit minima in w.unit_min); fills kp for later passes.
// Returns with *aborted set (and nothing further enqueued) when a cancellation is seen.
static cudaError_t run_front(const Plan& p, const void* d_Q, const Work& w, qubo_result* res, cudaStream_t stream,
                             int& nl, const volatile int* abort_flag, bool* aborted, const KernelTiming* timing,
                             KParams& kp) {
  cudaError_t e;
  // gbase: uploaded by the host for slices and ranges; otherwise one group starting at unit 0,
  // written by the prep kernel.
  prep_kernel<<<1, 256, 0, stream>>>(p.n, p.dtype, d_Q, w.hdr, w.U, w.U64, p.host_gbase ? nullptr : w.gbase,
                                     p.gbase0, w.gthr, p.ngroups);
  ++nl;
  if ((e = cudaGetLastError()) != cudaSuccess) return e;

  const uint64_t nTpad = ((uint64_t)1 << p.w) < 4 ? 4 : ((uint64_t)1 << p.w);
  const uint64_t tab_work = ((uint64_t)(p.n - p.C) << p.C) + ((uint64_t)1 << p.C) + nTpad;
  const int tab_blocks = (int)((tab_work + 255) / 256 < 4096 ? (tab_work + 255) / 256 : 4096);
  tables_kernel<<<tab_blocks, 256, 0, stream>>>(p.n, p.C, p.F, p.w, w.hdr, w.U, w.M, w.Ec, w.T, w.T2, nTpad);
  ++nl;
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  if (p.prune) {
    const uint32_t nb = 1u << (p.w - p.prune_r);
    // one group that holds unit 0 seeds its best with the least walked energy (the energies of
    // states of unit 0)
    const bool from_unit0 = !p.host_gbase && p.gbase0 == 0 && p.ngroups == 1;
    int32_t* seed = from_unit0 ? w.gthr : nullptr;
    block_table_kernel<<<(nb + 1 + 127) / 128, 128, 0, stream>>>(p.n, p.C, p.w, p.prune_r, w.hdr, w.T, w.blk, seed,
                                                                  w.unit_min, p.total_units);
    ++nl;
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    if (p.ngroups == 1) {
      // descents over every variable when the group is all units, else with its prefix fixed
      const bool all_units = from_unit0 && p.upg == ((uint64_t)1 << p.F);
      descent_seed_kernel<<<kSeedBlocks, kSeedThreads, 0, stream>>>(p.n, all_units ? 0 : p.F, p.upg, w.hdr, w.U,
                                                                    w.gbase, w.gthr);
      ++nl;
      if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
  }

  memset(&kp, 0, sizeof(kp));
  kp.n = p.n;
  kp.C = p.C;
  kp.F = p.F;
  kp.w = p.w;
  kp.dtype = p.dtype;
  kp.biased_active = p.biased ? 1 : 0;
  kp.packed_active = (p.packed || p.packed_pruned) ? 1 : 0;
  kp.seg_bits = p.seg_bits;
  kp.ngroups = p.ngroups;
  kp.upg = p.upg;
  kp.hdr = w.hdr;
  kp.U = w.U;
  kp.U64 = w.U64;
  kp.M = w.M;
  kp.Ec = w.Ec;
  kp.T = w.T;
  kp.T2 = w.T2;
  kp.blk = w.blk;
  kp.margin = p.bound_margin;
  kp.one = 1;
  kp.gthr = w.gthr;
  kp.gbase = w.gbase;
  kp.unit_min = w.unit_min;
  kp.tied = w.tied;
  kp.gmin = w.gmin;
  kp.grank = w.grank;
  kp.gties = w.gties;
  kp.gkey = w.gkey;
  kp.results = res;

  // Min pass, in chunks so that a cancellation request is seen between launches of long runs.
  const uint64_t states_per_unit = (uint64_t)1 << (p.n - p.F);
  uint64_t chunk = p.total_units;
  const uint64_t max_states_per_launch = (uint64_t)1 << 41;
  if (states_per_unit > 0 && p.total_units * states_per_unit > max_states_per_launch) {
    chunk = max_states_per_launch / states_per_unit;
    if (chunk < (uint64_t)p.blocks) chunk = p.blocks;
  }
  if (timing && (e = cudaEventRecord(timing->start, stream)) != cudaSuccess) return e;
  for (uint64_t u0 = 0; u0 < p.total_units; u0 += chunk) {
    if (abort_flag && *abort_flag) {
      if (aborted) *aborted = true;
      return cudaSuccess;
    }
    kp.unit_begin = u0;
    kp.unit_end = (u0 + chunk < p.total_units) ? u0 + chunk : p.total_units;
    const uint64_t nunits = kp.unit_end - kp.unit_begin;
    const int blocks = (int)(nunits < (uint64_t)p.blocks ? nunits : (uint64_t)p.blocks);
    if (p.packed_pruned) {
      // packed 16x2 CUDA-core pass with block bounds (exits at once unless it owns the minimum
      // pass) ...
      const int pb = (int)(nunits < (uint64_t)p.packed_pruned_blocks ? nunits : (uint64_t)p.packed_pruned_blocks);
      if ((e = launch_search_packed_pruned(p.prune_r, kp, pb, p.packed_pruned_smem, stream)) != cudaSuccess) return e;
      ++nl;
    } else if (p.packed) {
      // packed 16x2 CUDA-core pass (exits at once unless it owns the minimum pass) ...
      const int pb = (int)(nunits < (uint64_t)p.packed_blocks ? nunits : (uint64_t)p.packed_blocks);
      if ((e = launch_search_packed(kp, pb, p.packed_threads, p.packed_smem, stream)) != cudaSuccess) return e;
      ++nl;
    }
    if (p.biased) {
      // biased-binade CUDA-core pass, with block bounds where planned (exits at once unless it
      // owns the minimum pass) ...
      e = p.prune ? launch_search_biased_pruned(p.prune_r, kp, blocks, p.threads, p.smem_bytes, stream)
                  : launch_search_biased(kp, blocks, p.threads, p.smem_bytes, stream);
      if (e != cudaSuccess) return e;
      ++nl;
    }
    // ... and the int32 CUDA-core pass, with block bounds where planned (exits at once when
    // another pass ran)
    if (p.prune) {
      if ((e = launch_search_int_pruned(p.prune_r, kp, blocks, p.threads, p.smem_bytes, stream)) != cudaSuccess)
        return e;
    } else if (p.variant == kFast && p.w >= kIntMinR + 1) {
      if ((e = launch_search_int_min5(kp, blocks, p.threads, p.smem_bytes, stream)) != cudaSuccess) return e;
    } else if ((e = launch_search(p, kModeMin, kp, blocks, stream)) != cudaSuccess) {
      return e;
    }
    ++nl;
    if (kp.unit_end < p.total_units && abort_flag) {
      // long run: wait for this chunk so a cancellation request is honoured promptly
      if ((e = cudaStreamSynchronize(stream)) != cudaSuccess) return e;
    }
  }

  if (timing && (e = cudaEventRecord(timing->stop, stream)) != cudaSuccess) return e;
  return cudaSuccess;
}

cudaError_t run_search(const Plan& p, const void* d_Q, const Work& w, qubo_result* res, cudaStream_t stream,
                       int* launches, const volatile int* abort_flag, bool* aborted, const KernelTiming* timing) {
  int nl = 0;
  bool stop = false;
  KParams kp;
  cudaError_t e = run_front(p, d_Q, w, res, stream, nl, abort_flag, &stop, timing, kp);
  if (aborted) *aborted = stop;
  if (e != cudaSuccess || stop) {
    if (launches) *launches = nl;
    return e;
  }
  const int gblocks = p.ngroups < 1024 ? p.ngroups : 1024;
  group_min_kernel<<<gblocks, 256, 0, stream>>>(kp);
  ++nl;
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  const uint64_t tl_blocks64 = (p.total_units + 255) / 256;
  const int tl_blocks = (int)(tl_blocks64 < 4096 ? tl_blocks64 : 4096);
  tie_list_kernel<<<tl_blocks, 256, 0, stream>>>(kp, p.total_units);
  ++nl;
  if ((e = cudaGetLastError()) != cudaSuccess) return e;

  if (p.dtype == QUBO_INT32) {
    if ((e = launch_search(p, kModeTiesInt, kp, p.blocks, stream)) != cudaSuccess) return e;
    ++nl;
  } else {
    if ((e = launch_search(p, kModeKeyFp, kp, p.blocks, stream)) != cudaSuccess) return e;
    ++nl;
    if ((e = launch_search(p, kModeTiesFp, kp, p.blocks, stream)) != cudaSuccess) return e;
    ++nl;
  }
  finalize_kernel<<<(p.ngroups + 127) / 128, 128, 0, stream>>>(kp, res);
  ++nl;
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  if (launches) *launches = nl;
  return cudaSuccess;
}

// ------------------------------------------------------------------------------------------------
// Stages for drivers that decide between passes on the host (the k lowest energies).
// ------------------------------------------------------------------------------------------------
cudaError_t run_min_stage(const Plan& p, const void* d_Q, const Work& w, cudaStream_t stream, int* launches,
                          KParams* kp_out) {
  int nl = 0;
  bool stop = false;
  cudaError_t e = run_front(p, d_Q, w, nullptr, stream, nl, nullptr, &stop, nullptr, *kp_out);
  if (launches) *launches = nl;
  return e;
}

cudaError_t run_key_pass(const Plan& p, const KParams& base, int mode, int theta, uint64_t rho, KeyCand* cand,
                         uint32_t cap, unsigned long long* counter, cudaStream_t stream) {
  KParams kp = base;
  kp.theta = theta;
  kp.rho = rho;
  kp.cand = cand;
  kp.cand_cap = cap;
  kp.cand_count = counter;
  return launch_search(p, mode, kp, p.blocks, stream);
}

}  // namespace qgb
