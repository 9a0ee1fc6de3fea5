// Batched mode: many independent QUBO instances of equal size, one thread block per instance
// (independent subproblems, §III-C1; one problem per block). Each block folds its instance,
// builds the energy-component cache in shared memory (§II-C), walks every state with the same
// register walker as the single-problem kernel, records per-(warp, segment) minima, and then
// re-walks only the segments whose minimum equals the instance minimum to find the lowest
// rank and the tie count.
#include <algorithm>
#include <cstring>
#include <type_traits>

#include "qubo_packed_walk.cuh"
#include "qubo_seed.cuh"
#include "qubo_walk.cuh"

namespace qgb {

namespace {
constexpr int kBatchMaxN = 25;
constexpr int kBatchSegs = 32;  // segments per instance walk

__device__ __forceinline__ int fold_entry(const int32_t* Q, int n, int i, int j, long long* u) {
  long long v = 0;
  if (j == i) v = Q[i * n + i];
  else if (j > i) v = (long long)Q[i * n + j] + (long long)Q[j * n + i];
  *u = v;
  return 0;
}

// Direct value of M[v][j] and E_cached(j) from the folded triangle in shared memory.
__device__ __forceinline__ int m_entry(const int* sU, int n, int v, int j, int C) {
  int acc = 0;
  for (int b = 0; b < C; ++b)
    if ((j >> b) & 1) acc += sU[v * n + (n - 1 - b)];
  return acc;
}
__device__ __forceinline__ int ec_entry(const int* sU, int n, int j, int C) {
  int acc = 0;
  for (int b1 = C - 1; b1 >= 0; --b1) {
    if (!((j >> b1) & 1)) continue;
    const int a = n - 1 - b1;
    for (int b2 = b1; b2 >= 0; --b2)
      if ((j >> b2) & 1) acc += sU[a * n + (n - 1 - b2)];
  }
  return acc;
}

// Running energies and register rows of thread t (columns of the fast layout), directly.
template <class W>
__device__ __forceinline__ void direct_init(W& wk, const int* sU, int n, int C, int nthreads, int t) {
  wk.s = 0;
  wk.cnt = 0;
  wk.rmin = ~0ull;
  wk.kmin = ~0ull;
  wk.valid = true;
  wk.col0 = 0;
#pragma unroll
  for (int jj = 0; jj < kFastCPT; ++jj) {
    const int j = column_of<kFastCPT>(t, nthreads, jj);
    wk.V[jj] = ec_entry(sU, n, j, C);
#pragma unroll
    for (int a = 0; a < kFastR; ++a) wk.Row[a][jj] = m_entry(sU, n, n - C - 1 - a, j, C);
  }
}

__global__ void __launch_bounds__(256, 1) batched_kernel(int n, int C, const int32_t* __restrict__ Qall,
                                                         qubo_result* __restrict__ out) {
  extern __shared__ __align__(16) int4 smem4[];
  __shared__ int sL[64];
  __shared__ int s_segmin[8 * kBatchSegs];
  __shared__ unsigned long long s_sum, s_cnt, s_rmin;
  __shared__ int s_best;
  __shared__ int s_ntied;
  __shared__ unsigned short s_tied[8 * kBatchSegs];

  const int tid = threadIdx.x, nthreads = blockDim.x;
  const int lane = tid & 31, warp = tid >> 5, nwarps = nthreads >> 5;
  const int w = n - C;
  const int ncols = 1 << C;
  const int nq = ncols >> 2;
  const int ndyn = w - kFastR;
  const int64_t niter = walk_iterations<kFastR>(w);
  const int64_t per = niter / kBatchSegs;

  // shared memory: [dyn rows: ndyn * nq int4][T: 2^w int][U: n*n int]
  int4* rows4 = smem4;
  int* sT = reinterpret_cast<int*>(rows4 + (size_t)ndyn * nq);
  int* sU = sT + (1 << w);

  const int32_t* Q = Qall + (size_t)blockIdx.x * n * n;
  if (tid == 0) {
    s_sum = 0;
    s_cnt = 0;
    s_rmin = ~0ull;
    s_ntied = 0;
  }
  if (tid < 64) sL[tid] = 0;  // no fixed variables: all linear terms are zero
  __syncthreads();
  unsigned long long local = 0;
  for (int idx = tid; idx < n * n; idx += nthreads) {
    long long u;
    fold_entry(Q, n, idx / n, idx % n, &u);
    local += (unsigned long long)(u < 0 ? -u : u);
    sU[idx] = (int)u;
  }
  atomicAdd(&s_sum, local);
  __syncthreads();
  if (s_sum > (unsigned long long)kMaxAbsSum) {
    if (tid == 0) {
      qubo_result r;
      r.status = QUBO_ERR_RANGE;
      r.reserved = 0;
      r.min_energy = 0.0;
      r.argmin_rank = 0;
      r.tie_count = 0;
      out[blockIdx.x] = r;
    }
    return;
  }
  // walked rows a >= R and the Gray-ordered walked energies
  for (int idx = tid; idx < ndyn * nq; idx += nthreads) {
    const int rr = idx / nq, q = idx - rr * nq;
    const int v = n - C - 1 - (kFastR + rr);
    int4 m;
    m.x = m_entry(sU, n, v, 4 * q + 0, C);
    m.y = m_entry(sU, n, v, 4 * q + 1, C);
    m.z = m_entry(sU, n, v, 4 * q + 2, C);
    m.w = m_entry(sU, n, v, 4 * q + 3, C);
    rows4[idx] = m;
  }
  for (int i = tid; i < (1 << w); i += nthreads) {
    const unsigned g = (unsigned)(i ^ (i >> 1));
    int acc = 0;
    for (int a = 0; a < w; ++a) {
      if (!((g >> a) & 1u)) continue;
      const int va = n - C - 1 - a;
      for (int b = a; b < w; ++b)
        if ((g >> b) & 1u) acc += sU[(n - C - 1 - b) * n + va];
    }
    sT[i] = acc;
  }
  __syncthreads();

  WalkCtx c{};
  c.n = n;
  c.C = C;
  c.F = 0;
  c.w = w;
  c.nthreads = nthreads;
  c.thread = tid;
  c.sL = sL;
  c.rows4 = rows4;
  c.rows1 = nullptr;
  c.T = sT;
  c.t_global = false;

  // ---- minimum pass, one segment at a time (the walk continues across segments)
  {
    Walker<kFastCPT, kFastR, kModeMin> W;
    direct_init(W, sU, n, C, nthreads, tid);
    for (int seg = 0; seg < kBatchSegs; ++seg) {
      W.aux = kIntInf;
      W.walk(c, seg * per, (seg + 1) * per, niter, 0, nullptr, 0);
      int best = W.aux + W.s;
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) best = min(best, __shfl_xor_sync(0xffffffffu, best, off));
      if (lane == 0) s_segmin[warp * kBatchSegs + seg] = best;
    }
  }
  __syncthreads();
  if (tid == 0) {
    int b = kIntInf;
    for (int k = 0; k < nwarps * kBatchSegs; ++k) b = min(b, s_segmin[k]);
    s_best = b;
    int nt = 0;
    for (int k = 0; k < nwarps * kBatchSegs; ++k)
      if (s_segmin[k] == b) s_tied[nt++] = (unsigned short)k;
    s_ntied = nt;
  }
  __syncthreads();
  const int best = s_best;

  // ---- resolve: each tied (warp, segment) pair, split into its iterations, spread over warps
  {
    const int nitems = s_ntied * (int)per;
    for (int item = warp; item < nitems; item += nwarps) {
      const int pair = s_tied[item / (int)per];
      const int tw = pair / kBatchSegs, seg = pair % kBatchSegs;
      const int64_t it0 = seg * per + (item % (int)per);
      WalkCtx cw = c;
      cw.thread = tw * 32 + lane;  // emulate the columns of warp tw
      Walker<kFastCPT, kFastR, kModeTiesInt> W;
      direct_init(W, sU, n, C, nthreads, cw.thread);
      W.seek(cw, it0);
      W.aux = best - W.s;
      W.walk(cw, it0, it0 + 1, it0 + 1, 0, nullptr, 0);
      uint64_t cnt = W.cnt, rmin = W.rmin;
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) {
        cnt += __shfl_xor_sync(0xffffffffu, cnt, off);
        const uint64_t r2 = __shfl_xor_sync(0xffffffffu, rmin, off);
        rmin = r2 < rmin ? r2 : rmin;
      }
      if (lane == 0 && cnt) {
        atomicAdd(&s_cnt, (unsigned long long)cnt);
        atomicMin(&s_rmin, (unsigned long long)rmin);
      }
    }
  }
  __syncthreads();
  if (tid == 0) {
    qubo_result r;
    r.status = QUBO_OK;
    r.reserved = 0;
    r.min_energy = (double)best;
    r.argmin_rank = s_rmin;
    r.tie_count = s_cnt;
    out[blockIdx.x] = r;
  }
}

// ------------------------------------------------------------------------------------------------
// Table-based pipeline (18 <= n <= kBatchTabMaxN). Every instance gets the energy-component cache
// of the single-problem search in the workspace (the rows of M_int or their half-subset sums,
// E(U_B), the Gray-ordered walked energies), built by one kernel with a block per instance. Each
// instance is split into 2^F work units (§III-C1), and persistent minimum passes walk the units
// of every instance with the same walkers as the single-problem kernels: the packed 16x2 pass,
// the biased fp32-binade pass or the int32 pass, chosen per instance by its sum |U| (a pass skips
// the instances it does not own). A last pass re-walks, for the lowest rank and the tie count,
// only the parts that reach their instance's minimum: the iterations (packed pass, which records
// every iteration's minimum) or the units (the other passes).
// ------------------------------------------------------------------------------------------------
constexpr int kBatchTabMaxN = 32;
constexpr int kPackedTiesR = 4;  // register rows of the packed re-walk of the minimum iterations
static_assert(kPackedTiesR <= kPackedR, "a minimum-pass iteration is a whole number of re-walk iterations");
constexpr int kBatchMaxWalked = 11;     // walked bits per unit (plan_batched)
constexpr int kBatchMaxIters = 1 << (kBatchMaxWalked - kPackedR - 1);  // packed iterations per unit
constexpr int kBatchTabC = 12;
// The bounded packed pass walks blocks of 2^kBatchPruneR steps: one iteration of the packed
// minimum pass (kPackedR register rows), so its block minima index the same re-walk table.
constexpr int kBatchPruneR = kPackedR + 1;
static_assert(kBatchTabC == 12, "packed::HalfRows splits the cached bits 6 + 6");

struct BatchTables {
  int batch, n, C, F, w;
  const int32_t* Q;
  int32_t* U;  // batch x n*n        folded triangle
  int32_t* M;  // batch x (n-C)*2^C  interaction rows (instances of the biased and int32 passes)
  int32_t* H;  // batch x (n-C)*128  half-subset sums of the rows (packed pass: M[v][j] from two)
  int32_t* Ec; // batch x 2^C        cached self energies
  int32_t* T;  // batch x 2^w        walked energies in Gray order
  uint32_t* T2;  // batch x 2^w      T's low 16 bits in both halves (packed pass)
  int64_t* S;    // batch            sum |U|
  int32_t* status;
  int32_t* unit_min;  // batch x 2^F
  int32_t* seg_min;   // batch x 2^F x (packed iterations per unit): packed instances' iteration minima
  int32_t* gmin;
  unsigned long long* grank;
  unsigned long long* gties;
  BlockCtl* blk;      // batch x (2^(w - kBatchPruneR) + 1): block control tables (bounded packed pass)
  int32_t* gthr;      // batch: best energy published so far (bounded packed pass)
  int one;            // 1: the bounded walk derives its opaque constants from it
  size_t su, sm, sh, se, st;  // per-instance strides of U, M, H, Ec, T / T2
};

enum BatchClass : int { kBatchPacked = 0, kBatchBiased = 1, kBatchInt = 2 };

__device__ __forceinline__ int batch_class(int64_t S) {
  if (S <= kPackedMaxAbsSum) return kBatchPacked;
  if (S <= kBiasedWalkMaxAbsSum) return kBatchBiased;
  return kBatchInt;
}

// Fold, range check and caches of every instance (the single-problem tables, §II-C Table I), one
// block per instance. The C cached bits split into a low half (lo bits) and a high half, and the w
// walked bits likewise; with the partial sums of the halves in shared memory every table entry
// is a few adds:
//   M[v][j] = A_v[j_lo] + B_v[j_hi]                         (A, B: subset sums of U[v][cached])
//   E(U_B)[j] = El[j_lo] + Eh[j_hi] + sum_{b in j_lo} Y[j_hi][b]   (Y: coupling of a high subset
//                                                                   to low bit b)
//   T[i] = Tl[g_lo] + Th[g_hi] + sum_{a in g_lo} TY[g_hi][a]       (g = gray(i), walked bits)
constexpr int kBatchMaxHalf = 64;  // 2^(C/2) for C = kBatchTabC

__global__ void __launch_bounds__(256) btables_kernel(BatchTables b) {
  __shared__ int sU[kBatchTabMaxN * kBatchTabMaxN];
  __shared__ int sA[kBatchTabMaxN][kBatchMaxHalf];
  __shared__ int sB[kBatchTabMaxN][kBatchMaxHalf];
  __shared__ int sEl[kBatchMaxHalf], sEh[kBatchMaxHalf];
  __shared__ int sY[kBatchMaxHalf][kBatchTabC / 2];
  // the walked bits split the same way: wl low positions, wh high ones
  __shared__ int sTl[1 << (kBatchMaxWalked / 2)], sTh[1 << (kBatchMaxWalked - kBatchMaxWalked / 2)];
  __shared__ int sTY[1 << (kBatchMaxWalked - kBatchMaxWalked / 2)][kBatchMaxWalked / 2];
  __shared__ unsigned long long s_sum;
  const int g = blockIdx.x, tid = threadIdx.x, nt = blockDim.x;
  const int n = b.n, C = b.C, w = b.w;
  const int wl = w / 2, wh = w - wl;  // w <= kBatchMaxWalked (plan_batched)
  const int lo = C / 2, hi = C - lo;
  const int nlo = 1 << lo, nhi = 1 << hi;
  // U = the folded triangle of Q and S = sum |U|; the instance is searched when S fits int32
  if (tid == 0) s_sum = 0;
  __syncthreads();
  {
    const int32_t* Q = b.Q + (size_t)g * n * n;
    int32_t* U = b.U + (size_t)g * b.su;
    unsigned long long local = 0;
    for (int idx = tid; idx < n * n; idx += nt) {
      long long u;
      fold_entry(Q, n, idx / n, idx % n, &u);
      local += (unsigned long long)(u < 0 ? -u : u);
      sU[idx] = (int32_t)u;  // only used when the range check passes
      U[idx] = (int32_t)u;
    }
    atomicAdd(&s_sum, local);
  }
  __syncthreads();
  const int64_t S = (int64_t)s_sum;
  if (tid == 0) {
    b.S[g] = S;
    b.status[g] = S > kMaxAbsSum ? QUBO_ERR_RANGE : QUBO_OK;
    b.gmin[g] = kIntInf;
    b.grank[g] = ~0ull;
    b.gties[g] = 0;
  }
  if (S > kMaxAbsSum) return;
  const int nv = n - C;
  // cached bit k (0 = fastest) is variable n - 1 - k; low half k < lo, high half k >= lo
  for (int idx = tid; idx < nv * (nlo + nhi); idx += nt) {
    const int v = idx / (nlo + nhi), r = idx - v * (nlo + nhi);
    int acc = 0;
    if (r < nlo) {
      for (int k = 0; k < lo; ++k)
        if ((r >> k) & 1) acc += sU[v * n + (n - 1 - k)];
      sA[v][r] = acc;
    } else {
      const int h = r - nlo;
      for (int k = 0; k < hi; ++k)
        if ((h >> k) & 1) acc += sU[v * n + (n - 1 - (lo + k))];
      sB[v][h] = acc;
    }
  }
  for (int idx = tid; idx < nlo + nhi + nhi * lo; idx += nt) {
    if (idx < nlo) {  // energy of a low subset alone
      int acc = 0;
      for (int k1 = 0; k1 < lo; ++k1) {
        if (!((idx >> k1) & 1)) continue;
        const int a = n - 1 - k1;
        for (int k2 = k1; k2 < lo; ++k2)
          if ((idx >> k2) & 1) acc += sU[(n - 1 - k2) * n + a];  // n-1-k2 <= a
      }
      sEl[idx] = acc;
    } else if (idx < nlo + nhi) {  // energy of a high subset alone
      const int h = idx - nlo;
      int acc = 0;
      for (int k1 = 0; k1 < hi; ++k1) {
        if (!((h >> k1) & 1)) continue;
        const int a = n - 1 - (lo + k1);
        for (int k2 = k1; k2 < hi; ++k2)
          if ((h >> k2) & 1) acc += sU[(n - 1 - (lo + k2)) * n + a];
      }
      sEh[h] = acc;
    } else {  // coupling of high subset h to low bit k: sum_{k' in h} U[var(lo + k')][var(k)]
      const int r = idx - nlo - nhi, h = r / lo, k = r - h * lo;
      int acc = 0;
      for (int k2 = 0; k2 < hi; ++k2)
        if ((h >> k2) & 1) acc += sU[(n - 1 - (lo + k2)) * n + (n - 1 - k)];
      sY[h][k] = acc;
    }
  }
  // walked position a is variable n - C - 1 - a (a = 0 flips fastest)
  for (int idx = tid; idx < (1 << wl) + (1 << wh) + (1 << wh) * wl; idx += nt) {
    int acc = 0;
    if (idx < (1 << wl) + (1 << wh)) {  // energy of a low (or high) subset of walked positions alone
      const int base = idx < (1 << wl) ? 0 : wl, nb = idx < (1 << wl) ? wl : wh;
      const int sub = idx < (1 << wl) ? idx : idx - (1 << wl);
      for (int k1 = 0; k1 < nb; ++k1) {
        if (!((sub >> k1) & 1)) continue;
        const int va = n - C - 1 - (base + k1);
        for (int k2 = k1; k2 < nb; ++k2)
          if ((sub >> k2) & 1) acc += sU[(n - C - 1 - (base + k2)) * n + va];
      }
      if (idx < (1 << wl)) sTl[sub] = acc;
      else sTh[sub] = acc;
    } else {  // coupling of high subset h to low position a
      const int r = idx - (1 << wl) - (1 << wh), h = r / wl, a = r - h * wl;
      for (int k = 0; k < wh; ++k)
        if ((h >> k) & 1) acc += sU[(n - C - 1 - (wl + k)) * n + (n - C - 1 - a)];
      sTY[h][a] = acc;
    }
  }
  __syncthreads();
  const int ncols = 1 << C;
  if (batch_class(S) == kBatchPacked) {
    // the packed pass forms its rows from the half sums (packed::HalfRows): no M table
    int32_t* H = b.H + (size_t)g * b.sh;
    for (int idx = tid; idx < nv * packed::HalfRows::kStride; idx += nt) {
      const int v = idx / packed::HalfRows::kStride, r = idx % packed::HalfRows::kStride;
      H[idx] = r < 64 ? sA[v][r] : sB[v][r - 64];
    }
  } else {
    int32_t* M = b.M + (size_t)g * b.sm;
    for (int idx = tid; idx < nv * ncols; idx += nt) {
      const int v = idx >> C, j = idx & (ncols - 1);
      M[idx] = sA[v][j & (nlo - 1)] + sB[v][j >> lo];
    }
  }
  int32_t* Ec = b.Ec + (size_t)g * b.se;
  for (int j = tid; j < ncols; j += nt) {
    const int l = j & (nlo - 1), h = j >> lo;
    int acc = sEl[l] + sEh[h];
    for (int k = 0; k < lo; ++k)
      if ((l >> k) & 1) acc += sY[h][k];
    Ec[j] = acc;
  }
  int32_t* T = b.T + (size_t)g * b.st;
  uint32_t* T2 = b.T2 + (size_t)g * b.st;
  for (int i = tid; i < (1 << w); i += nt) {
    const unsigned gc = (unsigned)(i ^ (i >> 1));
    const int l = (int)(gc & ((1u << wl) - 1)), h = (int)(gc >> wl);
    int acc = sTl[l] + sTh[h];
    for (int a = 0; a < wl; ++a)
      if ((l >> a) & 1) acc += sTY[h][a];
    T[i] = acc;
    T2[i] = ((uint32_t)acc & 0xffffu) * 0x10001u;
  }
}

// Per-unit linear terms of instance g (F fixed bits), as unit_linear_terms of the main kernel.
__device__ __forceinline__ void bunit_terms(const int32_t* __restrict__ U, int n, int F, uint64_t P, int* sL) {
  for (int v = threadIdx.x; v < n; v += blockDim.x) {
    int acc = 0;
    if (v >= F) {
      for (int f = 0; f < F; ++f)
        if ((P >> (F - 1 - f)) & 1u) acc += U[f * n + v];
    } else if ((P >> (F - 1 - v)) & 1u) {
      for (int f2 = v; f2 < F; ++f2)
        if ((P >> (F - 1 - f2)) & 1u) acc += U[v * n + f2];
    }
    sL[v] = acc;
  }
}

// Minimum passes of the 16-column layout: VT = float (biased binade) or int; MODE kModeMin, or
// kModeTiesInt for the re-walk of the units at their instance's minimum.
template <int R, typename VT, int MODE>
__global__ void __launch_bounds__(256, 1) bwalk_kernel(BatchTables b) {
  extern __shared__ __align__(16) int4 s_rows4[];
  __shared__ int sL[64];
  __shared__ int s_red[32];
  __shared__ __align__(16) int s_slot[MODE != kModeMin ? kFastThreadsMax * kFastCPT : 4];
  constexpr int kClass = std::is_same<VT, float>::value ? kBatchBiased : kBatchInt;
  const int tid = threadIdx.x, nthreads = blockDim.x;
  const int n = b.n, C = b.C, F = b.F, w = b.w;
  const int nq = (1 << C) >> 2;
  const int ndyn = w - R;
  const uint64_t units = (uint64_t)b.batch << F;
  const int64_t niter = walk_iterations<R>(w);
  const int lane = tid & 31, warp = tid >> 5;
  int staged = -1;
  WalkCtx c{};
  c.n = n;
  c.C = C;
  c.F = F;
  c.w = w;
  c.nthreads = nthreads;
  c.thread = tid;
  c.sL = sL;
  c.rows4 = s_rows4;
  c.rows1 = nullptr;
  c.t_global = true;
  c.scratch = MODE != kModeMin ? reinterpret_cast<uint32_t*>(s_slot) : nullptr;
  // a contiguous range of units per block, so that a block stages each instance's rows once
  const uint64_t u_begin = units * blockIdx.x / gridDim.x, u_end = units * (blockIdx.x + 1) / gridDim.x;
  for (uint64_t u = u_begin, next; u < u_end; u = next) {
    const int g = (int)(u >> F);
    const uint64_t P = u & (((uint64_t)1 << F) - 1);
    next = u + 1;
    // instances this pass does not own are skipped whole (packed instances have their own re-walk)
    const bool owned = b.status[g] == QUBO_OK &&
                       (MODE == kModeMin ? batch_class(b.S[g]) == kClass : batch_class(b.S[g]) != kBatchPacked);
    if (!owned) {
      next = (uint64_t)(g + 1) << F;
      continue;
    }
    if (MODE != kModeMin && b.unit_min[u] != b.gmin[g]) continue;
    __syncthreads();  // the previous unit is done with sL and the staged rows
    if (g != staged) {
      const int4* M4 = reinterpret_cast<const int4*>(b.M + (size_t)g * b.sm);
#pragma unroll 8
      for (int idx = tid; idx < ndyn * nq; idx += nthreads) {
        const int rr = idx / nq, q = idx - rr * nq;
        const int v = n - C - 1 - (R + rr);
        const int4 m = M4[(size_t)v * nq + q];
        if constexpr (kClass == kBatchBiased)
          reinterpret_cast<float4*>(s_rows4)[idx] = make_float4((float)m.x, (float)m.y, (float)m.z, (float)m.w);
        else
          s_rows4[idx] = m;
      }
      staged = g;
    }
    const int32_t* U = b.U + (size_t)g * b.su;
    bunit_terms(U, n, F, P, sL);
    __syncthreads();
    int cP = 0;
    for (int f = 0; f < F; ++f) cP += sL[f];
    c.T = b.T + (size_t)g * b.st;
    const int32_t* Ec = b.Ec + (size_t)g * b.se;
    const int32_t* M = b.M + (size_t)g * b.sm;
    Walker<kFastCPT, R, MODE, VT> W;
    W.init(c, Ec, M, cP);
    if constexpr (MODE == kModeMin) {
      W.aux = kIntInf;
      W.walk(c, 0, niter, niter, 0, nullptr, 0);
      int best = W.aux - VOps<VT>::kBiasBits + W.s;
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) best = min(best, __shfl_xor_sync(0xffffffffu, best, off));
      if (lane == 0) s_red[warp] = best;
      __syncthreads();
      if (tid == 0) {
        int m = s_red[0];
        for (int k = 1; k < (nthreads >> 5); ++k) m = min(m, s_red[k]);
        b.unit_min[u] = m;
      }
    } else {
      W.aux = b.gmin[g] - W.s;
      const uint64_t prank = (F > 0) ? (P << (n - F)) : 0;
      W.walk(c, 0, niter, niter, prank, nullptr, 0);
      uint64_t cnt = W.cnt, rmin = W.rmin;
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) {
        cnt += __shfl_xor_sync(0xffffffffu, cnt, off);
        const uint64_t r2 = __shfl_xor_sync(0xffffffffu, rmin, off);
        rmin = r2 < rmin ? r2 : rmin;
      }
      if (lane == 0 && cnt) {
        atomicAdd(&b.gties[g], (unsigned long long)cnt);
        atomicMin(&b.grank[g], (unsigned long long)rmin);
      }
    }
  }
}

// Packed 16x2 passes over the units of the instances with sum |U| <= kPackedMaxAbsSum: the
// minimum (kModeMin) or the re-walk of the units at the instance minimum (kModeTiesInt).
template <int R, int MODE>
__global__ void __launch_bounds__(128, 2) bpacked_kernel(BatchTables b) {
  extern __shared__ __align__(16) int4 s_rows4[];
  __shared__ int sL[64];
  __shared__ int s_red[32];
  __shared__ __align__(16) int sH[(kBatchTabMaxN - kBatchTabC) * packed::HalfRows::kStride];
  __shared__ int s_seg[kBatchMaxIters];  // kModeMin: per-iteration minima of the current unit
  const int tid = threadIdx.x, nthreads = blockDim.x;
  const int n = b.n, C = b.C, F = b.F, w = b.w;
  const int ndyn = w - R;
  const uint64_t units = (uint64_t)b.batch << F;
  const int niter = (int)walk_iterations<R>(w);  // <= kBatchMaxIters (plan_batched)
  const int lane = tid & 31, warp = tid >> 5;
  uint32_t* s_words = reinterpret_cast<uint32_t*>(s_rows4);
  int staged = -1;
  WalkCtx c{};
  c.n = n;
  c.C = C;
  c.F = F;
  c.w = w;
  c.nthreads = nthreads;
  c.thread = tid;
  c.sL = sL;
  c.rows4 = s_rows4;
  c.rows1 = nullptr;
  c.t_global = true;
  // kModeTiesInt: the scan slots (packed::scan_slot_words<R>() words per thread) follow the rows
  c.scratch = MODE == kModeTiesInt ? s_words + ((size_t)ndyn << (C - 1)) : nullptr;
  // a contiguous range of units per block, so that a block stages each instance's rows once
  const uint64_t u_begin = units * blockIdx.x / gridDim.x, u_end = units * (blockIdx.x + 1) / gridDim.x;
  for (uint64_t u = u_begin, next; u < u_end; u = next) {
    const int g = (int)(u >> F);
    const uint64_t P = u & (((uint64_t)1 << F) - 1);
    next = u + 1;
    if (b.status[g] != QUBO_OK || batch_class(b.S[g]) != kBatchPacked) {  // not this pass's: skip it whole
      next = (uint64_t)(g + 1) << F;
      continue;
    }
    if (MODE == kModeTiesInt && b.unit_min[u] != b.gmin[g]) continue;
    __syncthreads();
    const packed::HalfRows rows{sH};
    if (g != staged) {
      // the instance's half sums, then its shared rows (positions >= R) formed from them
      const int nh = (n - C) * packed::HalfRows::kStride;
      const int4* H4 = reinterpret_cast<const int4*>(b.H + (size_t)g * b.sh);
      for (int idx = tid; idx < (nh >> 2); idx += nthreads) reinterpret_cast<int4*>(sH)[idx] = H4[idx];
      __syncthreads();
      if constexpr (MODE == kModeMin) {  // the re-walk forms the few rows it flips itself
        const int lq = C - 2;  // log2 of the int4 quads per row (two words each)
        for (int idx = tid; idx < (ndyn << lq); idx += nthreads) {
          const int rr = idx >> lq, q = idx & ((1 << lq) - 1);
          const int4 m = rows.quad(n - C - 1 - (R + rr), q);
          reinterpret_cast<uint2*>(s_words)[idx] = make_uint2(packed::combine(m.x, m.y), packed::combine(m.z, m.w));
        }
      }
      staged = g;
    }
    bunit_terms(b.U + (size_t)g * b.su, n, F, P, sL);
    if (MODE == kModeMin && tid < niter) s_seg[tid] = kIntInf;
    __syncthreads();
    int cP = 0;
    for (int f = 0; f < F; ++f) cP += sL[f];
    c.T = reinterpret_cast<const int*>(b.T2 + (size_t)g * b.st);
    packed::PackedWalker<R, MODE, packed::HalfRows> W;
    // one minimum per iteration of the minimum pass (kPackedR register rows) of the unit
    int32_t* seg_min = b.seg_min + (size_t)u * walk_iterations<kPackedR>(w);
    if constexpr (MODE == kModeMin) {
      W.init(c, b.Ec + (size_t)g * b.se, rows, cP);
      int best = W.walk(c, 0, niter, 0, s_seg);
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) best = min(best, __shfl_xor_sync(0xffffffffu, best, off));
      if (lane == 0) s_red[warp] = best;
      __syncthreads();
      if (tid == 0) {
        int m = s_red[0];
        for (int k = 1; k < (nthreads >> 5); ++k) m = min(m, s_red[k]);
        b.unit_min[u] = m;
      }
      if (tid < niter) seg_min[tid] = s_seg[tid];
    } else {
      // only the iterations whose minimum is the instance minimum
      const int gm = b.gmin[g];
      const uint64_t prank = (F > 0) ? (P << (n - F)) : 0;
      constexpr int f = 1 << (kPackedR - R);  // re-walk iterations per minimum-pass iteration
      const int nseg = niter / f;
      for (int it = 0; it < nseg; ++it) {
        if (seg_min[it] != gm) continue;
        W.init(c, b.Ec + (size_t)g * b.se, rows, cP);
        W.seek(c, it * f);
        W.aux = ((uint32_t)((int)packed::kHalfBias + gm - W.s) & 0xffffu) * 0x10001u;
        W.walk(c, it * f, (it + 1) * f, prank);
      }
      uint64_t cnt = W.cnt, rmin = W.rmin;
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) {
        cnt += __shfl_xor_sync(0xffffffffu, cnt, off);
        const uint64_t r2 = __shfl_xor_sync(0xffffffffu, rmin, off);
        rmin = r2 < rmin ? r2 : rmin;
      }
      if (lane == 0 && cnt) {
        atomicAdd(&b.gties[g], (unsigned long long)cnt);
        atomicMin(&b.grank[g], (unsigned long long)rmin);
      }
    }
  }
}

// Block bounds of the batched packed pass, per instance (one block of 128 threads each): the
// control table of its blocks of 2^R steps (as the single-problem block_table_kernel), and its
// starting best: sum |U|, lowered to the least walked energy (energies of states of unit 0) and
// to the least energy of four greedy descents (warp_descent; one per warp).
template <int R>
__global__ void __launch_bounds__(128) bseed_kernel(BatchTables b) {
  __shared__ int32_t sU[kBatchTabMaxN * kBatchTabMaxN];
  __shared__ int s_min;
  const int g = blockIdx.x, tid = threadIdx.x;
  if (b.status[g] != QUBO_OK || batch_class(b.S[g]) != kBatchPacked) return;
  const int n = b.n, C = b.C, w = b.w;
  const uint32_t nb = 1u << (w - R);
  const int32_t* T = b.T + (size_t)g * b.st;
  BlockCtl* blk = b.blk + (size_t)g * (nb + 1);
  const int32_t* U = b.U + (size_t)g * b.su;
  if (tid == 0) s_min = (int)b.S[g];  // no energy exceeds sum |U| (< 2^14 here)
  for (int idx = tid; idx < n * n; idx += blockDim.x) {
    const int i = idx / n, j = idx - i * n;
    sU[idx] = (j >= i) ? U[idx] : U[j * n + i];
  }
  __syncthreads();
  for (uint32_t m = tid; m <= nb; m += blockDim.x) {
    const uint32_t mm = m < nb ? m : nb - 1;
    const int4* T4 = reinterpret_cast<const int4*>(T + ((size_t)mm << R));
    int tmin = kIntInf;
    for (int q = 0; q < (1 << R) / 4; ++q) {
      const int4 t = T4[q];
      tmin = min(tmin, __vimin3_s32(t.x, t.y, min(t.z, t.w)));
    }
    if (m < nb) atomicMin(&s_min, tmin);
    BlockCtl bc;
    bc.tmin = tmin;
    if (m + 1 < nb) {
      const int rr = __ffs((int)(m + 1)) - 1;
      const bool up = !(((m + 1) >> (rr + 1)) & 1u);
      bc.row = rr << (C - 2);
      bc.dsgn = up ? 1.f : -1.f;
      bc.lvx = (up ? 0 : 64) + (n - C - 1 - (R + rr));
    } else {
      bc.row = 0;
      bc.dsgn = 0.f;
      bc.lvx = 128;
    }
    blk[m] = bc;
  }
  const int32_t e = warp_descent(sU, n, 0, 0, 1, (uint64_t)g * 4 + (tid >> 5));
  if ((tid & 31) == 0) atomicMin(&s_min, e);
  __syncthreads();
  if (tid == 0) b.gthr[g] = s_min;
}

// The packed minimum pass with block bounds (PackedPrunedWalker) over the units of the instances
// with sum |U| <= kPackedMaxAbsSum: the unit loop and staging of bpacked_kernel, each unit's
// minimum published to its instance's best, and the minima of the exactly walked blocks recorded
// for the re-walk (a block no warp walked exactly holds no state at the instance minimum).
template <int R>
__global__ void __launch_bounds__(128, 2) bpacked_pruned_kernel(BatchTables b) {
  static_assert(R == kPackedR + 1, "a block is one iteration of the packed minimum pass");
  extern __shared__ __align__(16) int4 s_rows4[];
  __shared__ int sL[129];  // L, -L at 64 + v and a zero at 128
  __shared__ int s_red[32];
  __shared__ __align__(16) int sH[(kBatchTabMaxN - kBatchTabC) * packed::HalfRows::kStride];
  __shared__ int s_seg[kBatchMaxIters];  // per-block minima of the current unit
  __shared__ uint4 s_dw[4 * 128];        // per-column changes (block bound)
  const int tid = threadIdx.x, nthreads = blockDim.x;
  const int n = b.n, C = b.C, F = b.F, w = b.w;
  const int ndyn = w - R;
  const int nblocks = 1 << (w - R);  // = the packed pass's iterations per unit
  const uint64_t units = (uint64_t)b.batch << F;
  const int lane = tid & 31, warp = tid >> 5;
  uint32_t* s_words = reinterpret_cast<uint32_t*>(s_rows4);
  int staged = -1;
  WalkCtx c{};
  c.n = n;
  c.C = C;
  c.F = F;
  c.w = w;
  c.nthreads = nthreads;
  c.thread = tid;
  c.sL = sL;
  c.rows4 = s_rows4;
  c.rows1 = nullptr;
  c.t_global = true;
  const uint64_t u_begin = units * blockIdx.x / gridDim.x, u_end = units * (blockIdx.x + 1) / gridDim.x;
  for (uint64_t u = u_begin, next; u < u_end; u = next) {
    const int g = (int)(u >> F);
    const uint64_t P = u & (((uint64_t)1 << F) - 1);
    next = u + 1;
    if (b.status[g] != QUBO_OK || batch_class(b.S[g]) != kBatchPacked) {  // not this pass's: skip it whole
      next = (uint64_t)(g + 1) << F;
      continue;
    }
    __syncthreads();
    const packed::HalfRows rows{sH};
    if (g != staged) {
      const int nh = (n - C) * packed::HalfRows::kStride;
      const int4* H4 = reinterpret_cast<const int4*>(b.H + (size_t)g * b.sh);
      for (int idx = tid; idx < (nh >> 2); idx += nthreads) reinterpret_cast<int4*>(sH)[idx] = H4[idx];
      __syncthreads();
      const int lq = C - 2;  // log2 of the int4 quads per row (two words each)
      for (int idx = tid; idx < (ndyn << lq); idx += nthreads) {
        const int rr = idx >> lq, q = idx & ((1 << lq) - 1);
        const int4 m = rows.quad(n - C - 1 - (R + rr), q);
        reinterpret_cast<uint2*>(s_words)[idx] = make_uint2(packed::combine(m.x, m.y), packed::combine(m.z, m.w));
      }
      staged = g;
    }
    bunit_terms(b.U + (size_t)g * b.su, n, F, P, sL);
    if (tid < nblocks) s_seg[tid] = kIntInf;
    __syncthreads();
    for (int v = tid; v <= 64; v += nthreads) sL[64 + v] = v < n ? -sL[v] : 0;
    __syncthreads();
    int cP = 0;
    for (int f = 0; f < F; ++f) cP += sL[f];
    const uint32_t* T2 = b.T2 + (size_t)g * b.st;
    c.T = reinterpret_cast<const int*>(T2);
    packed::PackedPrunedWalker<R, packed::HalfRows> W;
    W.init(c, b.Ec + (size_t)g * b.se, rows, cP);
    int best = W.walk(c, nblocks, b.blk + (size_t)g * (nblocks + 1), T2, b.gthr + g, 0, b.one, s_seg, s_dw);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) best = min(best, __shfl_xor_sync(0xffffffffu, best, off));
    if (lane == 0) s_red[warp] = best;
    __syncthreads();
    if (tid == 0) {
      int m = s_red[0];
      for (int k = 1; k < (nthreads >> 5); ++k) m = min(m, s_red[k]);
      b.unit_min[u] = m;
      atomicMin(b.gthr + g, m);
    }
    int32_t* seg_min = b.seg_min + (size_t)u * walk_iterations<kPackedR>(w);
    if (tid < nblocks) seg_min[tid] = s_seg[tid];
  }
}

// Instance minima over their units.
__global__ void bgroup_kernel(BatchTables b) {
  const int g = blockIdx.x * blockDim.x + threadIdx.x;
  if (g >= b.batch || b.status[g] != QUBO_OK) return;
  int m = kIntInf;
  for (uint64_t k = 0; k < ((uint64_t)1 << b.F); ++k) m = min(m, b.unit_min[((uint64_t)g << b.F) + k]);
  b.gmin[g] = m;
}

__global__ void bfinal_kernel(BatchTables b, qubo_result* out) {
  const int g = blockIdx.x * blockDim.x + threadIdx.x;
  if (g >= b.batch) return;
  qubo_result r;
  r.status = b.status[g];
  r.reserved = 0;
  r.min_energy = r.status == QUBO_OK ? (double)b.gmin[g] : 0.0;
  r.argmin_rank = r.status == QUBO_OK ? b.grank[g] : 0;
  r.tie_count = r.status == QUBO_OK ? b.gties[g] : 0;
  out[g] = r;
}

size_t al256(size_t x) { return (x + 255) & ~(size_t)255; }

// Workspace of the table-based pipeline; base may be null (sizes only).
BatchTables batch_tables(const BatchPlan& bp, unsigned char* base, size_t* bytes) {
  BatchTables t;
  std::memset(&t, 0, sizeof(t));
  t.batch = bp.batch;
  t.n = bp.n;
  t.C = bp.C;
  t.F = bp.F;
  t.w = bp.w;
  t.su = (size_t)bp.n * bp.n;
  t.sm = (size_t)(bp.n - bp.C) << bp.C;
  t.sh = (size_t)(bp.n - bp.C) * packed::HalfRows::kStride;
  t.se = (size_t)1 << bp.C;
  t.st = (size_t)1 << bp.w;
  size_t off = 0;
  auto take = [&](size_t nbytes) {
    unsigned char* p = base ? base + off : nullptr;
    off += al256(nbytes);
    return p;
  };
  const size_t B = (size_t)bp.batch;
  t.U = reinterpret_cast<int32_t*>(take(B * t.su * 4));
  t.M = reinterpret_cast<int32_t*>(take(B * t.sm * 4));
  t.H = reinterpret_cast<int32_t*>(take(B * t.sh * 4));
  t.Ec = reinterpret_cast<int32_t*>(take(B * t.se * 4));
  t.T = reinterpret_cast<int32_t*>(take(B * t.st * 4));
  t.T2 = reinterpret_cast<uint32_t*>(take(B * t.st * 4));
  t.S = reinterpret_cast<int64_t*>(take(B * 8));
  t.status = reinterpret_cast<int32_t*>(take(B * 4));
  t.unit_min = reinterpret_cast<int32_t*>(take((B << bp.F) * 4));
  t.seg_min = reinterpret_cast<int32_t*>(take((B << bp.F) * walk_iterations<kPackedR>(bp.w) * 4));
  t.gmin = reinterpret_cast<int32_t*>(take(B * 4));
  t.grank = reinterpret_cast<unsigned long long*>(take(B * 8));
  t.gties = reinterpret_cast<unsigned long long*>(take(B * 8));
  const size_t nblk = bp.w > kBatchPruneR ? ((size_t)1 << (bp.w - kBatchPruneR)) + 1 : 1;
  t.blk = reinterpret_cast<BlockCtl*>(take(B * nblk * sizeof(BlockCtl)));
  t.gthr = reinterpret_cast<int32_t*>(take(B * 4));
  t.one = 1;
  if (bytes) *bytes = off;
  return t;
}

template <typename K>
cudaError_t set_smem(K k, size_t smem) {
  return cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
}

}  // namespace

bool plan_batched(int batch, int n, BatchPlan* bp) {
  if (batch < 1 || n < 14) return false;
  const DevInfo& di = device_info();
  if (n >= 18 && n <= kBatchTabMaxN) {
    BatchPlan p;
    p.batch = batch;
    p.n = n;
    p.C = kBatchTabC;
    // units of 2^(n - F) states with at most 11 walked bits (on 4096 x n=24: 10 bits 2.63 ms,
    // 11 bits 2.59 ms per call; earlier, with slower tables, 9 bits 2.81, 10 bits 2.69, 11 bits
    // 2.74, 12 bits 3.22 ms; fewer bits cost more unit set-ups, more leave fewer units to
    // balance over the blocks)
    p.F = n - p.C - kBatchMaxWalked > 0 ? n - p.C - kBatchMaxWalked : 0;
    p.w = n - p.C - p.F;
    p.threads = (1 << p.C) / kFastCPT;
    p.tabled = true;
    p.smem_int = (size_t)(p.w - kFastR) << (p.C + 2);
    p.smem_biased = (size_t)(p.w - kBiasedR) << (p.C + 2);
    p.smem_packed = (size_t)(p.w - kPackedR) << (p.C + 1);
    if (p.w < kPackedR + 1 || p.smem_int + 4096 > di.smem_optin) return false;
    int occ = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, bwalk_kernel<kFastR, int, kModeMin>, p.threads,
                                                      p.smem_int) != cudaSuccess || occ < 1)
      occ = 1;
    p.blocks = std::max(1, di.sms) * occ;
    if (set_smem(bpacked_kernel<kPackedR, kModeMin>, p.smem_packed) != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, bpacked_kernel<kPackedR, kModeMin>, (1 << p.C) / 32,
                                                      p.smem_packed) != cudaSuccess ||
        occ < 1)
      occ = 1;
    p.packed_blocks = std::max(1, di.sms) * occ;
    // the packed pass with block bounds: at least two blocks of 2^kBatchPruneR steps per unit
    p.pruned = block_bounds_enabled() && p.w >= kBatchPruneR + 1;
    if (p.pruned) {
      p.smem_pruned = (size_t)(p.w - kBatchPruneR) << (p.C + 1);
      auto kp = bpacked_pruned_kernel<kBatchPruneR>;
      if (set_smem(kp, p.smem_pruned) != cudaSuccess ||
          cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kp, (1 << p.C) / 32, p.smem_pruned) != cudaSuccess ||
          occ < 1)
        occ = 1;
      p.pruned_blocks = std::max(1, di.sms) * occ;
    }
    *bp = p;
    return true;
  }
  if (n > kBatchMaxN) return false;
  // cache bits: 2^C columns = threads * 16; walked w = n - C needs w >= R + 1 + log2(segments)
  int C = n >= 24 ? 11 : n - (kFastR + 1 + 5);
  if (C > 12) C = 12;
  if (C < 9) C = 9;
  const int w = n - C;
  if (w < kFastR + 1 + 5) return false;  // at least one iteration per segment
  bp->batch = batch;
  bp->n = n;
  bp->C = C;
  bp->w = w;
  bp->threads = (1 << C) / kFastCPT;
  bp->smem_bytes = ((size_t)(w - kFastR) << (C + 2)) + ((size_t)1 << (w + 2)) + (size_t)n * n * 4;
  bp->tabled = false;
  if (bp->smem_bytes + 4096 > di.smem_optin) return false;
  return true;
}

size_t batched_workspace_bytes(const BatchPlan& bp) {
  if (!bp.tabled) return 256;
  size_t bytes = 0;
  batch_tables(bp, nullptr, &bytes);
  return bytes;
}

cudaError_t run_batched(const BatchPlan& bp, const void* d_Q, void* d_ws, qubo_result* res, cudaStream_t stream,
                        int* launches) {
  cudaError_t e;
  if (!bp.tabled) {
    (void)d_ws;
    if ((e = set_smem(batched_kernel, bp.smem_bytes)) != cudaSuccess) return e;
    batched_kernel<<<bp.batch, bp.threads, bp.smem_bytes, stream>>>(bp.n, bp.C, static_cast<const int32_t*>(d_Q),
                                                                       res);
    if (launches) *launches = 1;
    return cudaGetLastError();
  }
  BatchTables t = batch_tables(bp, static_cast<unsigned char*>(d_ws), nullptr);
  t.Q = static_cast<const int32_t*>(d_Q);
  int nl = 0;
  btables_kernel<<<bp.batch, 256, 0, stream>>>(t);
  ++nl;
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  if (bp.pruned) {
    // packed instances: block tables and starting bests, then the bounded packed pass
    bseed_kernel<kBatchPruneR><<<bp.batch, 128, 0, stream>>>(t);
    ++nl;
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    auto kp = bpacked_pruned_kernel<kBatchPruneR>;
    if ((e = set_smem(kp, bp.smem_pruned)) != cudaSuccess) return e;
    kp<<<bp.pruned_blocks, (1 << bp.C) / 32, bp.smem_pruned, stream>>>(t);
  } else {
    if ((e = set_smem(bpacked_kernel<kPackedR, kModeMin>, bp.smem_packed)) != cudaSuccess) return e;
    bpacked_kernel<kPackedR, kModeMin><<<bp.packed_blocks, (1 << bp.C) / 32, bp.smem_packed, stream>>>(t);
  }
  ++nl;
  auto kb = bwalk_kernel<kBiasedR, float, kModeMin>;
  if ((e = set_smem(kb, bp.smem_biased)) != cudaSuccess) return e;
  kb<<<bp.blocks, bp.threads, bp.smem_biased, stream>>>(t);
  ++nl;
  auto ki = bwalk_kernel<kIntMinR, int, kModeMin>;
  if ((e = set_smem(ki, bp.smem_int)) != cudaSuccess) return e;
  ki<<<bp.blocks, bp.threads, bp.smem_int, stream>>>(t);
  ++nl;
  bgroup_kernel<<<(bp.batch + 127) / 128, 128, 0, stream>>>(t);
  ++nl;
  const size_t smem_ties = ((size_t)(bp.w - kPackedTiesR) << (bp.C + 1)) +
                           (size_t)((1 << bp.C) / 32) * packed::scan_slot_words<kPackedTiesR>() * 4;
  if ((e = set_smem(bpacked_kernel<kPackedTiesR, kModeTiesInt>, smem_ties)) != cudaSuccess) return e;
  bpacked_kernel<kPackedTiesR, kModeTiesInt><<<bp.packed_blocks, (1 << bp.C) / 32, smem_ties, stream>>>(t);
  ++nl;
  auto kr = bwalk_kernel<kFastR, int, kModeTiesInt>;
  if ((e = set_smem(kr, bp.smem_int)) != cudaSuccess) return e;
  kr<<<bp.blocks, bp.threads, bp.smem_int, stream>>>(t);
  ++nl;
  bfinal_kernel<<<(bp.batch + 127) / 128, 128, 0, stream>>>(t, res);
  ++nl;
  if (launches) *launches = nl;
  return cudaGetLastError();
}

}  // namespace qgb
