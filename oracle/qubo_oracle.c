/*
 * qubo_oracle.c -- CPU oracle for exhaustive QUBO minimisation.
 *
 * TEST INFRASTRUCTURE ONLY. Only tests/, __graft_entry__.smoke() and bench.py's cpu_baseline /
 * reference leg may load this code. It shares nothing with the CUDA path: no headers, no
 * tables, no helpers. It is deliberately plain and slow.
 *
 * What it computes (Terastate-per-second QUBO Brute-Force on a Single GPU, §I, objective
 * E(x) = sum_{i,j} Q_ij x_i x_j over x in {0,1}^n, to be minimised):
 *   E_min  = min_x E(x)
 *   argmin = the minimiser with the lowest rank, rank(x) = sum_i x_i 2^(n-1-i)
 *            (x_0 is the most significant bit: the lexicographic state order of §II-B, Fig. 2)
 *   ties   = number of states x with E(x) = E_min
 *
 * Readings of the pages taken here (each is also listed with the design notes):
 *   - Q need not be triangular: E sums over all i, j. Folding gives the equivalent upper
 *     triangle U_ii = Q_ii, U_ij = Q_ij + Q_ji (i < j), which is what §II-A assumes.
 *   - Ties are broken by lowest rank (the pages keep the first minimum found in their own
 *     traversal order, which depends on the decomposition).
 *   - For fp32 input the energy of a state is the fixed-order fp64 sum eval64(): i ascending,
 *     j >= i ascending, additions only, compiled without FMA contraction.
 *
 * Two independent evaluators:
 *   oracle_direct_*  -- evaluates every state from scratch, O(n^2) per state (§I-D, naive).
 *   oracle_gray_*    -- Gray-code walk with local fields, O(n) per state (§I-D, ref. [2]):
 *                       flipping x_k changes E by d*(U_kk + h_k), h_v = sum_{u != v} U_uv x_u,
 *                       then every other field moves by d*U_kv.
 * Both take a fixed prefix (the first k variables), which is the subproblem split of §III-C1.
 *   oracle_lowest_i64 -- the k smallest keys (E, rank), every state evaluated from scratch.
 *   oracle_ising_direct_* -- the Ising energy H(s) of §I from its definition, per spin state
 *                       (no conversion to the QUBO form), for the Ising entry points.
 *
 * Parity pins for every function live in tests/test_oracle.py.
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <math.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_API __attribute__((visibility("default")))

/* Mistake planting for the pin-sensitivity tests: each value breaks one step on purpose.
 * 0 = correct oracle (the only build anything but tests/test_oracle_mutants.py loads). */
#ifndef ORACLE_MUTANT
#define ORACLE_MUTANT 0
#endif

/* ---------------------------------------------------------------- helpers */

ORACLE_API uint64_t oracle_gray_code(uint64_t i) { return i ^ (i >> 1); }

/* Bit position that changes between Gray codes i and i+1 (the lowest set bit of i+1). */
ORACLE_API int oracle_gray_flip_bit(uint64_t i) {
  uint64_t v = i + 1;
  int b = 0;
  while (!(v & 1)) { v >>= 1; ++b; }
  return b;
}

static int thread_count(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

ORACLE_API int oracle_num_threads(void) { return thread_count(); }

/* Threads of the following parallel regions (timing of the oracle on one core or on all). */
ORACLE_API void oracle_set_threads(int t) {
#ifdef _OPENMP
  if (t > 0) omp_set_num_threads(t);
#else
  (void)t;
#endif
}

/* ---------------------------------------------------------------- folding */

/* U (n x n, row-major) from int32 Q: U_ii = Q_ii, U_ij = Q_ij + Q_ji for i < j, 0 below. */
ORACLE_API void oracle_fold_i32(int n, const int32_t* Q, int64_t* U) {
  for (int i = 0; i < n; ++i)
    for (int j = 0; j < n; ++j) {
      int64_t v = 0;
      if (j == i) v = Q[i * n + i];
      else if (j > i) v = (int64_t)Q[i * n + j] + (int64_t)Q[j * n + i];
      U[i * n + j] = v;
    }
}

/* Same for fp32 Q, folded in fp64. */
ORACLE_API void oracle_fold_f32(int n, const float* Q, double* U) {
  for (int i = 0; i < n; ++i)
    for (int j = 0; j < n; ++j) {
      double v = 0.0;
      if (j == i) v = (double)Q[i * n + i];
      else if (j > i) v = (double)Q[i * n + j] + (double)Q[j * n + i];
      U[i * n + j] = v;
    }
}

/* The same fold for fp64 input (one fp64 add per off-diagonal pair). */
ORACLE_API void oracle_fold_f64(int n, const double* Q, double* U) {
  for (int i = 0; i < n; ++i)
    for (int j = 0; j < n; ++j) {
      double v = 0.0;
      if (j == i) v = Q[i * n + i];
      else if (j > i) v = Q[i * n + j] + Q[j * n + i];
      U[i * n + j] = v;
    }
}

/* ---------------------------------------------------------------- energies */

static void bits_of_rank(int n, uint64_t rank, uint8_t* x) {
  for (int i = 0; i < n; ++i) x[i] = (uint8_t)((rank >> (n - 1 - i)) & 1u);
}

/* E(x) = sum_{i <= j} U_ij x_i x_j over the folded triangle, exact in int64. */
ORACLE_API int64_t oracle_energy_i64(int n, const int64_t* U, const uint8_t* x) {
  int64_t e = 0;
  for (int i = 0; i < n; ++i) {
    if (!x[i]) continue;
    for (int j = i; j < n; ++j) {
#if ORACLE_MUTANT == 1
      if (j == i) continue; /* planted: diagonal dropped */
#endif
      if (x[j]) e += U[i * n + j];
    }
  }
  return e;
}

/* Fixed-order fp64 evaluation: i ascending, j >= i ascending, one addition per selected term. */
ORACLE_API double oracle_eval64(int n, const double* U, const uint8_t* x) {
  double e = 0.0;
  for (int i = 0; i < n; ++i) {
    if (!x[i]) continue;
    for (int j = i; j < n; ++j)
      if (x[j]) e = e + U[i * n + j];
  }
  return e;
}

/* E from the raw (unfolded) int32 Q, sum over all i, j: the objective exactly as written. */
ORACLE_API int64_t oracle_energy_raw_i32(int n, const int32_t* Q, const uint8_t* x) {
  int64_t e = 0;
  for (int i = 0; i < n; ++i)
    for (int j = 0; j < n; ++j)
      if (x[i] && x[j]) e += Q[i * n + j];
  return e;
}

/* ---------------------------------------------------------------- result merging */

typedef struct {
  int64_t e;
  uint64_t rank;
  uint64_t ties;
  int have;
} res_i64;

static void merge_i64(res_i64* a, const res_i64* b) {
  if (!b->have) return;
  if (!a->have || b->e < a->e) { *a = *b; return; }
  if (b->e == a->e) {
    a->ties += b->ties;
    if (b->rank < a->rank) a->rank = b->rank;
  }
}

static void see_i64(res_i64* r, int64_t e, uint64_t rank) {
  if (!r->have || e < r->e) { r->e = e; r->rank = rank; r->ties = 1; r->have = 1; }
  else if (e == r->e) { r->ties += 1; if (rank < r->rank) r->rank = rank; }
}

/* ---------------------------------------------------------------- direct search */

/* Every state with rank in [lo, hi), evaluated from scratch (O(n^2) each). */
ORACLE_API void oracle_direct_i64(int n, const int64_t* U, uint64_t lo, uint64_t hi, int64_t* emin,
                                  uint64_t* argmin, uint64_t* ties) {
  res_i64 total = {0, 0, 0, 0};
  int nt = thread_count();
  res_i64* part = (res_i64*)calloc((size_t)nt, sizeof(res_i64));
#pragma omp parallel
  {
    int t = 0;
#ifdef _OPENMP
    t = omp_get_thread_num();
#endif
    uint8_t x[64];
    res_i64 r = {0, 0, 0, 0};
#pragma omp for schedule(static)
    for (int64_t s = (int64_t)lo; s < (int64_t)hi; ++s) {
      bits_of_rank(n, (uint64_t)s, x);
      see_i64(&r, oracle_energy_i64(n, U, x), (uint64_t)s);
    }
    part[t] = r;
  }
  for (int t = 0; t < nt; ++t) merge_i64(&total, &part[t]);
  free(part);
  *emin = total.e;
  *argmin = total.rank;
  *ties = total.ties;
}

/* ---------------------------------------------------------------- Gray-code walker (int64) */

/* Walk all 2^m states whose first n-m variables form `rank0`'s prefix; rank0 has the walked
 * variables at zero. Gray bit b drives variable n-1-b, so rank changes by 2^b per flip. */
static void walk_block_i64(int n, const int64_t* U, uint64_t rank0, int m, res_i64* r) {
  uint8_t x[64];
  int64_t h[64];
  bits_of_rank(n, rank0, x);
  int64_t e = oracle_energy_i64(n, U, x);
  for (int v = 0; v < n; ++v) {
    int64_t s = 0;
    for (int u = 0; u < n; ++u) {
      if (u == v || !x[u]) continue;
      s += (u < v) ? U[u * n + v] : U[v * n + u];
    }
    h[v] = s;
  }
  uint64_t rank = rank0;
  see_i64(r, e, rank);
  uint64_t steps = (m >= 64) ? 0 : ((uint64_t)1 << m);
  for (uint64_t i = 0; i + 1 < steps; ++i) {
    int b = oracle_gray_flip_bit(i);
    int k = n - 1 - b;
    int64_t d = x[k] ? -1 : 1;
#if ORACLE_MUTANT == 2
    d = 1; /* planted: flip direction ignored */
#endif
    e += d * (U[k * n + k] + h[k]);
    x[k] ^= 1;
    rank ^= (uint64_t)1 << b;
    for (int v = 0; v < n; ++v) {
      if (v == k) continue;
#if ORACLE_MUTANT == 3
      h[v] += d * U[v * n + k]; /* planted: lower triangle (zeros) read instead of upper */
#else
      h[v] += d * ((k < v) ? U[k * n + v] : U[v * n + k]);
#endif
    }
    see_i64(r, e, rank);
  }
}

/* Minimum over the slice of states whose first k variables equal `prefix` (prefix bit k-1-f is
 * variable f). k = 0 searches everything. OpenMP splits the slice into blocks of at most 2^12
 * states, each re-initialised from scratch. */
ORACLE_API void oracle_gray_i64(int n, const int64_t* U, int k, uint64_t prefix, int64_t* emin,
                                uint64_t* argmin, uint64_t* ties) {
  int m = n - k;
  int mb = m < 12 ? m : 12;
  int sb = m - mb;
  uint64_t nblocks = (uint64_t)1 << sb;
  int nt = thread_count();
  res_i64* part = (res_i64*)calloc((size_t)nt, sizeof(res_i64));
#pragma omp parallel
  {
    int t = 0;
#ifdef _OPENMP
    t = omp_get_thread_num();
#endif
    res_i64 r = {0, 0, 0, 0};
#pragma omp for schedule(static)
    for (int64_t blk = 0; blk < (int64_t)nblocks; ++blk) {
      uint64_t rank0 = (prefix << m) | ((uint64_t)blk << mb);
      walk_block_i64(n, U, rank0, mb, &r);
    }
    part[t] = r;
  }
  res_i64 total = {0, 0, 0, 0};
  for (int t = 0; t < nt; ++t) merge_i64(&total, &part[t]);
  free(part);
  *emin = total.e;
  *argmin = total.rank;
  *ties = total.ties;
}

/* Walker energies of every state in Gray order from x = 0 (n <= 24), for pinning the walker
 * against direct evaluation and the Gray sequence against the pages' Fig. 5. */
ORACLE_API void oracle_gray_trace_i64(int n, const int64_t* U, int64_t* E, uint64_t* rank_out) {
  uint8_t x[64];
  int64_t h[64];
  memset(x, 0, sizeof(x));
  memset(h, 0, sizeof(h));
  int64_t e = 0;
  uint64_t rank = 0;
  uint64_t steps = (uint64_t)1 << n;
  E[0] = 0;
  rank_out[0] = 0;
  for (uint64_t i = 0; i + 1 < steps; ++i) {
    int b = oracle_gray_flip_bit(i);
    int k = n - 1 - b;
    int64_t d = x[k] ? -1 : 1;
    e += d * (U[k * n + k] + h[k]);
    x[k] ^= 1;
    rank ^= (uint64_t)1 << b;
    for (int v = 0; v < n; ++v)
      if (v != k) h[v] += d * ((k < v) ? U[k * n + v] : U[v * n + k]);
    E[i + 1] = e;
    rank_out[i + 1] = rank;
  }
}

/* ---------------------------------------------------------------- Gray-code walker (fp64) */

typedef struct {
  double e;
  uint64_t rank;
  uint64_t ties;
  int have;
} res_f64;

static void merge_f64(res_f64* a, const res_f64* b) {
  if (!b->have) return;
  if (!a->have || b->e < a->e) { *a = *b; return; }
  if (b->e == a->e) {
    a->ties += b->ties;
    if (b->rank < a->rank) a->rank = b->rank;
  }
}

/* fp64 walk of one block. Pass 1 (thr = NAN) records the lowest walked energy. Pass 2 re-walks
 * and, for every state whose walked energy is <= thr, evaluates eval64() and keeps the lowest
 * (then lowest-rank) value and the count of states equal to it. */
static void walk_block_f64(int n, const double* U, uint64_t rank0, int m, double thr, double* wmin,
                           res_f64* r) {
  uint8_t x[64];
  double h[64];
  bits_of_rank(n, rank0, x);
  double e = oracle_eval64(n, U, x);
  for (int v = 0; v < n; ++v) {
    double s = 0.0;
    for (int u = 0; u < n; ++u) {
      if (u == v || !x[u]) continue;
      s = s + ((u < v) ? U[u * n + v] : U[v * n + u]);
    }
    h[v] = s;
  }
  uint64_t rank = rank0;
  uint64_t steps = (uint64_t)1 << m;
  for (uint64_t i = 0;; ++i) {
    if (isnan(thr)) {
      if (e < *wmin) *wmin = e;
    } else if (e <= thr) {
      double ex = oracle_eval64(n, U, x);
      if (!r->have || ex < r->e) { r->e = ex; r->rank = rank; r->ties = 1; r->have = 1; }
      else if (ex == r->e) { r->ties += 1; if (rank < r->rank) r->rank = rank; }
    }
    if (i + 1 >= steps) break;
    int b = oracle_gray_flip_bit(i);
    int k = n - 1 - b;
    double d = x[k] ? -1.0 : 1.0;
    e = e + d * (U[k * n + k] + h[k]);
    x[k] ^= 1;
    rank ^= (uint64_t)1 << b;
    for (int v = 0; v < n; ++v)
      if (v != k) h[v] = h[v] + d * ((k < v) ? U[k * n + v] : U[v * n + k]);
  }
}

/* Rigorous bound on |walked energy - exact energy| inside one block of L = 2^mb states:
 * the initial direct sums have at most n^2 and n terms, every field update adds one rounding,
 * and every energy step adds the field error so far plus two roundings, each at most u*A with
 * A = sum |U_ij| (every partial sum is a sub-sum of U). Summing gives
 * u*A*(n^2 + L*(n+2) + L^2/2); it is doubled for safety. */
ORACLE_API double oracle_walk_bound_f64(int n, const double* U, int mb) {
  double A = 0.0;
  for (int i = 0; i < n; ++i)
    for (int j = i; j < n; ++j) A += fabs(U[i * n + j]);
  double L = (double)((uint64_t)1 << mb);
  double u = ldexp(1.0, -53);
  double nn = (double)n;
  return 2.0 * u * A * (nn * nn + L * (nn + 2.0) + 0.5 * L * L + 4.0 * nn * nn);
}

/* fp64 slice search: min of eval64 over the slice, lowest rank, ties by equal eval64.
 * Candidates are the states whose walked energy lies within 2*(bound) of the walked minimum,
 * which provably contains every eval64 minimiser. */
ORACLE_API void oracle_gray_f64(int n, const double* U, int k, uint64_t prefix, double* emin,
                                uint64_t* argmin, uint64_t* ties) {
  int m = n - k;
  int mb = m < 10 ? m : 10;
  int sb = m - mb;
  uint64_t nblocks = (uint64_t)1 << sb;
  int nt = thread_count();
  double* wpart = (double*)malloc((size_t)nt * sizeof(double));
  res_f64* part = (res_f64*)calloc((size_t)nt, sizeof(res_f64));
  for (int t = 0; t < nt; ++t) wpart[t] = INFINITY;
#pragma omp parallel
  {
    int t = 0;
#ifdef _OPENMP
    t = omp_get_thread_num();
#endif
    double w = INFINITY;
    res_f64 dummy = {0, 0, 0, 0};
#pragma omp for schedule(static)
    for (int64_t blk = 0; blk < (int64_t)nblocks; ++blk)
      walk_block_f64(n, U, (prefix << m) | ((uint64_t)blk << mb), mb, NAN, &w, &dummy);
    wpart[t] = w;
  }
  double wmin = INFINITY;
  for (int t = 0; t < nt; ++t) if (wpart[t] < wmin) wmin = wpart[t];
  double thr = wmin + 2.0 * oracle_walk_bound_f64(n, U, mb);
#pragma omp parallel
  {
    int t = 0;
#ifdef _OPENMP
    t = omp_get_thread_num();
#endif
    double w = 0;
    res_f64 r = {0, 0, 0, 0};
#pragma omp for schedule(static)
    for (int64_t blk = 0; blk < (int64_t)nblocks; ++blk)
      walk_block_f64(n, U, (prefix << m) | ((uint64_t)blk << mb), mb, thr, &w, &r);
    part[t] = r;
  }
  res_f64 total = {0, 0, 0, 0};
  for (int t = 0; t < nt; ++t) merge_f64(&total, &part[t]);
  free(part);
  free(wpart);
  *emin = total.e;
  *argmin = total.rank;
  *ties = total.ties;
}

/* fp64 direct search over ranks [lo, hi): min of eval64, lowest rank, ties by equal eval64. */
ORACLE_API void oracle_direct_f64(int n, const double* U, uint64_t lo, uint64_t hi, double* emin,
                                  uint64_t* argmin, uint64_t* ties) {
  res_f64 total = {0, 0, 0, 0};
  int nt = thread_count();
  res_f64* part = (res_f64*)calloc((size_t)nt, sizeof(res_f64));
#pragma omp parallel
  {
    int t = 0;
#ifdef _OPENMP
    t = omp_get_thread_num();
#endif
    uint8_t x[64];
    res_f64 r = {0, 0, 0, 0};
#pragma omp for schedule(static)
    for (int64_t s = (int64_t)lo; s < (int64_t)hi; ++s) {
      bits_of_rank(n, (uint64_t)s, x);
      double e = oracle_eval64(n, U, x);
      if (!r.have || e < r.e) { r.e = e; r.rank = (uint64_t)s; r.ties = 1; r.have = 1; }
      else if (e == r.e) { r.ties += 1; if ((uint64_t)s < r.rank) r.rank = (uint64_t)s; }
    }
    part[t] = r;
  }
  for (int t = 0; t < nt; ++t) merge_f64(&total, &part[t]);
  free(part);
  *emin = total.e;
  *argmin = total.rank;
  *ties = total.ties;
}

/* ---------------------------------------------------------------- subproblem split (§III-C1) */

/* For a fixed prefix x_f (first k variables): c = energy of the fixed part alone, and the
 * reduced matrix Q' = U_rr + diag(x_f U_fr) over the remaining n-k variables (upper triangle,
 * (n-k) x (n-k)), so that E(x) = c + E'(x_r). Written out for the slice-identity pin. */
ORACLE_API int64_t oracle_subproblem_i64(int n, const int64_t* U, int k, uint64_t prefix,
                                         int64_t* Qr) {
  int m = n - k;
  uint8_t xf[64];
  for (int f = 0; f < k; ++f) xf[f] = (uint8_t)((prefix >> (k - 1 - f)) & 1u);
  int64_t c = 0;
  for (int i = 0; i < k; ++i)
    for (int j = i; j < k; ++j)
      if (xf[i] && xf[j]) c += U[i * n + j];
  for (int a = 0; a < m; ++a)
    for (int b = 0; b < m; ++b) {
      int64_t v = 0;
      if (b >= a) v = U[(k + a) * n + (k + b)];
      if (a == b)
        for (int f = 0; f < k; ++f)
          if (xf[f]) v += U[f * n + (k + a)];
      Qr[a * m + b] = v;
    }
  return c;
}

/* ---------------------------------------------------------------- Ising form (§I) */

/* H(s) = sum_{i,j} J_ij s_i s_j + sum_i h_i s_i with s_i = 2 x_i - 1, evaluated from its
 * definition for every state with rank(x) in [lo, hi) (no conversion to the QUBO form): the
 * minimum, the lowest rank reaching it and the number of states reaching it. h may be NULL. */
ORACLE_API void oracle_ising_direct_i64(int n, const int64_t* J, const int64_t* h, uint64_t lo, uint64_t hi,
                                        int64_t* hmin, uint64_t* argmin, uint64_t* ties) {
  res_i64 total = {0, 0, 0, 0};
  int nt = thread_count();
  res_i64* part = (res_i64*)calloc((size_t)nt, sizeof(res_i64));
#pragma omp parallel
  {
    int t = 0;
#ifdef _OPENMP
    t = omp_get_thread_num();
#endif
    uint8_t x[64];
    res_i64 r = {0, 0, 0, 0};
#pragma omp for schedule(static)
    for (int64_t st = (int64_t)lo; st < (int64_t)hi; ++st) {
      bits_of_rank(n, (uint64_t)st, x);
      int64_t H = 0;
      for (int i = 0; i < n; ++i) {
        const int64_t si = x[i] ? 1 : -1;
        for (int j = 0; j < n; ++j) H += J[i * n + j] * si * (x[j] ? 1 : -1);
        if (h) H += h[i] * si;
      }
      see_i64(&r, H, (uint64_t)st);
    }
    part[t] = r;
  }
  for (int t = 0; t < nt; ++t) merge_i64(&total, &part[t]);
  free(part);
  *hmin = total.e;
  *argmin = total.rank;
  *ties = total.ties;
}

/* The same in fp64 (sum in the order written: i ascending, j ascending, then the field). */
ORACLE_API void oracle_ising_direct_f64(int n, const double* J, const double* h, uint64_t lo, uint64_t hi,
                                        double* hmin, uint64_t* argmin, uint64_t* ties) {
  res_f64 total = {0, 0, 0, 0};
  int nt = thread_count();
  res_f64* part = (res_f64*)calloc((size_t)nt, sizeof(res_f64));
#pragma omp parallel
  {
    int t = 0;
#ifdef _OPENMP
    t = omp_get_thread_num();
#endif
    uint8_t x[64];
    res_f64 r = {0, 0, 0, 0};
#pragma omp for schedule(static)
    for (int64_t st = (int64_t)lo; st < (int64_t)hi; ++st) {
      bits_of_rank(n, (uint64_t)st, x);
      double H = 0.0;
      for (int i = 0; i < n; ++i) {
        const double si = x[i] ? 1.0 : -1.0;
        for (int j = 0; j < n; ++j) H += J[i * n + j] * si * (x[j] ? 1.0 : -1.0);
        if (h) H += h[i] * si;
      }
      if (!r.have || H < r.e) { r.e = H; r.rank = (uint64_t)st; r.ties = 1; r.have = 1; }
      else if (H == r.e) { r.ties += 1; if ((uint64_t)st < r.rank) r.rank = (uint64_t)st; }
    }
    part[t] = r;
  }
  for (int t = 0; t < nt; ++t) merge_f64(&total, &part[t]);
  free(part);
  *hmin = total.e;
  *argmin = total.rank;
  *ties = total.ties;
}

/* ---------------------------------------------------------------- lowest part of the spectrum */

/* The k states with the smallest keys (E(x), rank(x)) among ranks [lo, hi), in ascending key
 * order, each state evaluated from scratch (O(n^2)). Writes min(k, hi - lo) entries and returns
 * that number. Each thread keeps a sorted array of its k best keys; the arrays are merged at the
 * end. */
typedef struct {
  int64_t e;
  uint64_t rank;
} key_i64;

static int key_less(key_i64 a, key_i64 b) { return a.e < b.e || (a.e == b.e && a.rank < b.rank); }

static void keep_lowest(key_i64* top, int* m, int k, key_i64 x) {
  if (*m == k && !key_less(x, top[k - 1])) return;
  int i = (*m < k) ? (*m)++ : k - 1;
  while (i > 0 && key_less(x, top[i - 1])) {
    top[i] = top[i - 1];
    --i;
  }
  top[i] = x;
}

ORACLE_API int oracle_lowest_i64(int n, const int64_t* U, int k, uint64_t lo, uint64_t hi, int64_t* out_e,
                                 uint64_t* out_rank) {
  if (k < 1) return 0;
  int nt = thread_count();
  key_i64* all = (key_i64*)calloc((size_t)nt * (size_t)k, sizeof(key_i64));
  int* cnt = (int*)calloc((size_t)nt, sizeof(int));
#pragma omp parallel
  {
    int t = 0;
#ifdef _OPENMP
    t = omp_get_thread_num();
#endif
    uint8_t x[64];
    key_i64* top = all + (size_t)t * (size_t)k;
    int m = 0;
#pragma omp for schedule(static)
    for (int64_t st = (int64_t)lo; st < (int64_t)hi; ++st) {
      bits_of_rank(n, (uint64_t)st, x);
      key_i64 v = {oracle_energy_i64(n, U, x), (uint64_t)st};
      keep_lowest(top, &m, k, v);
    }
    cnt[t] = m;
  }
  key_i64* best = (key_i64*)calloc((size_t)k, sizeof(key_i64));
  int m = 0;
  for (int t = 0; t < nt; ++t)
    for (int i = 0; i < cnt[t]; ++i) keep_lowest(best, &m, k, all[(size_t)t * (size_t)k + i]);
  for (int i = 0; i < m; ++i) {
    out_e[i] = best[i].e;
    out_rank[i] = best[i].rank;
  }
  free(best);
  free(cnt);
  free(all);
  return m;
}
