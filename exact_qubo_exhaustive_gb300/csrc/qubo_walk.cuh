// Device-side Gray-code walker of the prefix-suffix decomposition (sm_103a).
//
// Method (Terastate-per-second QUBO Brute-Force on a Single GPU):
//  * §III-C1: a work unit fixes the first F variables (prefix P); the rest is an independent
//    subproblem Q' = U_rr + diag(x_f U_fr) plus the constant c(P).
//  * §II-A..C: the free variables split into walked variables (the pages' prefix block, A bits)
//    and cached variables (the suffix block, B bits). For every cached assignment j (a column)
//    the energy is E = E_walked(g) + E_cached(j) + sum_{k in g} M_int[k][j] (eq. 8); the
//    interaction rows M_int and E_cached are the energy-component cache.
//  * §III-B, eq. 9: walked assignments are visited in Gray-code order, so one walked variable
//    flips per step and every column changes by exactly one row of M_int: one add per state.
//  * §III-C2: columns are split across threads; each thread keeps its columns' running
//    energies (and the rows of the lowest walked variables) in registers.
//  * §IV-B.3: the walked self-energy E_walked is read from a table stored in Gray order, so
//    the per-step read is sequential; all threads read the same entry (a broadcast).
//
// Per state the fast kernel issues one integer add (running energy += row) and half of a
// 3-input min (the chunk minimum over the thread's columns); per step and thread it adds one
// fused add-min (chunk minimum + walked energy, into the running best).
//
// Notation inside: a unit has n - F free variables = w walked + C cached. Gray position a
// (0 = fastest) drives walked variable n - C - 1 - a. Column j holds cached variable n - 1 - b
// in bit b. The state visited at Gray step i and column j has rank
//     (P << (n - F)) | (gray(i) << C) | j.
// Running quantities per thread:
//     V[j] = E_cached(j) + L_c(j) + sum over set walked positions a of M[v_a][j]
//            (+ L[v_a] for positions a < R, whose rows include the linear term),
//     s    = c(P) + sum over set walked positions a >= R of L[v_a],
// so the state's energy is s + T[i] + V[j], with T[i] = E_walked(gray(i)).
#pragma once

#include <cuda_runtime.h>

#include <cstdint>
#include <type_traits>

#include "qubo_internal.h"

namespace qgb {

constexpr int kIntInf = 0x7fffffff;

__device__ __forceinline__ uint64_t gray_code(uint64_t i) { return i ^ (i >> 1); }

__host__ __device__ constexpr int ctz_c(int x) { return (x & 1) ? 0 : 1 + ctz_c(x >> 1); }

// Order-preserving map from a (non-NaN) double to uint64.
__device__ __forceinline__ uint64_t order_key(double d) {
  const long long b = __double_as_longlong(d);
  return b < 0 ? ~static_cast<uint64_t>(b) : (static_cast<uint64_t>(b) | 0x8000000000000000ull);
}
__host__ __device__ inline double key_to_double(uint64_t k) {
  const uint64_t b = (k & 0x8000000000000000ull) ? (k & 0x7fffffffffffffffull) : ~k;
  double d;
  memcpy(&d, &b, sizeof(d));
  return d;
}

// Energy of the state `rank` from the fp64 folded triangle, fixed order (i ascending, j >= i
// ascending), correctly rounded additions only: the same sum the fp32 energy is defined by.
static __device__ __noinline__ double eval64_rank(const double* __restrict__ U64, int n, uint64_t rank) {
  double e = 0.0;
  for (int i = 0; i < n; ++i) {
    if (!((rank >> (n - 1 - i)) & 1u)) continue;
    for (int j = i; j < n; ++j)
      if ((rank >> (n - 1 - j)) & 1u) e = __dadd_rn(e, U64[i * n + j]);
  }
  return e;
}

// Minimum of N register values with 3-input mins (one ALU instruction per two values).
template <int N>
__device__ __forceinline__ int min_all(const int* v) {
  if constexpr (N == 1) {
    return v[0];
  } else if constexpr (N == 2) {
    return min(v[0], v[1]);
  } else {
    constexpr int G = (N + 2) / 3;
    int w[G];
#pragma unroll
    for (int g = 0; g < G; ++g) {
      if (3 * g + 2 < N) w[g] = __vimin3_s32(v[3 * g], v[3 * g + 1], v[3 * g + 2]);
      else if (3 * g + 1 < N) w[g] = min(v[3 * g], v[3 * g + 1]);
      else w[g] = v[3 * g];
    }
    return min_all<G>(w);
  }
}

// Representation of the running column energies V and walked rows in the walk.
//
// int: plain int32; every add and min runs on the integer ALU pipe (or the FMA pipe's
// integer multiply-add, at the compiler's choice).
//
// float (biased binade): V[j] is held as the fp32 number kBias + V[j], kBias = 1.5 * 2^23. While
// |V[j]| < 2^22 the number lies in [2^23, 2^24), where fp32 numbers are exactly the integers and
// the bit pattern of x is x + (0x4B000000 - 2^23): an affine, increasing image of the value.
// So the column update V += row is an exact FADD on the two FMA pipes, and the minimum over
// columns, the fused add-min with the walked energy and the running best are integer
// instructions on the bit patterns, exactly as in the int representation shifted by kBiasBits.
template <typename VT>
struct VOps;
template <>
struct VOps<int> {
  static constexpr bool kInt = true;
  static constexpr int kBiasBits = 0;
  using V4 = int4;
  static __device__ __forceinline__ int add(int a, int b) { return a + b; }
  static __device__ __forceinline__ int sub(int a, int b) { return a - b; }
  static __device__ __forceinline__ int energy(int x) { return x; }  // V representation of energy x
  static __device__ __forceinline__ int row(int x) { return x; }     // row representation of x
  static __device__ __forceinline__ int bits(int v) { return v; }    // order-preserving int image
};
template <>
struct VOps<float> {
  static constexpr bool kInt = false;
  static constexpr int kBiasBits = 0x4B400000;  // bit pattern of 1.5 * 2^23
  using V4 = float4;
  static __device__ __forceinline__ float add(float a, float b) { return __fadd_rn(a, b); }
  static __device__ __forceinline__ float sub(float a, float b) { return __fsub_rn(a, b); }
  static __device__ __forceinline__ float energy(int x) { return __int_as_float(kBiasBits + x); }
  static __device__ __forceinline__ float row(int x) { return static_cast<float>(x); }
  static __device__ __forceinline__ int bits(float v) { return __float_as_int(v); }
};

// Minimum of the order images of N register values, with 3-input mins (one ALU instruction
// per two values).
template <typename VT, int N>
__device__ __forceinline__ int vmin_bits(const VT* v) {
  int b[N];
#pragma unroll
  for (int k = 0; k < N; ++k) b[k] = VOps<VT>::bits(v[k]);
  return min_all<N>(b);
}

// Modes of one walk.
enum WalkMode : int {
  kModeMin = 0,     // minimum energy of the walked states
  kModeTiesInt = 1, // count states with energy <= threshold and keep the lowest rank
  kModeKeyFp = 2,   // lowest fp64 energy (order key) among states within the band
  kModeTiesFp = 3,  // count states whose fp64 energy equals the group's key, lowest rank
  kModeCountKey = 4,    // count states whose key (E, rank) is below (theta, rho)
  kModeCollectKey = 5,  // append every such state (E, rank) to a candidate buffer
};

// Everything one walk needs; pointers may be global or shared memory.
struct WalkCtx {
  int n, C, F, w;             // w = walked bits of this unit
  int nthreads;               // columns are distributed over this many threads
  int thread;                 // this thread's index among them
  const int* sL;              // linear terms L[v] of the unit (v >= F); L[v] for v < F: c(P) parts
  const void* rows4;          // walked rows a >= R (quad layout, int4 or float4), or
  const int* rows1;           //   the same rows, one int per column (generic)
  const int* T;               // walked energies in Gray order
  bool t_global;              // T lives in global memory (use the read-only path)
  // key modes: states with E < theta, or E == theta and rank < rho
  int theta;
  uint64_t rho;
  KeyCand* cand;              // kModeCollectKey: candidate buffer of cand_cap entries
  unsigned long long* cand_count;
  uint32_t cand_cap;
  uint32_t* scratch;          // out-of-line candidate scans: 16 words per thread (shared memory), or null
};

// Column of (thread t, slot jj). Fast layout: quads of 4 consecutive columns, quad k of thread t
// at index k * nthreads + t, so a warp's 16-byte loads of one row are contiguous.
template <int CPT>
__device__ __forceinline__ int column_of(int t, int nthreads, int jj) {
  if constexpr (CPT == 1) return t;
  else return ((((jj >> 2) * nthreads) + t) << 2) | (jj & 3);
}

// Result of a candidate scan (resolve modes).
struct CandScan {
  uint64_t cnt, rmin, kmin;
};

// Resolve-mode scan of one thread's CPT columns (fast layout) at Gray step i, out of line: the
// running energies are read back from the thread's shared-memory slot. Candidates are the
// columns with V + T <= aux (energy <= the mode's threshold); what is counted or kept per mode
// is the same as in Walker::visit_candidates. Called only when a column of the step passes the
// filter, so the unrolled walk stays small.
template <int CPT, int MODE>
static __device__ __noinline__ CandScan scan_candidates(const int* slot, int thread, int nthreads, int C, int n,
                                                       uint64_t prank, uint64_t i, int tv, int aux, int s,
                                                       const double* __restrict__ U64, uint64_t gkey, int theta,
                                                       uint64_t rho, KeyCand* cand, unsigned long long* cand_count,
                                                       uint32_t cand_cap) {
  CandScan r = {0, ~0ull, ~0ull};
  const uint64_t ib = prank | (gray_code(i) << C);
  for (int jj = 0; jj < CPT; ++jj) {
    const int v = slot[jj];
    if (v + tv > aux) continue;
    const int col = ((((jj >> 2) * nthreads) + thread) << 2) | (jj & 3);
    const uint64_t rank = ib | static_cast<uint64_t>(col);
    if constexpr (MODE == kModeTiesInt) {
      ++r.cnt;
      r.rmin = rank < r.rmin ? rank : r.rmin;
    } else if constexpr (MODE == kModeKeyFp) {
      const uint64_t k = order_key(eval64_rank(U64, n, rank));
      r.kmin = k < r.kmin ? k : r.kmin;
    } else if constexpr (MODE == kModeTiesFp) {
      if (order_key(eval64_rank(U64, n, rank)) == gkey) {
        ++r.cnt;
        r.rmin = rank < r.rmin ? rank : r.rmin;
      }
    } else if constexpr (MODE == kModeCountKey || MODE == kModeCollectKey) {
      const int E = v + tv + s;
      if (E < theta || rank < rho) {
        if constexpr (MODE == kModeCountKey) {
          ++r.cnt;
        } else {
          const unsigned long long idx = atomicAdd(cand_count, 1ull);
          if (idx < cand_cap) {
            cand[idx].e = E;
            cand[idx].rank = rank;
          }
        }
      }
    }
  }
  return r;
}

template <int CPT, int R, int MODE, typename VT = int>
struct Walker {
  static_assert(MODE == kModeMin || VOps<VT>::kInt, "resolve modes walk in int32");
  static_assert(VOps<VT>::kInt || (CPT >= 4 && R >= 1), "the biased walk uses the fast layout");
  using O = VOps<VT>;
  using V4 = typename O::V4;
  static constexpr int kSteps = 1 << (R + 1);  // Gray steps per loop iteration
  VT V[CPT];
  VT Row[R > 0 ? R : 1][CPT];
  int s;        // c(P) + sum of L over set walked positions >= R
  int aux;      // kModeMin: order image of (running best minus s); resolve modes: threshold minus s
  bool valid;   // this thread owns real columns (generic blocks may have idle lanes)
  int col0;     // generic: this thread's column
  // resolve accumulators
  uint64_t cnt, rmin, kmin;
  int hq = kIntInf;  // resolve modes, fast layout: minimum of (chunk minimum + T) over the current half

  // --- set-up: running energies of all columns at walked assignment 0, and register rows.
  __device__ __forceinline__ void init(const WalkCtx& c, const int* __restrict__ Ec, const int* __restrict__ M,
                                       int cP) {
    const int t = c.thread, T = c.nthreads, n = c.n, C = c.C;
    s = cP;
    cnt = 0;
    rmin = ~0ull;
    kmin = ~0ull;
    if constexpr (CPT == 1) {
      const int ncols = 1 << C;
      valid = t < ncols;
      col0 = valid ? t : ncols - 1;
      int lc = 0;
      for (int b = 0; b < C; ++b)
        if ((col0 >> b) & 1) lc += c.sL[n - 1 - b];
      V[0] = O::energy(Ec[col0] + lc);
    } else {
      valid = true;
      col0 = 0;
      const int lt = 31 - __clz(T);  // log2(threads)
      constexpr int kq = CPT / 4;    // quads per thread
      constexpr int lk = ctz_c(kq);
      int Lt = 0;
      for (int b = 0; b < lt; ++b)
        if ((t >> b) & 1) Lt += c.sL[n - 1 - (2 + b)];
      const int Le1 = c.sL[n - 1], Le2 = c.sL[n - 2];
      const int4* Ec4 = reinterpret_cast<const int4*>(Ec);
#pragma unroll
      for (int k = 0; k < kq; ++k) {
        int Lk = Lt;
#pragma unroll
        for (int b = 0; b < lk; ++b)
          if ((k >> b) & 1) Lk += c.sL[n - 1 - (2 + lt + b)];
        const int4 e = Ec4[k * T + t];
        V[4 * k + 0] = O::energy(e.x + Lk);
        V[4 * k + 1] = O::energy(e.y + Lk + Le1);
        V[4 * k + 2] = O::energy(e.z + Lk + Le2);
        V[4 * k + 3] = O::energy(e.w + Lk + Le1 + Le2);
      }
      const int nq = (1 << C) >> 2;
      const int4* M4 = reinterpret_cast<const int4*>(M);
#pragma unroll
      for (int a = 0; a < R; ++a) {
        const int v = n - C - 1 - a;
        const int Lv = c.sL[v];
#pragma unroll
        for (int k = 0; k < kq; ++k) {
          const int4 m = M4[(size_t)v * nq + k * T + t];
          Row[a][4 * k + 0] = O::row(m.x + Lv);
          Row[a][4 * k + 1] = O::row(m.y + Lv);
          Row[a][4 * k + 2] = O::row(m.z + Lv);
          Row[a][4 * k + 3] = O::row(m.w + Lv);
        }
      }
    }
  }

  // --- one walked row in shared memory (position a >= R) added with sign d.
  __device__ __forceinline__ void add_dyn_row(const WalkCtx& c, int a, int d) {
    const int rr = a - R;
    if constexpr (CPT == 1) {
      const int m = c.rows1[(rr << c.C) + col0];
      if (d > 0) V[0] += m;
      else V[0] -= m;
    } else {
      constexpr int kq = CPT / 4;
      const int nq = (1 << c.C) >> 2;
      const V4* rp = reinterpret_cast<const V4*>(c.rows4) + (size_t)rr * nq + c.thread;
      if (d > 0) {
#pragma unroll
        for (int k = 0; k < kq; ++k) {
          const V4 m = rp[k * c.nthreads];
          V[4 * k + 0] = O::add(V[4 * k + 0], m.x);
          V[4 * k + 1] = O::add(V[4 * k + 1], m.y);
          V[4 * k + 2] = O::add(V[4 * k + 2], m.z);
          V[4 * k + 3] = O::add(V[4 * k + 3], m.w);
        }
      } else {
#pragma unroll
        for (int k = 0; k < kq; ++k) {
          const V4 m = rp[k * c.nthreads];
          V[4 * k + 0] = O::sub(V[4 * k + 0], m.x);
          V[4 * k + 1] = O::sub(V[4 * k + 1], m.y);
          V[4 * k + 2] = O::sub(V[4 * k + 2], m.z);
          V[4 * k + 3] = O::sub(V[4 * k + 3], m.w);
        }
      }
    }
  }

  // Flip of a shared-memory position: rows change V, the linear term moves the offset s.
  __device__ __forceinline__ void dyn_flip(const WalkCtx& c, int a, int d) {
    add_dyn_row(c, a, d);
    const int Lv = c.sL[c.n - c.C - 1 - a];
    if (d > 0) {
      s += Lv;
      aux -= Lv;
    } else {
      s -= Lv;
      aux += Lv;
    }
  }

  // Walk state at the start of iteration it0 (gray(i0) has only positions >= R set).
  __device__ __forceinline__ void seek(const WalkCtx& c, int64_t it0) {
    if (it0 == 0) return;
    const uint64_t g0 = gray_code(static_cast<uint64_t>(it0) << (R + 1));
    for (int a = R; a < c.w; ++a)
      if ((g0 >> a) & 1u) {
        add_dyn_row(c, a, +1);
        s += c.sL[c.n - c.C - 1 - a];
      }
  }

  // Resolve-mode visit of one step: candidates have V[j] + t <= aux.
  __device__ __forceinline__ void visit_candidates(const WalkCtx& c, uint64_t prank, uint64_t i, int tv,
                                                   const double* __restrict__ U64, uint64_t gkey) {
    const uint64_t ib = prank | (gray_code(i) << c.C);
#pragma unroll
    for (int jj = 0; jj < CPT; ++jj) {
      if (V[jj] + tv <= aux) {
        const uint64_t rank = ib | static_cast<uint64_t>(CPT == 1 ? col0 : column_of<CPT>(c.thread, c.nthreads, jj));
        if constexpr (MODE == kModeTiesInt) {
          ++cnt;
          rmin = rank < rmin ? rank : rmin;
        } else if constexpr (MODE == kModeKeyFp) {
          const uint64_t k = order_key(eval64_rank(U64, c.n, rank));
          kmin = k < kmin ? k : kmin;
        } else if constexpr (MODE == kModeTiesFp) {
          if (order_key(eval64_rank(U64, c.n, rank)) == gkey) {
            ++cnt;
            rmin = rank < rmin ? rank : rmin;
          }
        } else if constexpr (MODE == kModeCountKey || MODE == kModeCollectKey) {
          const int E = V[jj] + tv + s;  // <= theta by the filter above
          if (E < c.theta || rank < c.rho) {
            if constexpr (MODE == kModeCountKey) {
              ++cnt;
            } else {
              const unsigned long long idx = atomicAdd(c.cand_count, 1ull);
              if (idx < c.cand_cap) {
                c.cand[idx].e = E;
                c.cand[idx].rank = rank;
              }
            }
          }
        }
      }
    }
  }

  __device__ __forceinline__ void step(const WalkCtx& c, uint64_t prank, uint64_t i, int tv,
                                       const double* __restrict__ U64, uint64_t gkey) {
    const int m = vmin_bits<VT, CPT>(V);
    if constexpr (MODE == kModeMin) {
      aux = __viaddmin_s32(m, tv, aux);
    } else {
      const bool hit = valid && (m + tv <= aux);
      if (__any_sync(0xffffffffu, hit)) {
        if constexpr (CPT >= 4) {
          if (hit && c.scratch != nullptr) {
            // hand the columns to the out-of-line scan (keeps the unrolled walk small)
            int4* slot = reinterpret_cast<int4*>(c.scratch) + (CPT / 4) * c.thread;
#pragma unroll
            for (int k = 0; k < CPT / 4; ++k) slot[k] = make_int4(V[4 * k], V[4 * k + 1], V[4 * k + 2], V[4 * k + 3]);
            const CandScan r = scan_candidates<CPT, MODE>(reinterpret_cast<const int*>(slot), c.thread, c.nthreads,
                                                           c.C, c.n, prank, i, tv, aux, s, U64, gkey, c.theta, c.rho,
                                                           c.cand, c.cand_count, c.cand_cap);
            cnt += r.cnt;
            rmin = r.rmin < rmin ? r.rmin : rmin;
            kmin = r.kmin < kmin ? r.kmin : kmin;
          } else if (hit) {
            visit_candidates(c, prank, i, tv, U64, gkey);
          }
        } else {
          if (hit) visit_candidates(c, prank, i, tv, U64, gkey);
        }
      }
    }
  }

  // ----- fast layout (CPT >= 4): the loads of an iteration are issued ahead of their use.
  // The walked energies of the next iteration replace those of this one quad by quad as they
  // are consumed, and each shared-memory row is read a few steps before its flip, so neither
  // the read-only cache nor shared memory latency stalls the adds.
  static constexpr int kMid = 1 << R;                          // step after which position R flips
  static constexpr int kAhead = kMid >= 16 ? 8 : (kMid >> 1);  // steps between a row read and its use
  struct RowBuf {
    V4 q[CPT >= 4 ? CPT / 4 : 1];
  };

  __device__ __forceinline__ void load_dyn_row(const WalkCtx& c, int a, RowBuf& b) const {
    constexpr int kq = CPT / 4;
    const int nq = (1 << c.C) >> 2;
    const V4* rp = reinterpret_cast<const V4*>(c.rows4) + (size_t)(a - R) * nq + c.thread;
#pragma unroll
    for (int k = 0; k < kq; ++k) b.q[k] = rp[k * c.nthreads];
  }

  __device__ __forceinline__ void apply_dyn_row(const WalkCtx& c, int a, const RowBuf& b, bool up) {
    constexpr int kq = CPT / 4;
    const int Lv = c.sL[c.n - c.C - 1 - a];
    if (up) {
#pragma unroll
      for (int k = 0; k < kq; ++k) {
        V[4 * k + 0] = O::add(V[4 * k + 0], b.q[k].x);
        V[4 * k + 1] = O::add(V[4 * k + 1], b.q[k].y);
        V[4 * k + 2] = O::add(V[4 * k + 2], b.q[k].z);
        V[4 * k + 3] = O::add(V[4 * k + 3], b.q[k].w);
      }
      s += Lv;
      aux -= Lv;
    } else {
#pragma unroll
      for (int k = 0; k < kq; ++k) {
        V[4 * k + 0] = O::sub(V[4 * k + 0], b.q[k].x);
        V[4 * k + 1] = O::sub(V[4 * k + 1], b.q[k].y);
        V[4 * k + 2] = O::sub(V[4 * k + 2], b.q[k].z);
        V[4 * k + 3] = O::sub(V[4 * k + 3], b.q[k].w);
      }
      s -= Lv;
      aux += Lv;
    }
  }

  template <int E>
  static __device__ __forceinline__ int comp(const int4& x) {
    if constexpr (E == 0) return x.x;
    else if constexpr (E == 1) return x.y;
    else if constexpr (E == 2) return x.z;
    else return x.w;
  }

  static __device__ __forceinline__ int4 load_t4(const WalkCtx& c, const int4* p) {
    return c.t_global ? __ldg(p) : *p;
  }

  // Walked energies are read in quads (int4) through a ring of kRing quads. When a quad has been
  // consumed, the quad kRing positions ahead (in this iteration or the next) is loaded into its
  // slot, so each load has kRing * 4 steps to arrive while few registers hold them. kRing
  // divides the quads of an iteration, so slot q % kRing holds quad q in every iteration.
  static constexpr int kQuads = kSteps >= 4 ? kSteps / 4 : 1;
  static constexpr int kRing = kQuads < 4 ? kQuads : 4;  // divides kQuads
  static_assert(kQuads % kRing == 0, "the ring must divide an iteration's quads");

  // Resolve modes, fast layout: the warp walks the half-iteration that starts at step i0 once
  // more, now with the per-step filter and candidate scan (`step`). Over a half only the register
  // rows flip; their bits follow the reflected Gray code of R bits, from 0 to 2^(R-1) in the
  // first half and back in the second, so the half's first state is one row away from its last.
  // The walk ends where it began, at the half's last state. Runs only when a thread of the warp
  // has a candidate in the half.
  __device__ __forceinline__ void rescan_half(const WalkCtx& c, uint64_t prank, uint64_t i0, bool second,
                                           const double* __restrict__ U64, uint64_t gkey) {
    if constexpr (MODE != kModeMin && CPT >= 4 && R >= 1) {
      add_reg_row(R - 1, second);
      unsigned cur = second ? (1u << (R - 1)) : 0u;
      for (int l = 0; l < kMid; ++l) {
        const uint64_t i = i0 + l;
        const int tv = c.t_global ? __ldg(c.T + i) : c.T[i];
        step(c, prank, i, tv, U64, gkey);
        if (l + 1 < kMid) {
          const int a = __ffs(l + 1) - 1;
          add_reg_row(a, !((cur >> a) & 1u));
          cur ^= 1u << a;
        }
      }
    }
  }

  // V += Row[a] (up) or V -= Row[a], for a run-time register position a.
  __device__ __forceinline__ void add_reg_row(int a, bool up) {
#pragma unroll
    for (int b = 0; b < R; ++b)
      if (b == a) {
#pragma unroll
        for (int jj = 0; jj < CPT; ++jj) V[jj] = up ? O::add(V[jj], Row[b][jj]) : O::sub(V[jj], Row[b][jj]);
      }
  }

  // Steps L.. of one iteration, unrolled by recursion so that every register row index, every
  // flip sign and every prefetch point is a compile-time constant. `tq` is the ring; `tc` points
  // at this iteration's walked energies, `tn` at the next iteration's (or at this one's, on the
  // last).
  template <int L>
  __device__ __forceinline__ void steps_fast(const WalkCtx& c, uint64_t prank, uint64_t base, int64_t iter,
                                             int a_end, int4* tq, const int4* tc, const int4* tn, RowBuf& rb,
                                             const double* __restrict__ U64, uint64_t gkey) {
    if constexpr (L < kSteps) {
      if constexpr (MODE == kModeMin) {
        step(c, prank, base + L, comp<L & 3>(tq[(L >> 2) % kRing]), U64, gkey);
      } else {
        // resolve modes: the minimum pass's work per step, one filter test per half-iteration
        hq = __viaddmin_s32(vmin_bits<VT, CPT>(V), comp<L & 3>(tq[(L >> 2) % kRing]), hq);
        if constexpr (L == kMid - 1 || L == kSteps - 1) {
          const bool hit = hq <= aux;
          hq = kIntInf;
          if (__any_sync(0xffffffffu, hit)) rescan_half(c, prank, base + (L == kMid - 1 ? 0 : kMid), L == kSteps - 1, U64, gkey);
        }
      }
      if constexpr ((L & 3) == 3) {
        constexpr int q = L >> 2;
        if constexpr (q + kRing < kQuads) tq[q % kRing] = load_t4(c, tc + q + kRing);
        else tq[q % kRing] = load_t4(c, tn + (q + kRing - kQuads));
      }
      if constexpr (L == kMid - 1 - kAhead) load_dyn_row(c, R, rb);
      if constexpr (L == kSteps - 1 - kAhead) load_dyn_row(c, a_end, rb);
      if constexpr (L + 1 < kSteps) {
        if constexpr (L + 1 == kMid) {
          // between the two halves: position R, rising on even iterations
          apply_dyn_row(c, R, rb, (iter & 1) == 0);
        } else {
          // register position a < R; its direction depends on L only
          constexpr int a = ctz_c(L + 1);
          constexpr int bit = ((L >> a) ^ (L >> (a + 1))) & 1;
          if constexpr (bit) {
#pragma unroll
            for (int jj = 0; jj < CPT; ++jj) V[jj] = O::sub(V[jj], Row[a][jj]);
          } else {
#pragma unroll
            for (int jj = 0; jj < CPT; ++jj) V[jj] = O::add(V[jj], Row[a][jj]);
          }
        }
      }
      steps_fast<L + 1>(c, prank, base, iter, a_end, tq, tc, tn, rb, U64, gkey);
    }
  }

  // ----- generic layout (one column per thread, R = 0): two steps per iteration.
  __device__ __forceinline__ void steps_generic(const WalkCtx& c, uint64_t prank, uint64_t base, int64_t iter,
                                                const double* __restrict__ U64, uint64_t gkey) {
    const int2* T2 = reinterpret_cast<const int2*>(c.T) + (base >> 1);
    const int2 x = c.t_global ? __ldg(T2) : T2[0];
    step(c, prank, base, x.x, U64, gkey);
    dyn_flip(c, R, (iter & 1) ? -1 : +1);
    step(c, prank, base + 1, x.y, U64, gkey);
  }

  // Walk Gray iterations [it0, it1) of 2^(R+1) steps each. The flip that leaves an iteration is
  // applied while iter + 1 < it_flip_end (it1 for a closed walk; later for a walk that a
  // following call continues).
  __device__ __forceinline__ void walk(const WalkCtx& c, int64_t it0, int64_t it1, int64_t it_flip_end,
                                       uint64_t prank, const double* __restrict__ U64, uint64_t gkey) {
    if constexpr (CPT >= 4 && kSteps >= 4) {
      const int4* T4 = reinterpret_cast<const int4*>(c.T);
      int4 tq[kRing];
      if (it0 < it1) {
#pragma unroll
        for (int q = 0; q < kRing; ++q) tq[q] = load_t4(c, T4 + (static_cast<uint64_t>(it0) << (R - 1)) + q);
      }
      RowBuf rb;
      for (int64_t iter = it0; iter < it1; ++iter) {
        const uint64_t base = static_cast<uint64_t>(iter) << (R + 1);
        const bool flip_end = iter + 1 < it_flip_end;
        // a_end is only read when flip_end; otherwise a valid row (R) is read and left unused
        const int a_end = flip_end ? R + 1 + __ffsll(static_cast<long long>(iter + 1)) - 1 : R;
        const int4* tc = T4 + (base >> 2);
        const int4* tn = T4 + (((iter + 1 < it1) ? base + kSteps : base) >> 2);
        steps_fast<0>(c, prank, base, iter, a_end, tq, tc, tn, rb, U64, gkey);
        if (flip_end) {
          const uint64_t ilast = base + kSteps - 1;
          apply_dyn_row(c, a_end, rb, ((gray_code(ilast) >> a_end) & 1u) == 0);
        }
      }
    } else {
      for (int64_t iter = it0; iter < it1; ++iter) {
        const uint64_t base = static_cast<uint64_t>(iter) << (R + 1);
        static_assert(CPT == 1 && R == 0, "generic layout");
        steps_generic(c, prank, base, iter, U64, gkey);
        if (iter + 1 < it_flip_end) {
          const int a = R + 1 + __ffsll(static_cast<long long>(iter + 1)) - 1;
          const uint64_t ilast = base + kSteps - 1;
          dyn_flip(c, a, ((gray_code(ilast) >> a) & 1u) ? -1 : +1);
        }
      }
    }
  }
};

// ------------------------------------------------------------------------------------------------
// Minimum walk with block bounds (kModeMin, 16 columns x 256 threads; column energies in the
// biased fp32 binade, or in int32 where sum |U_ij| is too large for the binade).
//
// Every state still costs its one add (eq. 9): each Gray step adds a walked row to all of the
// thread's column energies, in a form the compiler can neither merge nor drop, so every
// intermediate column energy is formed:
//  * fp32: an fp32 add, two columns per fp32x2 instruction (fp32 addition does not reassociate);
//  * int32: a fused add-min against a bound of INT_MAX that the compiler cannot see (ALU pipe)
//    where the flip adds the row, and a multiply-add by a -1 it cannot see (the FMA pipe's
//    integer unit) where it subtracts it or where the sign is only known at run time. Plain
//    integer adds would not do: additions whose intermediate sums nobody reads reassociate, and
//    the compiler folds them. The two kinds split the adds between the two pipes.
// What a block bound saves is the minimum over the columns. A block is the 2^R steps between two
// shared-memory flips; inside it only the register rows flip, so s is constant and, for every
// step d of block m and column j,
//     E(d, j) - s = T[2^R m + d] + V_d[j] >= Tmin_m + min_j V_0[j] + D_par,
// where Tmin_m is the least walked energy of the block (a table), V_0 the columns at the
// block's first state and D_par <= 0 the most negative change of any of the thread's columns
// over a block of that parity. A block visits every pattern of the R register bits once, so the
// most negative change of column j is the sum of the negative parts of its signed register rows
// (row R-1 enters added in even blocks, removed in odd ones): D_par is fixed per unit. When the
// bound is above the threshold for every lane of the warp, no state of the block can be at or
// below the threshold, and the block's per-step minima are not formed; otherwise the block is
// walked with them, exactly as the plain minimum walk does.
//
// The threshold is min(this thread's best, G) + band (the fp32 resolution band, plus any margin a
// driver asks for so that unit minima up to E* + margin stay exact). G is the best energy any
// warp of the grid has published for this group so far, starting from sum |U_ij| (which bounds
// every energy from above) lowered by the seeds: the least walked energy (energies of states of
// unit 0, when the group holds it) and the least energy reached by greedy one-flip descents
// inside the group (qubo_seed.cuh).
// Every value involved is an energy some state of the group attains, so the threshold is never
// below the group's minimum E*: a state with E <= E* + band is never in a skipped block. Hence a
// unit holding such a state reports its minimum exactly, every other unit reports the energy of
// a state it evaluated (above E* + band), and the group minimum and the list of units within the
// band are exactly those of the plain walk; the resolution passes are unchanged.
//
// Ranges (int32, sum |U_ij| = S < 2^30): column energies, walked energies, D_par and energies lie
// in [-S, S], the running best minus s in [-2S, 2S]; the bound with band and margin (up to 2S)
// reaches -4S and is formed in 64 bits.
// ------------------------------------------------------------------------------------------------
template <int R, typename VT = float>
struct PrunedMinWalker : Walker<16, R, kModeMin, VT> {
  using B = Walker<16, R, kModeMin, VT>;
  using O = VOps<VT>;
  using V4 = typename O::V4;
  using RowBuf = typename B::RowBuf;
  using LB = typename std::conditional<O::kInt, long long, int>::type;  // bound arithmetic
  static constexpr bool kInt = O::kInt;
  static constexpr int kCPT = 16;
  static constexpr int kThreads = 256;      // 2^12 columns: the quad stride is a constant
  static constexpr int kBlock = 1 << R;     // steps per block
  static constexpr int kRefreshMask = 3;    // blocks between two publications of the warp's best
  static constexpr int kReadMask = 7;       // blocks between two reads of the group's best
  static_assert(R >= 3, "whole quads of walked energies per block");
  static_assert(kThreads * kCPT == 4096, "the control table's row offsets assume 2^12 columns");

  int dmin0, dmin1;  // D_par of even and odd blocks
  int g_best;        // G: the group's best energy known to this warp (absolute, image units)
  int g_pend;        // the group's published best, loaded a block ago and not yet folded into G
  int big;           // int32 walk: INT_MAX, the add-min's bound (from a kernel parameter)
  int mone;          // int32 walk: -1 (from a kernel parameter)

  // --- column updates of the column pair (jj, jj + 1): the row added, subtracted, or added with
  // a sign known only at run time (+1, -1, or 0 for no change).
  __device__ __forceinline__ void cols_add(int jj, VT r0, VT r1) {
    if constexpr (kInt) {
      this->V[jj] = __viaddmin_s32(this->V[jj], r0, big);
      this->V[jj + 1] = __viaddmin_s32(this->V[jj + 1], r1, big);
    } else {
      const float2 t = __fadd2_rn(make_float2(this->V[jj], this->V[jj + 1]), make_float2(r0, r1));
      this->V[jj] = t.x;
      this->V[jj + 1] = t.y;
    }
  }
  __device__ __forceinline__ void cols_sgn(int jj, VT r0, VT r1, VT sg) {
    if constexpr (kInt) {
      asm("mad.lo.s32 %0, %1, %2, %0;" : "+r"(this->V[jj]) : "r"(r0), "r"(sg));
      asm("mad.lo.s32 %0, %1, %2, %0;" : "+r"(this->V[jj + 1]) : "r"(r1), "r"(sg));
    } else {
      const float2 t = __ffma2_rn(make_float2(r0, r1), make_float2(sg, sg), make_float2(this->V[jj], this->V[jj + 1]));
      this->V[jj] = t.x;
      this->V[jj + 1] = t.y;
    }
  }
  __device__ __forceinline__ VT minus_one() const {
    if constexpr (kInt) return mone;
    else return -1.f;
  }
  __device__ __forceinline__ void cols_sub(int jj, VT r0, VT r1) { cols_sgn(jj, r0, r1, minus_one()); }
  __device__ __forceinline__ void row_add(const VT* row) {
#pragma unroll
    for (int jj = 0; jj < kCPT; jj += 2) cols_add(jj, row[jj], row[jj + 1]);
  }
  __device__ __forceinline__ void row_sgn(const VT* row, VT sg) {
#pragma unroll
    for (int jj = 0; jj < kCPT; jj += 2) cols_sgn(jj, row[jj], row[jj + 1], sg);
  }

  // Flips of steps 0..kBlock-2 of a block; position R-1 flips once, with sign sgn (+1 in even
  // blocks, -1 in odd ones); the others with the sign their Gray bit fixes.
  template <int D>
  __device__ __forceinline__ void body(VT sgn) {
    if constexpr (D + 1 < kBlock) {
      constexpr int a = ctz_c(D + 1);
      if constexpr (a == R - 1) {
        row_sgn(this->Row[a], sgn);
      } else {
        constexpr int bit = ((D >> a) ^ (D >> (a + 1))) & 1;  // bit a of gray(D): 1 -> the flip clears it
        if (bit) row_sgn(this->Row[a], minus_one());
        else row_add(this->Row[a]);
      }
      body<D + 1>(sgn);
    }
  }

  __device__ __forceinline__ void init_bounds() {
    if constexpr (kInt) {
      int lo0 = 0, lo1 = 0;
#pragma unroll
      for (int jj = 0; jj < kCPT; ++jj) {
        int neg = 0;  // sum of the negative parts of rows 0..R-2
#pragma unroll
        for (int a = 0; a < R - 1; ++a) neg += min(this->Row[a][jj], 0);
        const int r = this->Row[R - 1][jj];
        lo0 = min(lo0, neg + min(r, 0));
        lo1 = min(lo1, neg + min(-r, 0));
      }
      dmin0 = lo0;
      dmin1 = lo1;
    } else {
      float lo0 = 0.f, lo1 = 0.f;
#pragma unroll
      for (int jj = 0; jj < kCPT; ++jj) {
        float neg = 0.f;  // sum of the negative parts of rows 0..R-2 (exact: integer-valued)
#pragma unroll
        for (int a = 0; a < R - 1; ++a) neg = __fadd_rn(neg, fminf(this->Row[a][jj], 0.f));
        const float r = this->Row[R - 1][jj];
        lo0 = fminf(lo0, __fadd_rn(neg, fminf(r, 0.f)));
        lo1 = fminf(lo1, __fadd_rn(neg, fminf(-r, 0.f)));
      }
      dmin0 = static_cast<int>(lo0);
      dmin1 = static_cast<int>(lo1);
    }
  }

  // One block: bound test and the walk with or without per-step minima. On return V holds the
  // block's last state. lbo = the block's least walked energy + D_par - band; thr = min(this
  // thread's best, G) relative to s, both in the order image of the column energies.
  // Long blocks (R = 7) do the adds of all their steps first, in one straight run of code with the
  // test, which they do not wait for (the scheduler overlaps the minimum tree and the vote with the
  // adds); where the bound then does not clear (rare), the block is walked again from its first
  // state with every per-step minimum: over a block the register rows below R-1 return to zero and
  // row R-1 enters once with sign sgn, so the first state is the last one minus sgn * row R-1.
  // Short blocks fail the bound more often, and there the second walk costs more than the overlap
  // saves: they branch first (measured: n=40 28.43 -> 28.24 ms with the overlap at R = 7; n=32,
  // R = 6, 0.178 -> 0.188 ms).
  __device__ __forceinline__ void block(const WalkCtx& c, int m, LB lbo, int thr, VT sgn) {
    const int m0 = vmin_bits<VT, kCPT>(this->V);
    // biased binade: |every term| <= 4 sum|U| < 2^24, far inside int32 around the bias;
    // int32: the sum is formed in 64 bits
    const bool clear = __all_sync(0xffffffffu, static_cast<LB>(m0) + lbo > thr);
    if constexpr (R >= 7) {
      body<0>(sgn);
      if (!clear) {
        row_sgn(this->Row[R - 1], -sgn);
        exact_block(c, m, m0, sgn);
      }
    } else {
      if (clear) body<0>(sgn);
      else exact_block(c, m, m0, sgn);
    }
  }

  // Register row a (2 <= a < R) added with sign sg.
  template <int A = 2>
  __device__ __forceinline__ void flip_row_rt(int a, VT sg) {
    if constexpr (A < R) {
      if (a == A) row_sgn(this->Row[A], sg);
      else flip_row_rt<A + 1>(a, sg);
    }
  }

  // The block walked with every per-step minimum (rare: the bound did not clear it). A loop over
  // groups of four steps keeps the code small: in group k the flips of steps 4k and 4k + 2 are
  // row 0 (+, -), of step 4k + 1 row 1 (- when k is odd), of step 4k + 3 row 2 + ctz(k + 1).
  __device__ __forceinline__ void exact_block(const WalkCtx& c, int m, int m0, VT sgn) {
    static_assert(R >= 3, "groups of four steps: rows 0 and 1 inside, rows 2..R-1 between");
    const int4* T4 = reinterpret_cast<const int4*>(c.T) + (static_cast<uint32_t>(m) << (R - 2));
    const VT one = -minus_one();
    int4 tq = __ldg(T4);
    this->aux = __viaddmin_s32(m0, tq.x, this->aux);
#pragma unroll 1
    for (int k = 0; k < kBlock / 4; ++k) {
      row_add(this->Row[0]);
      this->aux = __viaddmin_s32(vmin_bits<VT, kCPT>(this->V), tq.y, this->aux);
      row_sgn(this->Row[1], (k & 1) ? minus_one() : one);
      this->aux = __viaddmin_s32(vmin_bits<VT, kCPT>(this->V), tq.z, this->aux);
      row_sgn(this->Row[0], minus_one());
      this->aux = __viaddmin_s32(vmin_bits<VT, kCPT>(this->V), tq.w, this->aux);
      if (k + 1 == kBlock / 4) break;  // the block's last state
      const int a = 2 + __ffs(k + 1) - 1;
      const int d = 4 * k + 3;
      const VT sg = (a == R - 1) ? sgn : ((((d >> a) ^ (d >> (a + 1))) & 1) ? minus_one() : one);
      flip_row_rt(a, sg);
      tq = __ldg(T4 + k + 1);
      this->aux = __viaddmin_s32(vmin_bits<VT, kCPT>(this->V), tq.x, this->aux);
    }
  }

  // The group's best. Every kRefreshMask + 1 blocks the warp publishes its best if it improved on
  // what it last published (a reduction whose result nobody waits for: after the first blocks
  // almost no warp improves, so the shared word sees few updates); every kReadMask + 1 blocks it
  // also loads the grid's value, which walk() folds into G only after the next block's adds, so
  // that the load's latency is hidden behind them.
  __device__ __forceinline__ void exchange_best(int* gbest, bool read) {
    const int v = __reduce_min_sync(0xffffffffu, this->aux - O::kBiasBits + this->s);
    if (v < g_best) {
      if ((threadIdx.x & 31) == 0) atomicMin(gbest, v);
      g_best = v;
    }
    if (read) g_pend = __ldcg(gbest);
  }

  // Whole unit: nblocks (even, < 2^31) blocks of 2^R steps, each but the last followed by a
  // shared-row flip; blk: per-block control (least T, the flip that follows; one padding entry);
  // c.sL holds L, -L at 64 + v and a zero at 128. gbest: the group's published best (absolute
  // image units); band: resolution band plus margin; one: a kernel parameter equal to 1.
  __device__ __forceinline__ void walk(const WalkCtx& c, int nblocks, const BlockCtl* __restrict__ blk, int* gbest,
                                       int band, int one) {
    big = kIntInf - (one - 1);
    mone = -one;
    init_bounds();
    const LB dmb0 = static_cast<LB>(dmin0) - band, dmb1 = static_cast<LB>(dmin1) - band;
    g_best = __ldcg(gbest);
    g_pend = kIntInf;
    // a real best from the first state's columns, so the running best never leaves its range
    this->aux = __viaddmin_s32(vmin_bits<VT, kCPT>(this->V), __ldg(c.T), kIntInf);
    const int4* ctl4 = reinterpret_cast<const int4*>(blk);
    const V4* rows = reinterpret_cast<const V4*>(c.rows4) + c.thread;
    int4 ctl = __ldg(ctl4);
    for (int m = 0; m < nblocks; ++m) {
      const int4 next = __ldg(ctl4 + m + 1);  // one block ahead (the table has a padding entry)
      RowBuf rb;
      {
        const V4* rp = rows + ctl.y;  // in flight while the block is walked
#pragma unroll
        for (int k = 0; k < kCPT / 4; ++k) rb.q[k] = rp[k * kThreads];
      }
      const bool odd = m & 1;
      const int thr = min(this->aux, O::kBiasBits + g_best - this->s);
      block(c, m, static_cast<LB>(ctl.x) + (odd ? dmb1 : dmb0), thr, odd ? minus_one() : -minus_one());
      g_best = min(g_best, g_pend);  // loaded a block ago (kIntInf when nothing was loaded)
      g_pend = kIntInf;
      // the flip that follows (a no-op after the last block: sign 0, linear term 0)
      const float dsgn_f = __int_as_float(ctl.z);
      VT dsgn;
      if constexpr (kInt) dsgn = static_cast<int>(dsgn_f);
      else dsgn = dsgn_f;
#pragma unroll
      for (int k = 0; k < kCPT / 4; ++k) {
        cols_sgn(4 * k + 0, rb.q[k].x, rb.q[k].y, dsgn);
        cols_sgn(4 * k + 2, rb.q[k].z, rb.q[k].w, dsgn);
      }
      const int dl = c.sL[ctl.w];
      this->s += dl;
      this->aux -= dl;
      ctl = next;
      if ((m & kRefreshMask) == kRefreshMask) exchange_best(gbest, (m & kReadMask) == kReadMask);
    }
  }
};

// Iterations of 2^(R+1) steps in a walk over w bits (generic variant: R = 0, w may be 0).
template <int R>
__host__ __device__ inline int64_t walk_iterations(int w) {
  return (w >= R + 1) ? (int64_t(1) << (w - R - 1)) : 0;
}

}  // namespace qgb
