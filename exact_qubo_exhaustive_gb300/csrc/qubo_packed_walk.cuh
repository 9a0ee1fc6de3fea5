// Packed narrow walker: two column energies per 32-bit register (16-bit halves).
//
// Terastate-per-second QUBO Brute-Force on a Single GPU, §IV-B.5: when every energy the walk
// forms fits 16 bits, two of them share one 32-bit word and one instruction advances both, which
// doubles the states per instruction. Here the range is proven rather than estimated: every
// running column energy is a sum of distinct entries of U and every (best - offset) difference
// is at most 2 sum |U|, so sum |U| <= kPackedMaxAbsSum = 2^14 - 1 keeps each value v inside
// (-2^15, 2^15), held as the unsigned half B + v with B = 2^15.
//
// Word of columns (lo, hi): (B + V_hi) * 2^16 + (B + V_lo). Adding the signed combination
// r_hi * 2^16 + r_lo with one 32-bit add gives (B + V_hi + r_hi) * 2^16 + (B + V_lo + r_lo)
// exactly, and since the low half stays inside [0, 2^16) no carry crosses the halves. The
// minimum over columns is a tree of 3-input unsigned 16x2 minima, and the walked energy enters
// through a per-half add-then-min (both DPX instructions), with T stored as its low 16 bits in
// both halves (per-half arithmetic is modulo 2^16, so that pattern adds T to each half).
//
// Layout: 32 columns per thread (16 words = 4 quads of 4 words); word quad k of thread t is
// quad index k*T + t, so word (k, e) holds columns 2*((k*T + t)*4 + e) + {0, 1}. The walk is the
// fast walk of the int32 pass (R register rows, shared rows and walked energies read ahead).
#pragma once

#include "qubo_walk.cuh"

namespace qgb {
namespace packed {

constexpr int kPW = 16;              // words per thread (32 columns)
constexpr uint32_t kHalfBias = 1u << 15;

__device__ __forceinline__ uint32_t pmin3(uint32_t a, uint32_t b, uint32_t c) { return __vimin3_u16x2(a, b, c); }

template <int N>
__device__ __forceinline__ uint32_t pmin_all(const uint32_t* v) {
  if constexpr (N == 1) {
    return v[0];
  } else if constexpr (N == 2) {
    return pmin3(v[0], v[1], v[1]);
  } else {
    constexpr int G = (N + 2) / 3;
    uint32_t w[G];
#pragma unroll
    for (int g = 0; g < G; ++g) {
      if (3 * g + 2 < N) w[g] = pmin3(v[3 * g], v[3 * g + 1], v[3 * g + 2]);
      else if (3 * g + 1 < N) w[g] = pmin3(v[3 * g], v[3 * g + 1], v[3 * g + 1]);
      else w[g] = v[3 * g];
    }
    return pmin_all<G>(w);
  }
}

// Two signed values as the exact signed combination hi * 2^16 + lo.
__device__ __forceinline__ uint32_t combine(int lo, int hi) { return (uint32_t)(hi * 65536 + lo); }

struct TieScan {
  uint64_t cnt, rmin;
};

// The columns of one thread's 16 words (read back from `slot`) at Gray step i whose energy
// relative to s, (half + T) mod 2^16, equals the target t: their number and lowest rank.
static __device__ __noinline__ TieScan scan_ties(const uint4* slot, int thread, int nthreads, int C, uint64_t prank,
                                                 uint64_t i, uint32_t tv, uint32_t t) {
  TieScan r = {0, ~0ull};
  const uint64_t ib = prank | (gray_code(i) << C);
  for (int k = 0; k < kPW / 4; ++k) {
    const uint4 q = slot[k];
    const uint32_t words[4] = {q.x, q.y, q.z, q.w};
    for (int e = 0; e < 4; ++e)
      for (int h = 0; h < 2; ++h) {
        const uint32_t val = (((words[e] >> (16 * h)) & 0xffffu) + tv) & 0xffffu;
        if (val == t) {
          const uint64_t rank = ib | (uint64_t)((((k * nthreads + thread) << 3)) | (e << 1) | h);
          ++r.cnt;
          r.rmin = rank < r.rmin ? rank : r.rmin;
        }
      }
  }
  return r;
}

// MODE kModeMin: running per-half minimum. MODE kModeTiesInt: count the states whose energy
// equals a target (the known minimum) and keep the lowest rank among them; `aux` then holds the
// target relative to s, B + (target - s), in both halves.
template <int R, int MODE = kModeMin>
struct PackedWalker {
  static_assert(MODE == kModeMin || MODE == kModeTiesInt, "");
  static_assert(R >= 1, "");
  static constexpr int kSteps = 1 << (R + 1);
  static constexpr int kMid = 1 << R;
  static constexpr int kAhead = kMid >= 16 ? 8 : (kMid >> 1);
  static constexpr int kQuads = kSteps / 4;                 // walked-energy quads per iteration
  static constexpr int kRing = kQuads < 4 ? kQuads : 4;     // quads held ahead; divides kQuads
  static_assert(kQuads % kRing == 0, "the ring must divide an iteration's quads");
  uint32_t V[kPW];
  uint32_t Row[R][kPW];
  int s;          // c(P) + sum of L over set walked positions >= R
  uint32_t aux;   // per half: B + (running best - s), or B + (target - s)
  uint64_t cnt = 0, rmin = ~0ull;  // kModeTiesInt
  struct RowBuf {
    uint4 q[kPW / 4];
  };

  __device__ __forceinline__ void init(const WalkCtx& c, const int* __restrict__ Ec, const int* __restrict__ M,
                                       int cP) {
    const int t = c.thread, T = c.nthreads, n = c.n, C = c.C;
    s = cP;
    aux = 0xffffffffu;
    const int lt = 31 - __clz(T);
    int Lt = 0;
    for (int b = 0; b < lt; ++b)
      if ((t >> b) & 1) Lt += c.sL[n - 1 - (3 + b)];
    const int L0 = c.sL[n - 1], L1 = c.sL[n - 2], L2 = c.sL[n - 3];
    const int4* Ec4 = reinterpret_cast<const int4*>(Ec);
#pragma unroll
    for (int k = 0; k < kPW / 4; ++k) {
      int Lk = Lt;
#pragma unroll
      for (int b = 0; b < 2; ++b)
        if ((k >> b) & 1) Lk += c.sL[n - 1 - (3 + lt + b)];
      const int qi = k * T + t;  // word quad: columns qi*8 .. qi*8+7
      const int4 e0 = Ec4[2 * qi], e1 = Ec4[2 * qi + 1];
      const int ec[8] = {e0.x, e0.y, e0.z, e0.w, e1.x, e1.y, e1.z, e1.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int Le = Lk + ((e & 1) ? L1 : 0) + ((e & 2) ? L2 : 0);
        const int lo = ec[2 * e] + Le, hi = ec[2 * e + 1] + Le + L0;
        V[4 * k + e] = ((kHalfBias + (uint32_t)hi) << 16) | ((kHalfBias + (uint32_t)lo) & 0xffffu);
      }
    }
    const int ncols = 1 << C;
#pragma unroll
    for (int a = 0; a < R; ++a) {
      const int v = n - C - 1 - a;
      const int Lv = c.sL[v];
      const int4* Mv4 = reinterpret_cast<const int4*>(M + (size_t)v * ncols);
#pragma unroll
      for (int k = 0; k < kPW / 4; ++k) {
        const int qi = k * T + t;
        const int4 m0 = Mv4[2 * qi], m1 = Mv4[2 * qi + 1];
        Row[a][4 * k + 0] = combine(m0.x + Lv, m0.y + Lv);
        Row[a][4 * k + 1] = combine(m0.z + Lv, m0.w + Lv);
        Row[a][4 * k + 2] = combine(m1.x + Lv, m1.y + Lv);
        Row[a][4 * k + 3] = combine(m1.z + Lv, m1.w + Lv);
      }
    }
  }

  __device__ __forceinline__ void load_dyn_row(const WalkCtx& c, int a, RowBuf& b) const {
    const int nq = (1 << c.C) >> 3;  // word quads per row
    const uint4* rp = reinterpret_cast<const uint4*>(c.rows4) + (size_t)(a - R) * nq + c.thread;
#pragma unroll
    for (int k = 0; k < kPW / 4; ++k) b.q[k] = rp[k * c.nthreads];
  }

  __device__ __forceinline__ void apply_dyn_row(const WalkCtx& c, int a, const RowBuf& b, bool up) {
    const int Lv = c.sL[c.n - c.C - 1 - a];
    if (up) {
#pragma unroll
      for (int k = 0; k < kPW / 4; ++k) {
        V[4 * k + 0] += b.q[k].x;
        V[4 * k + 1] += b.q[k].y;
        V[4 * k + 2] += b.q[k].z;
        V[4 * k + 3] += b.q[k].w;
      }
      s += Lv;
      aux -= (uint32_t)(Lv * 65537);
    } else {
#pragma unroll
      for (int k = 0; k < kPW / 4; ++k) {
        V[4 * k + 0] -= b.q[k].x;
        V[4 * k + 1] -= b.q[k].y;
        V[4 * k + 2] -= b.q[k].z;
        V[4 * k + 3] -= b.q[k].w;
      }
      s -= Lv;
      aux += (uint32_t)(Lv * 65537);
    }
  }

  template <int E>
  static __device__ __forceinline__ uint32_t comp(const uint4& x) {
    if constexpr (E == 0) return x.x;
    else if constexpr (E == 1) return x.y;
    else if constexpr (E == 2) return x.z;
    else return x.w;
  }

  template <int L>
  __device__ __forceinline__ void steps(const WalkCtx& c, uint64_t prank, uint64_t base, int64_t iter, int a_end,
                                        uint4* tq, const uint4* tc, const uint4* tn, RowBuf& rb) {
    if constexpr (L < kSteps) {
      if constexpr (MODE == kModeMin) {
        aux = __viaddmin_u16x2(pmin_all<kPW>(V), comp<L & 3>(tq[(L >> 2) % kRing]), aux);
      } else {
        // per half m + T (no state lies below the target, so a hit is an equal half)
        const uint32_t q = __viaddmin_u16x2(pmin_all<kPW>(V), comp<L & 3>(tq[(L >> 2) % kRing]), 0xffffffffu);
        const uint32_t t = aux & 0xffffu;
        const bool hit = (q & 0xffffu) <= t || (q >> 16) <= t;
        if (__any_sync(0xffffffffu, hit) && hit) {
          // rare: hand the thread's words to an out-of-line scan (keeps the unrolled walk small)
          uint4* slot = reinterpret_cast<uint4*>(c.scratch) + 4 * c.thread;
#pragma unroll
          for (int k = 0; k < kPW / 4; ++k) slot[k] = make_uint4(V[4 * k], V[4 * k + 1], V[4 * k + 2], V[4 * k + 3]);
          const TieScan r = scan_ties(slot, c.thread, c.nthreads, c.C, prank, base + L,
                                      comp<L & 3>(tq[(L >> 2) % kRing]) & 0xffffu, t);
          cnt += r.cnt;
          rmin = r.rmin < rmin ? r.rmin : rmin;
        }
      }
      if constexpr ((L & 3) == 3) {
        constexpr int q = L >> 2;
        if constexpr (q + kRing < kQuads) tq[q % kRing] = __ldg(tc + q + kRing);
        else tq[q % kRing] = __ldg(tn + (q + kRing - kQuads));
      }
      if constexpr (L == kMid - 1 - kAhead) load_dyn_row(c, R, rb);
      if constexpr (L == kSteps - 1 - kAhead) load_dyn_row(c, a_end, rb);
      if constexpr (L + 1 < kSteps) {
        if constexpr (L + 1 == kMid) {
          apply_dyn_row(c, R, rb, (iter & 1) == 0);
        } else {
          constexpr int a = ctz_c(L + 1);
          constexpr int bit = ((L >> a) ^ (L >> (a + 1))) & 1;
          if constexpr (bit) {
#pragma unroll
            for (int jj = 0; jj < kPW; ++jj) V[jj] -= Row[a][jj];
          } else {
#pragma unroll
            for (int jj = 0; jj < kPW; ++jj) V[jj] += Row[a][jj];
          }
        }
      }
      steps<L + 1>(c, prank, base, iter, a_end, tq, tc, tn, rb);
    }
  }

  // The whole walk of one unit (iterations [0, niter)); returns this thread's best energy
  // (kModeMin). prank: the unit's prefix bits in rank position (kModeTiesInt).
  __device__ __forceinline__ int walk(const WalkCtx& c, int64_t niter, uint64_t prank = 0) {
    const uint4* T4 = reinterpret_cast<const uint4*>(c.T);
    uint4 tq[kRing];
#pragma unroll
    for (int q = 0; q < kRing; ++q) tq[q] = __ldg(T4 + q);
    RowBuf rb;
    for (int64_t iter = 0; iter < niter; ++iter) {
      const uint64_t base = static_cast<uint64_t>(iter) << (R + 1);
      const bool flip_end = iter + 1 < niter;
      const int a_end = flip_end ? R + 1 + __ffsll(static_cast<long long>(iter + 1)) - 1 : R;
      const uint4* tc = T4 + (base >> 2);
      const uint4* tn = T4 + ((flip_end ? base + kSteps : base) >> 2);
      steps<0>(c, prank, base, iter, a_end, tq, tc, tn, rb);
      if (flip_end) {
        const uint64_t ilast = base + kSteps - 1;
        apply_dyn_row(c, a_end, rb, ((gray_code(ilast) >> a_end) & 1u) == 0);
      }
    }
    const int lo = (int)(aux & 0xffffu) - (int)kHalfBias;
    const int hi = (int)(aux >> 16) - (int)kHalfBias;
    return min(lo, hi) + s;
  }
};

}  // namespace packed
}  // namespace qgb
