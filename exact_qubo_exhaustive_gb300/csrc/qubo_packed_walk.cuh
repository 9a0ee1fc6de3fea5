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

#include <type_traits>

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

// Where a walker reads the interaction rows M[v][*] of the cached columns (int4 q holds columns
// 4q .. 4q+3): a table in global memory, or the row's two half-subset sums in shared memory.
struct GlobalRows {
  const int* M;
  int ncols;
  __device__ __forceinline__ int4 quad(int v, int q) const {
    return reinterpret_cast<const int4*>(M + (size_t)v * ncols)[q];
  }
};
// 12 cached bits split 6 + 6: M[v][j] = H[v][j mod 64] + H[v][64 + j / 64], with H[v][l] the sum
// of U[v][c] over the cached variables c of the low subset l and H[v][64 + h] over the high
// subset h.
struct HalfRows {
  static constexpr int kStride = 128;
  const int* H;
  __device__ __forceinline__ int4 quad(int v, int q) const {
    const int* h = H + v * kStride;
    const int4 a = reinterpret_cast<const int4*>(h)[q & 15];
    const int b = h[64 + (q >> 4)];
    return make_int4(a.x + b, a.y + b, a.z + b, a.w + b);
  }
};

struct TieScan {
  uint64_t cnt, rmin;
};

// Words per thread of the tie walk's scan slot: the 16 column words and the R register rows.
template <int R>
constexpr int scan_slot_words() { return 16 * (1 + R); }

// The states of one half-iteration of thread `owner` (2^R Gray steps from step i0, over which
// only the register rows a < R flip) whose energy relative to s, (half + T) mod 2^16, equals the
// target t: their number and lowest rank. Called by all 32 lanes of a warp together; lane L
// tests steps L, L + 32, ... of the half. `slot` holds the owner's 16 words at the half's last
// step and its register rows. The words at step i differ from those at the last step by the
// register rows whose bits differ between the two Gray codes (+row where step i has the bit,
// -row where the last step has it). Each step is tested with the walk's minimum tree; only a
// step that reaches the target is searched column by column.
template <int R>
static __device__ __noinline__ TieScan scan_half(const uint32_t* slot, int owner, int nthreads, int C,
                                                 uint64_t prank, uint64_t i0, const uint32_t* __restrict__ T2,
                                                 uint32_t t) {
  constexpr int kW = 16, kH = 1 << R;
  const uint4* s4 = reinterpret_cast<const uint4*>(slot);  // quads 0..3: words; 4 + 4a ..: row a
  const unsigned rmask = (1u << R) - 1;
  const unsigned cend = (unsigned)gray_code(i0 + kH - 1) & rmask;
  TieScan r = {0, ~0ull};
  for (int L = threadIdx.x & 31; L < kH; L += 32) {
    const uint64_t i = i0 + L;
    const unsigned cur = (unsigned)gray_code(i) & rmask;
    uint32_t V[kW];
#pragma unroll
    for (int k = 0; k < kW / 4; ++k) {
      const uint4 q = s4[k];
      V[4 * k] = q.x;
      V[4 * k + 1] = q.y;
      V[4 * k + 2] = q.z;
      V[4 * k + 3] = q.w;
    }
#pragma unroll
    for (int a = 0; a < R; ++a) {
      const unsigned here = (cur >> a) & 1u, last = (cend >> a) & 1u;
      if (here != last) {
#pragma unroll
        for (int k = 0; k < kW / 4; ++k) {
          const uint4 q = s4[4 + 4 * a + k];
          const uint32_t rw[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) V[4 * k + e] = here ? V[4 * k + e] + rw[e] : V[4 * k + e] - rw[e];
        }
      }
    }
    const uint32_t tw = __ldg(T2 + i);
    const uint32_t m = __viaddmin_u16x2(pmin_all<kW>(V), tw, 0xffffffffu);
    if ((m & 0xffffu) <= t || (m >> 16) <= t) {
      const uint32_t tv = tw & 0xffffu;
      const uint64_t ib = prank | (gray_code(i) << C);
#pragma unroll 1
      for (int jj = 0; jj < kW; ++jj)
        for (int h = 0; h < 2; ++h) {
          const uint32_t val = (((V[jj] >> (16 * h)) & 0xffffu) + tv) & 0xffffu;
          if (val == t) {
            const int k = jj >> 2, e = jj & 3;
            const uint64_t rank = ib | (uint64_t)((((k * nthreads + owner) << 3)) | (e << 1) | h);
            ++r.cnt;
            r.rmin = rank < r.rmin ? rank : r.rmin;
          }
        }
    }
  }
  return r;
}

// MODE kModeMin: running per-half minimum. MODE kModeTiesInt: count the states whose energy
// equals a target (the known minimum) and keep the lowest rank among them; `aux` then holds the
// target relative to s, B + (target - s), in both halves. The ties walk does the minimum walk's
// work per step and tests once per half-iteration; only a half that reaches the target is
// scanned state by state.
template <int R, int MODE = kModeMin, class RS = GlobalRows>
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
  uint32_t hq = 0xffffffffu;       // kModeTiesInt: per-half minimum of the current half-iteration
  struct RowBuf {
    uint4 q[kPW / 4];
  };
  // The re-walk of a few iterations from half sums (kModeTiesInt with HalfRows) forms the shared
  // rows it flips from the half sums, for its own columns, instead of reading rows staged for the
  // whole block: it needs only the rows of the seek and two flips per iteration.
  static constexpr bool kDirectRows = MODE == kModeTiesInt && std::is_same<RS, HalfRows>::value;
  RS rs_;

  __device__ __forceinline__ void init(const WalkCtx& c, const int* __restrict__ Ec, const RS& rs, int cP) {
    const int t = c.thread, T = c.nthreads, n = c.n, C = c.C;
    rs_ = rs;
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
#pragma unroll
    for (int a = 0; a < R; ++a) {
      const int v = n - C - 1 - a;
      const int Lv = c.sL[v];
#pragma unroll
      for (int k = 0; k < kPW / 4; ++k) {
        const int qi = k * T + t;
        const int4 m0 = rs.quad(v, 2 * qi), m1 = rs.quad(v, 2 * qi + 1);
        Row[a][4 * k + 0] = combine(m0.x + Lv, m0.y + Lv);
        Row[a][4 * k + 1] = combine(m0.z + Lv, m0.w + Lv);
        Row[a][4 * k + 2] = combine(m1.x + Lv, m1.y + Lv);
        Row[a][4 * k + 3] = combine(m1.z + Lv, m1.w + Lv);
      }
    }
  }

  __device__ __forceinline__ void load_dyn_row(const WalkCtx& c, int a, RowBuf& b) const {
    if constexpr (kDirectRows) {
      const int v = c.n - c.C - 1 - a;
#pragma unroll
      for (int k = 0; k < kPW / 4; ++k) {
        const int qi = k * c.nthreads + c.thread;  // word quad: columns qi*8 .. qi*8+7
        const int4 m0 = rs_.quad(v, 2 * qi), m1 = rs_.quad(v, 2 * qi + 1);
        b.q[k] = make_uint4(combine(m0.x, m0.y), combine(m0.z, m0.w), combine(m1.x, m1.y), combine(m1.z, m1.w));
      }
      return;
    }
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
        // running per-half minimum of m + T over the half-iteration; s and the target are
        // constant inside a half, so one test at its end finds every half that reaches the
        // target (no state lies below it, so a hit is an equal value)
        hq = __viaddmin_u16x2(pmin_all<kPW>(V), comp<L & 3>(tq[(L >> 2) % kRing]), hq);
        if constexpr (L == kMid - 1 || L == kSteps - 1) {
          const uint32_t t = aux & 0xffffu;
          const bool hit = (hq & 0xffffu) <= t || (hq >> 16) <= t;
          hq = 0xffffffffu;
          if (__any_sync(0xffffffffu, hit)) {
            // rare: the warp re-scans each hitting thread's half out of line, one step per lane
            // (keeps the unrolled walk small); the counts may land in any lane of the warp, whose
            // totals are summed at the end of the unit
            constexpr int kSlot = scan_slot_words<R>();
            if (hit) {
              uint4* slot = reinterpret_cast<uint4*>(c.scratch + kSlot * c.thread);
#pragma unroll
              for (int k = 0; k < kPW / 4; ++k) slot[k] = make_uint4(V[4 * k], V[4 * k + 1], V[4 * k + 2], V[4 * k + 3]);
#pragma unroll
              for (int a = 0; a < R; ++a)
#pragma unroll
                for (int k = 0; k < kPW / 4; ++k)
                  slot[4 + 4 * a + k] = make_uint4(Row[a][4 * k], Row[a][4 * k + 1], Row[a][4 * k + 2], Row[a][4 * k + 3]);
            }
            __syncwarp();
            constexpr bool second = L == kSteps - 1;
            for (unsigned hm = __ballot_sync(0xffffffffu, hit); hm; hm &= hm - 1) {
              const int owner = (c.thread & ~31) + __ffs(hm) - 1;
              const TieScan r = scan_half<R>(c.scratch + kSlot * owner, owner, c.nthreads, c.C, prank,
                                             base + (second ? kMid : 0), reinterpret_cast<const uint32_t*>(c.T), t);
              cnt += r.cnt;
              rmin = r.rmin < rmin ? r.rmin : rmin;
            }
            __syncwarp();
          }
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

  // Moves the walk to the first state of iteration it0 (Gray step it0 * 2^(R+1)): there the
  // register bits are 0 and the shared-row positions hold that step's Gray code bits.
  __device__ __forceinline__ void seek(const WalkCtx& c, int64_t it0) {
    const uint64_t g0 = gray_code(static_cast<uint64_t>(it0) << (R + 1));
    RowBuf rb;
    for (int a = R; a < c.w; ++a)
      if ((g0 >> a) & 1u) {
        load_dyn_row(c, a, rb);
        apply_dyn_row(c, a, rb, true);
      }
  }

  // The walk of iterations [it0, it1) of one unit (from the state `seek` gives); returns this
  // thread's best energy (kModeMin). prank: the unit's prefix bits in rank position
  // (kModeTiesInt). With s_seg (kModeMin), the minimum of each iteration over the block goes to
  // s_seg[iteration] (shared; atomicMin from each warp).
  __device__ __forceinline__ int walk(const WalkCtx& c, int64_t it0, int64_t it1, uint64_t prank = 0,
                                      int* s_seg = nullptr) {
    const uint4* T4 = reinterpret_cast<const uint4*>(c.T);
    uint4 tq[kRing];
#pragma unroll
    for (int q = 0; q < kRing; ++q) tq[q] = __ldg(T4 + (static_cast<uint64_t>(it0) << (R - 1)) + q);
    RowBuf rb;
    int best = kIntInf;
    for (int64_t iter = it0; iter < it1; ++iter) {
      const uint64_t base = static_cast<uint64_t>(iter) << (R + 1);
      const bool flip_end = iter + 1 < it1;
      const int a_end = flip_end ? R + 1 + __ffsll(static_cast<long long>(iter + 1)) - 1 : R;
      const uint4* tc = T4 + (base >> 2);
      const uint4* tn = T4 + ((flip_end ? base + kSteps : base) >> 2);
      steps<0>(c, prank, base, iter, a_end, tq, tc, tn, rb);
      if constexpr (MODE == kModeMin) {
        if (s_seg) {
          // this iteration's minimum (s is constant from the middle flip to here)
          const int m = min((int)(aux & 0xffffu), (int)(aux >> 16)) - (int)kHalfBias + s;
          best = min(best, m);
          const int wm = __reduce_min_sync(0xffffffffu, m);
          if ((c.thread & 31) == 0) atomicMin(s_seg + iter, wm);
        }
      }
      if (flip_end) {
        const uint64_t ilast = base + kSteps - 1;
        apply_dyn_row(c, a_end, rb, ((gray_code(ilast) >> a_end) & 1u) == 0);
      }
      if constexpr (MODE == kModeMin) {
        // a fresh running minimum for the next iteration, set after the flip (the flip's shift
        // of aux by -L would wrap the all-ones start value)
        if (s_seg) aux = 0xffffffffu;
      }
    }
    if constexpr (MODE == kModeMin) {
      if (s_seg) return best;
    }
    const int lo = (int)(aux & 0xffffu) - (int)kHalfBias;
    const int hi = (int)(aux >> 16) - (int)kHalfBias;
    return min(lo, hi) + s;
  }
};

// ------------------------------------------------------------------------------------------------
// Packed minimum walk with block bounds (128 threads x 32 columns, two per 32-bit word).
//
// The block bound, the threshold and the exactness argument are those of PrunedMinWalker
// (qubo_walk.cuh), taken over the 32 columns (both halves of every word). What changes is how
// every state still gets its add: one word instruction adds a row to two columns, in forms no
// compiler can fold because they depend on values it cannot see: a flip that adds the row is an
// unsigned fused add-min against a UINT_MAX read from a kernel parameter (ALU pipe); a flip that
// subtracts it, or whose sign is known only at run time, is a multiply-add by -1 from the same
// parameter or by the sign (the FMA pipe's integer unit). Word arithmetic modulo 2^32 is exact
// per half (the representation above), so each instruction advances two states exactly.
// ------------------------------------------------------------------------------------------------
template <int R, class RS = GlobalRows>
struct PackedPrunedWalker : PackedWalker<R, kModeMin, RS> {
  using B = PackedWalker<R, kModeMin, RS>;
  using RowBuf = typename B::RowBuf;
  static constexpr int kThreads = 128;    // 2^12 columns: the word-quad stride is a constant
  static constexpr int kBlock = 1 << R;   // steps per block
  static constexpr int kRefreshMask = 3;  // blocks between two publications of the warp's best
  static constexpr int kReadMask = 7;     // blocks between two reads of the group's best
  static_assert(R >= 3, "whole quads of walked energies per block");

  // Per column, the most negative change over an even block, as the packed signed pair of each
  // word: DW = combine(D_lo, D_hi), kept in shared memory (s_dw: 4 word quads per thread, quad k
  // of thread t at k * kThreads + t) so that it takes no registers from the block body. Over an
  // odd block row R-1 enters removed, so the change is DW - Row[R-1]. The per-column bound is
  // min_j (V_0[j] + D[j]) + Tmin_m, the tightest bound that takes the walked energies and the
  // columns apart (every state of the block has E - s = T[d] + V_d[j] >= Tmin_m + V_0[j] + D[j]);
  // the cheap one uses min_j V_0[j] + min_j D[j] and is tested first.
  uint4* s_dw;
  int dmin0, dmin1;  // the least of those changes over the thread's columns (even, odd blocks)
  // The per-column bound pays where blocks often fail the cheap one: short units (R = 6; the
  // batched n=24 workload had 18 % of its warp-blocks walked exactly with the cheap bound alone,
  // and its pass went from 2.60 to 2.23 ms with both). With R = 7 it is compiled out: there the
  // cheap bound clears almost every block (n=40 with entries in [-4, 4]: 0.001 % walked
  // exactly), and the extra code cost 4 % (19.05 against 19.88 ms).
  static constexpr bool kColumnBound = R <= 6;
  int g_best;        // G: the group's best energy known to this warp
  int g_pend;        // the group's published best, loaded a block ago and not yet folded into G
  int best;          // this thread's best energy minus s
  uint32_t big;      // UINT_MAX, the add-min's bound (from a kernel parameter)
  uint32_t mone;     // -1 modulo 2^32 (from a kernel parameter)

  __device__ __forceinline__ void words_add(const uint32_t* row) {
#pragma unroll
    for (int jj = 0; jj < kPW; ++jj) this->V[jj] = __viaddmin_u32(this->V[jj], row[jj], big);
  }
  __device__ __forceinline__ void words_sgn(const uint32_t* row, uint32_t sg) {
#pragma unroll
    for (int jj = 0; jj < kPW; ++jj) asm("mad.lo.u32 %0, %1, %2, %0;" : "+r"(this->V[jj]) : "r"(row[jj]), "r"(sg));
  }

  // Flips of steps 0..kBlock-2 of a block; position R-1 flips once, with sign sgn (+1 in even
  // blocks, -1 in odd ones); the others with the sign their Gray bit fixes.
  template <int D>
  __device__ __forceinline__ void body(uint32_t sgn) {
    if constexpr (D + 1 < kBlock) {
      constexpr int a = ctz_c(D + 1);
      if constexpr (a == R - 1) {
        words_sgn(this->Row[a], sgn);
      } else {
        constexpr int bit = ((D >> a) ^ (D >> (a + 1))) & 1;  // bit a of gray(D): 1 -> the flip clears it
        if (bit) words_sgn(this->Row[a], mone);
        else words_add(this->Row[a]);
      }
      body<D + 1>(sgn);
    }
  }

  // The two signed values of a row word combine(lo, hi) = hi * 2^16 + lo.
  static __device__ __forceinline__ void split(uint32_t w, int& lo, int& hi) {
    lo = (int)(int16_t)(w & 0xffffu);
    hi = ((int)w - lo) >> 16;
  }

  __device__ __forceinline__ void init_bounds() {
    int lo0 = 0, lo1 = 0;
#pragma unroll
    for (int jj = 0; jj < kPW; ++jj) {
      int neg_l = 0, neg_h = 0;  // sums of the negative parts of rows 0..R-2, per half
#pragma unroll
      for (int a = 0; a < R - 1; ++a) {
        int l, h;
        split(this->Row[a][jj], l, h);
        neg_l += min(l, 0);
        neg_h += min(h, 0);
      }
      int rl, rh;
      split(this->Row[R - 1][jj], rl, rh);
      if (kColumnBound && s_dw) {
        uint32_t* q = reinterpret_cast<uint32_t*>(s_dw + (jj >> 2) * kThreads + threadIdx.x);
        q[jj & 3] = combine(neg_l + min(rl, 0), neg_h + min(rh, 0));
      }
      lo0 = min(lo0, min(neg_l + min(rl, 0), neg_h + min(rh, 0)));
      lo1 = min(lo1, min(neg_l + min(-rl, 0), neg_h + min(-rh, 0)));
    }
    dmin0 = lo0;
    dmin1 = lo1;
  }

  // Least lower bound over the thread's columns, relative to s without the walked energy:
  // min_j (V_0[j] + D[j]) for a block of parity odd. Every sum stays inside a half's range
  // (|V_0 + D| <= 2 sum |U| < 2^15), so the word adds are exact per half.
  __device__ __forceinline__ int column_bound(bool odd) const {
    uint32_t x[kPW];
#pragma unroll
    for (int k = 0; k < kPW / 4; ++k) {
      const uint4 d = s_dw[k * kThreads + threadIdx.x];
      x[4 * k + 0] = this->V[4 * k + 0] + d.x;
      x[4 * k + 1] = this->V[4 * k + 1] + d.y;
      x[4 * k + 2] = this->V[4 * k + 2] + d.z;
      x[4 * k + 3] = this->V[4 * k + 3] + d.w;
    }
    if (odd) {
#pragma unroll
      for (int jj = 0; jj < kPW; ++jj) x[jj] -= this->Row[R - 1][jj];
    }
    return lesser_half(pmin_all<kPW>(x));
  }

  // Least column value of the two halves of a 16x2 minimum word.
  static __device__ __forceinline__ int lesser_half(uint32_t m) {
    return min((int)(m & 0xffffu), (int)(m >> 16)) - (int)kHalfBias;
  }

  // The block walked with every per-step minimum (rare: the bound did not clear it), in groups of
  // four steps as in PrunedMinWalker::exact_block, with the packed per-half add-min of the walked
  // energy (T2: T modulo 2^16 in both halves). With s_seg, the warp's minimum over the block goes
  // to s_seg[m] (shared; atomicMin): a block no warp walked exactly holds no state at or below
  // the threshold, so its entry may stay at its start value.
  __device__ __forceinline__ void exact_block(const uint32_t* __restrict__ T2, int m, uint32_t pm0, uint32_t sgn,
                                              int* s_seg) {
    const uint4* T4 = reinterpret_cast<const uint4*>(T2) + (static_cast<uint32_t>(m) << (R - 2));
    const uint32_t one = 0u - mone;
    uint4 tq = __ldg(T4);
    uint32_t pa = __viaddmin_u16x2(pm0, tq.x, 0xffffffffu);
#pragma unroll 1
    for (int k = 0; k < kBlock / 4; ++k) {
      words_add(this->Row[0]);
      pa = __viaddmin_u16x2(pmin_all<kPW>(this->V), tq.y, pa);
      words_sgn(this->Row[1], (k & 1) ? mone : one);
      pa = __viaddmin_u16x2(pmin_all<kPW>(this->V), tq.z, pa);
      words_sgn(this->Row[0], mone);
      pa = __viaddmin_u16x2(pmin_all<kPW>(this->V), tq.w, pa);
      if (k + 1 == kBlock / 4) break;  // the block's last state
      const int a = 2 + __ffs(k + 1) - 1;
      const int d = 4 * k + 3;
      const uint32_t sg = (a == R - 1) ? sgn : ((((d >> a) ^ (d >> (a + 1))) & 1) ? mone : one);
      flip_row_rt(a, sg);
      tq = __ldg(T4 + k + 1);
      pa = __viaddmin_u16x2(pmin_all<kPW>(this->V), tq.x, pa);
    }
    const int bm = lesser_half(pa);
    best = min(best, bm);
    if (s_seg) {
      const int wm = __reduce_min_sync(0xffffffffu, bm + this->s);
      if ((threadIdx.x & 31) == 0) atomicMin(s_seg + m, wm);
    }
  }

  template <int A = 2>
  __device__ __forceinline__ void flip_row_rt(int a, uint32_t sg) {
    if constexpr (A < R) {
      if (a == A) words_sgn(this->Row[A], sg);
      else flip_row_rt<A + 1>(a, sg);
    }
  }

  __device__ __forceinline__ void exchange_best(int* gbest, bool read) {
    const int v = __reduce_min_sync(0xffffffffu, best + this->s);
    if (v < g_best) {
      if ((threadIdx.x & 31) == 0) atomicMin(gbest, v);
      g_best = v;
    }
    if (read) g_pend = __ldcg(gbest);  // folded into G after the next block (PrunedMinWalker)
  }

  // Whole unit: nblocks (even) blocks of 2^R steps, each but the last followed by a shared-row
  // flip, as PrunedMinWalker::walk (blk: the same control table; its row offsets count the 16-
  // column layout's quads, twice this layout's word quads). Returns this thread's best energy.
  // s_seg (optional): per-block minima of the exactly walked blocks (see exact_block). dw:
  // shared memory for the per-column changes (kThreads x 16 words), or null for the cheap bound
  // alone.
  __device__ __forceinline__ int walk(const WalkCtx& c, int nblocks, const BlockCtl* __restrict__ blk,
                                      const uint32_t* __restrict__ T2, int* gbest, int band, int one,
                                      int* s_seg = nullptr, uint4* dw = nullptr) {
    big = 0xffffffffu - (uint32_t)(one - 1);
    mone = 0u - (uint32_t)one;
    s_dw = dw;
    init_bounds();
    g_best = __ldcg(gbest);
    g_pend = kIntInf;
    // a real best from the first state's columns
    best = lesser_half(__viaddmin_u16x2(pmin_all<kPW>(this->V), __ldg(T2), 0xffffffffu));
    const int4* ctl4 = reinterpret_cast<const int4*>(blk);
    const uint4* rows = reinterpret_cast<const uint4*>(c.rows4) + c.thread;
    int4 ctl = __ldg(ctl4);
    for (int m = 0; m < nblocks; ++m) {
      const int4 next = __ldg(ctl4 + m + 1);  // one block ahead (the table has a padding entry)
      RowBuf rb;
      {
        const uint4* rp = rows + (ctl.y >> 1);  // in flight while the block is walked
#pragma unroll
        for (int k = 0; k < kPW / 4; ++k) rb.q[k] = rp[k * kThreads];
      }
      const bool odd = m & 1;
      const int thr = min(best, g_best - this->s);
      const uint32_t sgn = odd ? mone : 0u - mone;
      // the cheap bound (least column plus least change) first; where it does not clear every
      // lane, the per-column one
      const uint32_t pm0 = pmin_all<kPW>(this->V);
      bool clear = __all_sync(0xffffffffu, lesser_half(pm0) + ctl.x + (odd ? dmin1 : dmin0) - band > thr);
      if constexpr (kColumnBound) {
        if (!clear && s_dw) clear = __all_sync(0xffffffffu, column_bound(odd) + ctl.x - band > thr);
        if (clear) {
          body<0>(sgn);
        } else {
          exact_block(T2, m, pm0, sgn, s_seg);
        }
      } else {
        // long blocks: the adds first, overlapped with the test, and a second walk from the
        // block's first state where the bound does not clear (as PrunedMinWalker::block)
        body<0>(sgn);
        if (!clear) {
          words_sgn(this->Row[R - 1], 0u - sgn);
          exact_block(T2, m, pm0, sgn, s_seg);
        }
      }
      g_best = min(g_best, g_pend);  // loaded a block ago (kIntInf when nothing was loaded)
      g_pend = kIntInf;
      // the flip that follows (a no-op after the last block: sign 0, linear term 0)
      const uint32_t dsg = (uint32_t)static_cast<int>(__int_as_float(ctl.z));
#pragma unroll
      for (int k = 0; k < kPW / 4; ++k) {
        asm("mad.lo.u32 %0, %1, %2, %0;" : "+r"(this->V[4 * k + 0]) : "r"(rb.q[k].x), "r"(dsg));
        asm("mad.lo.u32 %0, %1, %2, %0;" : "+r"(this->V[4 * k + 1]) : "r"(rb.q[k].y), "r"(dsg));
        asm("mad.lo.u32 %0, %1, %2, %0;" : "+r"(this->V[4 * k + 2]) : "r"(rb.q[k].z), "r"(dsg));
        asm("mad.lo.u32 %0, %1, %2, %0;" : "+r"(this->V[4 * k + 3]) : "r"(rb.q[k].w), "r"(dsg));
      }
      const int dl = c.sL[ctl.w];
      this->s += dl;
      best -= dl;
      ctl = next;
      if ((m & kRefreshMask) == kRefreshMask) exchange_best(gbest, (m & kReadMask) == kReadMask);
    }
    return best + this->s;
  }
};

}  // namespace packed
}  // namespace qgb
