// Packed narrow minimum pass: two columns per 32-bit register (16-bit halves).
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
#include "qubo_search_kernel.cuh"

namespace qgb {
namespace {

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

template <int R>
struct PackedWalker {
  static_assert(R >= 1, "");
  static constexpr int kSteps = 1 << (R + 1);
  static constexpr int kMid = 1 << R;
  static constexpr int kAhead = kMid >= 16 ? 8 : (kMid >> 1);
  uint32_t V[kPW];
  uint32_t Row[R][kPW];
  int s;          // c(P) + sum of L over set walked positions >= R
  uint32_t aux;   // per half: B + (running best - s)
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
  __device__ __forceinline__ void steps(const WalkCtx& c, int64_t iter, int a_end, uint4* tq, const uint4* tn,
                                        RowBuf& rb) {
    if constexpr (L < kSteps) {
      aux = __viaddmin_u16x2(pmin_all<kPW>(V), comp<L & 3>(tq[L >> 2]), aux);
      if constexpr ((L & 3) == 3) tq[L >> 2] = __ldg(tn + (L >> 2));
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
      steps<L + 1>(c, iter, a_end, tq, tn, rb);
    }
  }

  // The whole walk of one unit (iterations [0, niter)), then this thread's best energy.
  __device__ __forceinline__ int walk(const WalkCtx& c, int64_t niter) {
    const uint4* T4 = reinterpret_cast<const uint4*>(c.T);
    uint4 tq[kSteps / 4];
#pragma unroll
    for (int q = 0; q < kSteps / 4; ++q) tq[q] = __ldg(T4 + q);
    RowBuf rb;
    for (int64_t iter = 0; iter < niter; ++iter) {
      const uint64_t base = static_cast<uint64_t>(iter) << (R + 1);
      const bool flip_end = iter + 1 < niter;
      const int a_end = flip_end ? R + 1 + __ffsll(static_cast<long long>(iter + 1)) - 1 : R;
      const uint4* tn = T4 + ((flip_end ? base + kSteps : base) >> 2);
      steps<0>(c, iter, a_end, tq, tn, rb);
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

template <int R>
__global__ void __launch_bounds__(128, 2) packed_min_kernel(const KParams p) {
  extern __shared__ __align__(16) int4 s_rows4[];
  __shared__ int sL[64];
  __shared__ int s_red[32];
  if (p.hdr->status != QUBO_OK) return;
  if (min_pass_owner(p) != kOwnerPacked) return;

  const int tid = threadIdx.x;
  const int nthreads = blockDim.x;
  const int n = p.n, C = p.C, F = p.F, w = p.w;
  const int ncols = 1 << C;
  const int nwords = ncols >> 1;
  const int ndyn = w - R;

  // Stage the walked rows of positions >= R as packed words (without the unit's linear terms).
  uint32_t* s_words = reinterpret_cast<uint32_t*>(s_rows4);
  for (int idx = tid; idx < ndyn * nwords; idx += nthreads) {
    const int rr = idx >> (C - 1), q = idx & (nwords - 1);
    const int v = n - C - 1 - (R + rr);
    const int2 m = reinterpret_cast<const int2*>(p.M + (size_t)v * ncols)[q];
    s_words[idx] = combine(m.x, m.y);
  }

  WalkCtx c;
  c.n = n;
  c.C = C;
  c.F = F;
  c.w = w;
  c.nthreads = nthreads;
  c.thread = tid;
  c.sL = sL;
  c.rows4 = s_rows4;
  c.rows1 = nullptr;
  c.T = reinterpret_cast<const int*>(p.T2);
  c.t_global = true;

  const int64_t niter = walk_iterations<R>(w);
  const int lane = tid & 31, warp = tid >> 5;
  const uint64_t nitems = p.unit_end - p.unit_begin;
  for (uint64_t item = blockIdx.x; item < nitems; item += gridDim.x) {
    const uint64_t u = p.unit_begin + item;
    const uint64_t g = u / p.upg;
    const uint64_t P = p.gbase[g] + (u - g * p.upg);
    __syncthreads();  // previous item is done with sL; staged rows are visible
    unit_linear_terms(p.U, n, F, P, sL, tid, nthreads);
    __syncthreads();
    int cP = 0;
    for (int f = 0; f < F; ++f) cP += sL[f];
    PackedWalker<R> W;
    W.init(c, p.Ec, p.M, cP);
    int best = W.walk(c, niter);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) best = min(best, __shfl_xor_sync(0xffffffffu, best, off));
    if (lane == 0) s_red[warp] = best;
    __syncthreads();
    if (tid == 0) {
      int b = s_red[0];
      for (int k = 1; k < (nthreads >> 5); ++k) b = min(b, s_red[k]);
      p.unit_min[u] = b;
    }
  }
}

}  // namespace

size_t packed_smem_bytes(int C, int w) { return (size_t)(w - kPackedR) << (C + 1); }

cudaError_t launch_search_packed(const KParams& p, int blocks, int threads, size_t smem, cudaStream_t s) {
  auto k = packed_min_kernel<kPackedR>;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  k<<<blocks, threads, smem, s>>>(p);
  return cudaGetLastError();
}

cudaError_t occupancy_packed(int threads, size_t smem, int* blocks_per_sm) {
  auto k = packed_min_kernel<kPackedR>;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  return cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks_per_sm, k, threads, smem);
}

}  // namespace qgb
