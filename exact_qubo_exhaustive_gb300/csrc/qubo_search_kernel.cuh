// Enumeration kernel: a persistent grid walks work units (fixed prefixes, §III-C1) or, in the
// resolve modes, segments of the units whose minimum reached their group's minimum.
#pragma once

#include <type_traits>

#include "qubo_walk.cuh"

namespace qgb {

struct KParams {
  int n, C, F, w;           // w = walked bits per unit
  int dtype;
  int biased_active;        // a biased-binade minimum pass runs when sum |U| <= kBiasedWalkMaxAbsSum
  int packed_active;        // a packed 16x2 minimum pass runs when sum |U| <= kPackedMaxAbsSum
  int seg_bits;             // resolve: segments per tied unit = 2^seg_bits
  int ngroups;
  uint64_t upg;             // units per group
  uint64_t unit_begin, unit_end;  // kModeMin: global unit range of this launch
  DevHeader* hdr;
  const int32_t* U;         // n x n int32 image
  const double* U64;        // n x n fp64 folded (fp32 path)
  const int32_t* M;
  const int32_t* Ec;
  const int32_t* T;
  const uint32_t* T2;       // packed pass: T's low 16 bits in both halves
  const BlockCtl* blk;      // block-bounded minimum pass: per-block minimum of T and following flip
  int32_t* gthr;            // pruned minimum passes: best energy published so far, per group
  int margin;               // extra margin of the block bound test (image units)
  int one;                  // 1: the int32 bounded walk derives its opaque constants from it
  const uint64_t* gbase;
  int32_t* unit_min;
  uint32_t* tied;
  int32_t* gmin;
  uint64_t* grank;
  uint64_t* gties;
  uint64_t* gkey;
  qubo_result* results;
  // key modes (k lowest energies)
  int theta;
  uint64_t rho;
  KeyCand* cand;
  unsigned long long* cand_count;  // kModeCountKey: the count; kModeCollectKey: the append index
  uint32_t cand_cap;
};

// Which of the minimum passes of one launch sequence does the work; the others exit at once.
// The narrowest representation that the proven range admits wins.
enum MinPassOwner : int { kOwnerPacked = 1, kOwnerBiased = 2, kOwnerInt = 3 };
__device__ __forceinline__ int min_pass_owner(const KParams& p) {
  const int64_t S = p.hdr->abs_sum;
  if (p.packed_active && S <= kPackedMaxAbsSum) return kOwnerPacked;
  if (p.biased_active && S <= kBiasedWalkMaxAbsSum) return kOwnerBiased;
  return kOwnerInt;
}

// Linear terms of a unit with prefix P (F bits, bit F-1-f is x_f):
//   sL[v] = sum_{f<F, x_f=1} U[f][v]                 for free v >= F (diag(x_f U_fr) of §III-C1),
//   sL[f] = x_f * sum_{f<=f2<F, x_f2=1} U[f][f2]      for fixed f < F (their sum is c(P)).
__device__ __forceinline__ void unit_linear_terms(const int32_t* __restrict__ U, int n, int F, uint64_t P, int* sL,
                                                  int tid, int nthreads) {
  for (int v = tid; v < n; v += nthreads) {
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

// The same terms formed by one warp for its own use (lane l: variables l and l + 32; n <= 62),
// with -L at 64 + v and a zero at 128 (the block-bounded walkers' signed linear terms).
__device__ __forceinline__ void warp_linear_terms(const int32_t* __restrict__ U, int n, int F, uint64_t P, int* sl,
                                                  int lane) {
  for (int v = lane; v < 64; v += 32) {
    int acc = 0;
    if (v < n) {
      if (v >= F) {
        for (int f = 0; f < F; ++f)
          if ((P >> (F - 1 - f)) & 1u) acc += U[f * n + v];
      } else if ((P >> (F - 1 - v)) & 1u) {
        for (int f2 = v; f2 < F; ++f2)
          if ((P >> (F - 1 - f2)) & 1u) acc += U[v * n + f2];
      }
    }
    sl[v] = acc;
    sl[64 + v] = -acc;
  }
  if (lane == 0) sl[128] = 0;
}

// Minimum-pass walk of one unit in value type VT; returns this thread's best energy (int32).
template <int CPT, int R, typename VT>
__device__ __forceinline__ int min_walk(const WalkCtx& c, const KParams& p, int cP, int64_t niter) {
  Walker<CPT, R, kModeMin, VT> W;
  W.init(c, p.Ec, p.M, cP);
  W.aux = kIntInf;
  W.walk(c, 0, niter, niter, 0, nullptr, 0);
  return W.aux - VOps<VT>::kBiasBits + W.s;
}

// BIASED: the minimum pass with column energies in the biased fp32 binade (VOps<float>). Which
// minimum pass of a launch sequence runs is decided on the device by min_pass_owner.
// PRUNE: the minimum pass with block bounds (PrunedMinWalker, biased fp32 or int32 columns);
// unit minima above the group's best are then only upper bounds of the true ones (see
// PrunedMinWalker).
template <int CPT, int R, int MODE, bool BIASED = false, bool PRUNE = false>
__global__ void __launch_bounds__(CPT == 1 ? 1024 : 256, 1) search_kernel(const KParams p) {
  static_assert(!BIASED || (MODE == kModeMin && CPT >= 4), "biased walk: fast layout, minimum pass");
  static_assert(!PRUNE || (MODE == kModeMin && CPT == 16), "pruned walk: minimum pass, fast layout");
  extern __shared__ __align__(16) int4 s_rows4[];
  // linear terms of the current unit; the block-bounded pass keeps them per warp, with -L at
  // 64 + v and a zero at 128
  __shared__ int sL[PRUNE ? 1 : 64];
  __shared__ int sLw[PRUNE ? (256 / 32) * 129 : 1];
  __shared__ int s_red[32];
  // resolve modes: per-thread slots for the out-of-line candidate scan
  __shared__ __align__(16) int s_slot[(MODE != kModeMin && CPT >= 4) ? kFastThreadsMax * CPT : 4];
  if (p.hdr->status != QUBO_OK) return;
  if constexpr (MODE == kModeMin) {
    if (min_pass_owner(p) != (BIASED ? kOwnerBiased : kOwnerInt)) return;  // another pass does it
  }

  const int tid = threadIdx.x;
  const int nthreads = blockDim.x;
  const int n = p.n, C = p.C, F = p.F, w = p.w;
  const int ncols = 1 << C;
  const int ndyn = w > R ? w - R : 0;
  constexpr bool f32 = BIASED;  // staged rows in fp32 for the biased walk

  // Stage the walked rows of positions >= R (slice-independent) in shared memory.
  if constexpr (CPT >= 4) {
    const int nq = ncols >> 2;
    const int4* M4 = reinterpret_cast<const int4*>(p.M);
    for (int idx = tid; idx < ndyn * nq; idx += nthreads) {
      const int rr = idx / nq, q = idx - rr * nq;
      const int v = n - C - 1 - (R + rr);
      const int4 m = M4[(size_t)v * nq + q];
      if (f32) reinterpret_cast<float4*>(s_rows4)[idx] = make_float4((float)m.x, (float)m.y, (float)m.z, (float)m.w);
      else s_rows4[idx] = m;
    }
  } else {
    int* s_rows = reinterpret_cast<int*>(s_rows4);
    for (int idx = tid; idx < ndyn * ncols; idx += nthreads) {
      const int rr = idx >> C, j = idx & (ncols - 1);
      const int v = n - C - 1 - (R + rr);
      s_rows[idx] = p.M[(size_t)v * ncols + j];
    }
  }

  WalkCtx c{};
  c.n = n;
  c.C = C;
  c.F = F;
  c.w = w;
  c.nthreads = nthreads;
  c.thread = tid;
  c.sL = sL;
  c.rows4 = s_rows4;
  c.rows1 = reinterpret_cast<const int*>(s_rows4);
  c.T = p.T;
  c.t_global = true;
  c.theta = p.theta;
  c.rho = p.rho;
  c.cand = p.cand;
  c.cand_count = p.cand_count;
  c.cand_cap = p.cand_cap;
  c.scratch = (MODE != kModeMin && CPT >= 4) ? reinterpret_cast<uint32_t*>(s_slot) : nullptr;

  const int64_t niter = walk_iterations<R>(w);
  const int lane = tid & 31, warp = tid >> 5;

  uint64_t nitems;
  if constexpr (MODE == kModeMin) nitems = p.unit_end - p.unit_begin;
  else nitems = static_cast<uint64_t>(p.hdr->tied_count) << p.seg_bits;

  if constexpr (PRUNE) {
    // The block-bounded minimum pass. Its warps share only the staged rows, which never change,
    // so no block barrier comes between units: each warp forms the unit's linear terms itself and
    // publishes its minimum with atomics (unit_min starts at INT_MAX: block_table_kernel).
    using VT = typename std::conditional<BIASED, float, int>::type;
    __syncthreads();  // the staged rows are visible
    int* sl = sLw + warp * 129;
    c.sL = sl;
    for (uint64_t item = blockIdx.x; item < nitems; item += gridDim.x) {
      const uint64_t u = p.unit_begin + item;
      const uint64_t g = u / p.upg;
      const uint64_t P = p.gbase[g] + (u - g * p.upg);
      warp_linear_terms(p.U, n, F, P, sl, lane);
      __syncwarp();
      int cP = 0;
      for (int f = 0; f < F; ++f) cP += sl[f];
      PrunedMinWalker<R, VT> W;
      W.init(c, p.Ec, p.M, cP);
      // two blocks per iteration
      W.walk(c, static_cast<int>(niter << 1), p.blk, p.gthr + g, p.hdr->band + p.margin, p.one);
      const int best = __reduce_min_sync(0xffffffffu, W.aux - VOps<VT>::kBiasBits + W.s);
      if (lane == 0) {
        atomicMin(p.unit_min + u, best);
        atomicMin(p.gthr + g, best);
      }
      __syncwarp();  // the walk's last reads of this warp's linear terms are done
    }
  } else {
  for (uint64_t item = blockIdx.x; item < nitems; item += gridDim.x) {
    uint64_t u;
    int64_t it0 = 0, it1 = niter;
    if constexpr (MODE == kModeMin) {
      u = p.unit_begin + item;
    } else {
      u = p.tied[item >> p.seg_bits];
      const int64_t per = niter >> p.seg_bits;
      const int64_t seg = static_cast<int64_t>(item & ((uint64_t(1) << p.seg_bits) - 1));
      it0 = seg * per;
      it1 = it0 + per;
    }
    const uint64_t g = u / p.upg;
    const uint64_t P = p.gbase[g] + (u - g * p.upg);
    const uint64_t prank = (F > 0) ? (P << (n - F)) : 0;

    __syncthreads();  // previous item is done with sL; staged rows are visible
    unit_linear_terms(p.U, n, F, P, sL, tid, nthreads);
    __syncthreads();
    int cP = 0;
    for (int f = 0; f < F; ++f) cP += sL[f];

    if constexpr (MODE == kModeMin) {
      int best;
      if (niter == 0) {
        // no walked variable (generic variant only): the single walked assignment is 0
        Walker<CPT, R, MODE> W;
        W.init(c, p.Ec, p.M, cP);
        W.aux = kIntInf;
        W.step(c, prank, 0, p.T[0], p.U64, 0);
        best = W.aux + W.s;
      } else {
        best = min_walk<CPT, R, typename std::conditional<BIASED, float, int>::type>(c, p, cP, niter);
      }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) best = min(best, __shfl_xor_sync(0xffffffffu, best, off));
      if (lane == 0) s_red[warp] = best;
      __syncthreads();
      if (tid == 0) {
        int b = s_red[0];
        for (int k = 1; k < (nthreads >> 5); ++k) b = min(b, s_red[k]);
        p.unit_min[u] = b;
      }
    } else {
      Walker<CPT, R, MODE> W;
      W.init(c, p.Ec, p.M, cP);
      W.seek(c, it0);
      uint64_t gk = 0;
      if constexpr (MODE == kModeCountKey || MODE == kModeCollectKey) {
        W.aux = p.theta - W.s;
      } else {
        W.aux = p.gmin[g] + p.hdr->band - W.s;
      }
      if constexpr (MODE == kModeTiesFp) gk = p.gkey[g];
      if (niter == 0) W.step(c, prank, 0, p.T[0], p.U64, gk);
      else W.walk(c, it0, it1, it1, prank, p.U64, gk);
      uint64_t cnt = W.cnt, rmin = W.rmin, kmin = W.kmin;
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) {
        cnt += __shfl_xor_sync(0xffffffffu, cnt, off);
        const uint64_t r2 = __shfl_xor_sync(0xffffffffu, rmin, off);
        rmin = r2 < rmin ? r2 : rmin;
        const uint64_t k2 = __shfl_xor_sync(0xffffffffu, kmin, off);
        kmin = k2 < kmin ? k2 : kmin;
      }
      if (lane == 0) {
        if constexpr (MODE == kModeKeyFp) {
          if (kmin != ~0ull) atomicMin(reinterpret_cast<unsigned long long*>(&p.gkey[g]), kmin);
        } else if constexpr (MODE == kModeCountKey) {
          if (cnt) atomicAdd(p.cand_count, (unsigned long long)cnt);
        } else if constexpr (MODE == kModeCollectKey) {
          // appended one by one during the walk
        } else {
          if (cnt) {
            atomicAdd(reinterpret_cast<unsigned long long*>(&p.gties[g]), cnt);
            atomicMin(reinterpret_cast<unsigned long long*>(&p.grank[g]), rmin);
          }
        }
      }
    }
  }
  }  // not PRUNE
}

// Launch helpers (one translation unit per variant).
cudaError_t launch_search_fast(int mode, const KParams& p, int blocks, int threads, size_t smem, cudaStream_t s);
cudaError_t launch_search_biased(const KParams& p, int blocks, int threads, size_t smem, cudaStream_t s);
cudaError_t launch_search_int_min5(const KParams& p, int blocks, int threads, size_t smem, cudaStream_t s);
cudaError_t launch_search_biased_pruned(int R, const KParams& p, int blocks, int threads, size_t smem, cudaStream_t s);
cudaError_t launch_search_int_pruned(int R, const KParams& p, int blocks, int threads, size_t smem, cudaStream_t s);
cudaError_t launch_search_packed(const KParams& p, int blocks, int threads, size_t smem, cudaStream_t s);
cudaError_t launch_search_packed_pruned(int R, const KParams& p, int blocks, size_t smem, cudaStream_t s);
cudaError_t occupancy_packed_pruned(int R, size_t smem, int* blocks_per_sm);
size_t packed_pruned_smem_bytes(int C, int w, int R);
cudaError_t occupancy_packed(int threads, size_t smem, int* blocks_per_sm);
size_t packed_smem_bytes(int C, int w);

// Fold, tables and minimum pass only (w.unit_min holds every unit's minimum afterwards); kp_out
// receives the parameters for run_key_pass.
cudaError_t run_min_stage(const Plan& p, const void* d_Q, const Work& w, cudaStream_t stream, int* launches,
                          KParams* kp_out);
// One pass over the units listed in w.tied (hdr->tied_count of them, 2^seg_bits segments each)
// in mode kModeCountKey (adds to *counter the states with key (E, rank) < (theta, rho)) or
// kModeCollectKey (appends them to cand[0, cap) at index atomicAdd(counter, 1)).
cudaError_t run_key_pass(const Plan& p, const KParams& base, int mode, int theta, uint64_t rho, KeyCand* cand,
                         uint32_t cap, unsigned long long* counter, cudaStream_t stream);
cudaError_t launch_search_generic(int mode, const KParams& p, int blocks, int threads, size_t smem, cudaStream_t s);
cudaError_t occupancy_fast(int threads, size_t smem, int* blocks_per_sm);
cudaError_t occupancy_generic(int threads, size_t smem, int* blocks_per_sm);

}  // namespace qgb
