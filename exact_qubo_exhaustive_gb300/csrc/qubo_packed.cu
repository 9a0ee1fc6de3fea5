// Packed narrow minimum pass: the kernel around the packed walker (qubo_packed_walk.cuh) for
// int32 input with sum |U| <= kPackedMaxAbsSum (Terastate-per-second QUBO Brute-Force on a Single
// GPU, §IV-B.5): staging of the packed shared rows, the persistent loop over work units and the
// block reduction of each unit's minimum.
#include "qubo_packed_walk.cuh"
#include "qubo_search_kernel.cuh"

namespace qgb {
namespace {
using packed::combine;
using packed::PackedPrunedWalker;
using packed::PackedWalker;

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
    W.init(c, p.Ec, packed::GlobalRows{p.M, 1 << C}, cP);
    int best = W.walk(c, 0, niter);
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

// The packed pass with block bounds (PackedPrunedWalker): the same staging and unit loop, the
// block control table of the bounded passes, and each unit's minimum published to its group.
template <int R>
__global__ void __launch_bounds__(128, 2) packed_pruned_kernel(const KParams p) {
  extern __shared__ __align__(16) int4 s_rows4[];
  __shared__ int sL[129];  // L, -L at 64 + v and a zero at 128
  __shared__ int s_red[32];
  __shared__ uint4 s_dw[4 * PackedPrunedWalker<R>::kThreads];  // per-column changes (block bound)
  if (p.hdr->status != QUBO_OK) return;
  if (min_pass_owner(p) != kOwnerPacked) return;

  const int tid = threadIdx.x;
  const int nthreads = blockDim.x;
  const int n = p.n, C = p.C, F = p.F, w = p.w;
  const int ncols = 1 << C;
  const int nwords = ncols >> 1;
  const int ndyn = w - R;

  uint32_t* s_words = reinterpret_cast<uint32_t*>(s_rows4);
  for (int idx = tid; idx < ndyn * nwords; idx += nthreads) {
    const int rr = idx >> (C - 1), q = idx & (nwords - 1);
    const int v = n - C - 1 - (R + rr);
    const int2 m = reinterpret_cast<const int2*>(p.M + (size_t)v * ncols)[q];
    s_words[idx] = combine(m.x, m.y);
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
  c.rows1 = nullptr;
  c.T = reinterpret_cast<const int*>(p.T2);
  c.t_global = true;

  const int nblocks = 1 << (w - R);
  const int lane = tid & 31, warp = tid >> 5;
  const uint64_t nitems = p.unit_end - p.unit_begin;
  for (uint64_t item = blockIdx.x; item < nitems; item += gridDim.x) {
    const uint64_t u = p.unit_begin + item;
    const uint64_t g = u / p.upg;
    const uint64_t P = p.gbase[g] + (u - g * p.upg);
    __syncthreads();  // previous item is done with sL; staged rows are visible
    unit_linear_terms(p.U, n, F, P, sL, tid, nthreads);
    __syncthreads();
    for (int v = tid; v <= 64; v += nthreads) sL[64 + v] = v < n ? -sL[v] : 0;
    __syncthreads();
    int cP = 0;
    for (int f = 0; f < F; ++f) cP += sL[f];
    PackedPrunedWalker<R> W;
    W.init(c, p.Ec, packed::GlobalRows{p.M, 1 << C}, cP);
    int best = W.walk(c, nblocks, p.blk, p.T2, p.gthr + g, p.hdr->band + p.margin, p.one, nullptr, s_dw);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) best = min(best, __shfl_xor_sync(0xffffffffu, best, off));
    if (lane == 0) s_red[warp] = best;
    __syncthreads();
    if (tid == 0) {
      int b = s_red[0];
      for (int k = 1; k < (nthreads >> 5); ++k) b = min(b, s_red[k]);
      p.unit_min[u] = b;
      atomicMin(p.gthr + g, b);
    }
  }
}

template <int R>
cudaError_t launch_pruned(const KParams& p, int blocks, size_t smem, cudaStream_t s) {
  auto k = packed_pruned_kernel<R>;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  k<<<blocks, PackedPrunedWalker<R>::kThreads, smem, s>>>(p);
  return cudaGetLastError();
}

template <int R>
cudaError_t occupancy_pruned(size_t smem, int* blocks_per_sm) {
  auto k = packed_pruned_kernel<R>;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  return cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks_per_sm, k, PackedPrunedWalker<R>::kThreads, smem);
}

}  // namespace

size_t packed_smem_bytes(int C, int w) { return (size_t)(w - kPackedR) << (C + 1); }

size_t packed_pruned_smem_bytes(int C, int w, int R) { return (size_t)(w - R) << (C + 1); }

cudaError_t launch_search_packed_pruned(int R, const KParams& p, int blocks, size_t smem, cudaStream_t s) {
  if (p.C != 12) return cudaErrorInvalidConfiguration;  // 128 threads x 32 columns
  if (R == kPruneRLong) return launch_pruned<kPruneRLong>(p, blocks, smem, s);
  if (R == kPruneRShort) return launch_pruned<kPruneRShort>(p, blocks, smem, s);
  return cudaErrorInvalidValue;
}

cudaError_t occupancy_packed_pruned(int R, size_t smem, int* blocks_per_sm) {
  if (R == kPruneRLong) return occupancy_pruned<kPruneRLong>(smem, blocks_per_sm);
  if (R == kPruneRShort) return occupancy_pruned<kPruneRShort>(smem, blocks_per_sm);
  return cudaErrorInvalidValue;
}

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
