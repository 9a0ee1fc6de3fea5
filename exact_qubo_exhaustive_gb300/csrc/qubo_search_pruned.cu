// Minimum passes with block bounds (biased fp32 binade and int32), 16 columns per thread and the
// kFastR lowest walked rows in registers: blocks of 2^kFastR steps whose lower bound is above the
// group's best skip their per-step minima (PrunedMinWalker).
#include "qubo_search_kernel.cuh"

namespace qgb {

template <bool BIASED>
static cudaError_t launch_one(const KParams& p, int blocks, int threads, size_t smem, cudaStream_t s) {
  auto k = search_kernel<kFastCPT, kFastR, kModeMin, BIASED, true>;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  k<<<blocks, threads, smem, s>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_search_pruned(bool biased, const KParams& p, int blocks, int threads, size_t smem, cudaStream_t s) {
  return biased ? launch_one<true>(p, blocks, threads, smem, s) : launch_one<false>(p, blocks, threads, smem, s);
}

}  // namespace qgb
