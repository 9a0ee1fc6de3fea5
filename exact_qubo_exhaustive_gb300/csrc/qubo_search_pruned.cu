// Biased-binade minimum pass with block bounds: 16 columns per thread, 256 threads (2^12 cached
// columns), the kPruneR lowest walked rows in registers; blocks of 2^kPruneR steps whose lower
// bound is above the group's best skip their per-step minima (PrunedMinWalker).
#include "qubo_search_kernel.cuh"

namespace qgb {

cudaError_t launch_search_biased_pruned(const KParams& p, int blocks, int threads, size_t smem, cudaStream_t s) {
  if (threads != PrunedMinWalker<kPruneR>::kThreads) return cudaErrorInvalidConfiguration;
  auto k = search_kernel<kFastCPT, kPruneR, kModeMin, true, true>;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  k<<<blocks, threads, smem, s>>>(p);
  return cudaGetLastError();
}

}  // namespace qgb
