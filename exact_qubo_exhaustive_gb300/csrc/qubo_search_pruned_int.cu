// int32 minimum pass with block bounds, for int32 input whose sum |U_ij| is too large for the
// fp32 binade: 16 columns per thread, 256 threads (2^12 cached columns), the R lowest walked rows
// in registers (R = kPruneRShort or kPruneRLong, as planned); blocks of 2^R steps whose lower
// bound is above the group's best skip their per-step minima (PrunedMinWalker<R, int>: every
// state is still added, by a fused add-min or a multiply-add the compiler cannot fold).
#include "qubo_search_kernel.cuh"

namespace qgb {

template <int R>
static cudaError_t launch_one(const KParams& p, int blocks, int threads, size_t smem, cudaStream_t s) {
  if (threads != PrunedMinWalker<R, int>::kThreads) return cudaErrorInvalidConfiguration;
  auto k = search_kernel<kFastCPT, R, kModeMin, false, true>;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  k<<<blocks, threads, smem, s>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_search_int_pruned(int R, const KParams& p, int blocks, int threads, size_t smem, cudaStream_t s) {
  if (R == kPruneRLong) return launch_one<kPruneRLong>(p, blocks, threads, smem, s);
  if (R == kPruneRShort) return launch_one<kPruneRShort>(p, blocks, threads, smem, s);
  return cudaErrorInvalidValue;
}

}  // namespace qgb
