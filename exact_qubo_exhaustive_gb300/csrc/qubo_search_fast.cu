// Register-cached enumeration kernel: 16 columns per thread, the lowest walked rows in
// registers (5 for the minimum passes, 4 for the resolution passes), the other walked rows in
// shared memory.
#include "qubo_search_kernel.cuh"

namespace qgb {

template <int MODE>
static cudaError_t launch_one(const KParams& p, int blocks, int threads, size_t smem, cudaStream_t s) {
  auto k = search_kernel<kFastCPT, kFastR, MODE>;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  k<<<blocks, threads, smem, s>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_search_fast(int mode, const KParams& p, int blocks, int threads, size_t smem, cudaStream_t s) {
  switch (mode) {
    case kModeMin: return launch_one<kModeMin>(p, blocks, threads, smem, s);
    case kModeTiesInt: return launch_one<kModeTiesInt>(p, blocks, threads, smem, s);
    case kModeKeyFp: return launch_one<kModeKeyFp>(p, blocks, threads, smem, s);
    case kModeTiesFp: return launch_one<kModeTiesFp>(p, blocks, threads, smem, s);
    case kModeCountKey: return launch_one<kModeCountKey>(p, blocks, threads, smem, s);
    case kModeCollectKey: return launch_one<kModeCollectKey>(p, blocks, threads, smem, s);
  }
  return cudaErrorInvalidValue;
}

cudaError_t launch_search_biased(const KParams& p, int blocks, int threads, size_t smem, cudaStream_t s) {
  auto k = search_kernel<kFastCPT, kBiasedR, kModeMin, true>;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  k<<<blocks, threads, smem, s>>>(p);
  return cudaGetLastError();
}

// int32 minimum pass with five register rows (needs at least 2^6 walked steps per unit).
cudaError_t launch_search_int_min5(const KParams& p, int blocks, int threads, size_t smem, cudaStream_t s) {
  auto k = search_kernel<kFastCPT, kIntMinR, kModeMin, false>;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  k<<<blocks, threads, smem, s>>>(p);
  return cudaGetLastError();
}

cudaError_t occupancy_fast(int threads, size_t smem, int* blocks_per_sm) {
  auto k = search_kernel<kFastCPT, kFastR, kModeMin>;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  return cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks_per_sm, k, threads, smem);
}

}  // namespace qgb
