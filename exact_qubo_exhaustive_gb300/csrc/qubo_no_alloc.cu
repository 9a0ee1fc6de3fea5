// A search entry point that allocates nothing.
//
// Some callers cannot call cudaMalloc at the point where they want a result: a latency-critical
// loop for which cudaMalloc's implicit synchronisation of the whole device would be a stall, or
// a plug-in running inside a host framework that owns all device memory and hands out no
// workspace. qubo_solve_device_no_alloc() serves them: it runs the same search as
// qubo_solve_device(), but its scratch memory is the fixed array below instead of a caller
// workspace, and it never calls cudaMalloc, cudaFree or any allocating routine.
//
// The array is QUBO_NO_ALLOC_SCRATCH_BYTES (8 MiB). Every GPU that loads this library holds it
// until the process exits. Problems whose workspace is larger (n above about 46 with the default
// plan) are rejected with QUBO_ERR_ARG. All calls share the one array, and its contents persist
// from one call to the next. Nothing in it has to start at zero: the first kernel of every call
// rewrites the header (status, band, tied-unit count), and every table and accumulator after it
// is written before it is read. Two calls whose work overlaps on the GPU (two streams, or two
// host threads) race on the array; order them on one stream.
#include <mutex>

#include "qubo_internal.h"

namespace qgb {
namespace {

static __device__ __align__(256) unsigned char g_no_alloc_scratch[QUBO_NO_ALLOC_SCRATCH_BYTES];

std::mutex g_setup_mu;
void* g_scratch_ptr[64] = {nullptr};  // device address of the array, per device

// Device address of the scratch array on device `dev` (which must be current). In host code the
// array's name is only a stand-in, so the address is looked up once per device.
int scratch_address(int dev, void** out) {
  if (dev < 0 || dev >= 64) return QUBO_ERR_ARG;
  std::lock_guard<std::mutex> lk(g_setup_mu);
  if (!g_scratch_ptr[dev]) {
    void* ptr = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&ptr, g_no_alloc_scratch);
    if (e != cudaSuccess || ptr == nullptr) return record_cuda_error(e, "cudaGetSymbolAddress(scratch)");
    g_scratch_ptr[dev] = ptr;
  }
  *out = g_scratch_ptr[dev];
  return QUBO_OK;
}

}  // namespace
}  // namespace qgb

using namespace qgb;

extern "C" int qubo_solve_device_no_alloc(int n, const void* d_Q, int dtype, int k_prefix, int cache_bits,
                                          void* cuda_stream, qubo_result* d_result) {
  if (n < 1 || n > 62 || d_Q == nullptr || d_result == nullptr || !valid_dtype(dtype))
    return QUBO_ERR_ARG;
  if (k_prefix > n || cache_bits > n) return QUBO_ERR_PLAN;
  int count = 0, dev = 0;
  cudaError_t e = cudaGetDeviceCount(&count);
  if (e != cudaSuccess || count == 0) return QUBO_ERR_NODEV;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return record_cuda_error(e, "cudaGetDevice");
  Plan p;
  int st = plan_whole_problem(n, dtype, k_prefix, cache_bits, &p);
  if (st) return st;
  const size_t need = layout_workspace(p, nullptr).bytes;
  if (need > (size_t)QUBO_NO_ALLOC_SCRATCH_BYTES) return QUBO_ERR_ARG;  // beyond the fixed array
  void* base = nullptr;
  if ((st = scratch_address(dev, &base))) return st;
  Work w = layout_workspace(p, static_cast<unsigned char*>(base));
  int launches = 0;
  e = run_search(p, d_Q, w, d_result, static_cast<cudaStream_t>(cuda_stream), &launches, nullptr, nullptr, nullptr);
  record_launch_count(launches);
  if (e != cudaSuccess) return record_cuda_error(e, "kernel launch");
  return QUBO_OK;
}
