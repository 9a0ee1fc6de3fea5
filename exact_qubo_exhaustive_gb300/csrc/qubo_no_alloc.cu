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
//
// The array's device address belongs to the CUDA context the module was loaded into. It is
// looked up (cudaGetSymbolAddress) on the first call in a context and kept together with that
// context's unique id; a call from another context (after cudaDeviceReset, or under a context the
// caller created with the driver API) looks it up again. Make the first call in each context
// before any stream capture.
#include <cuda.h>

#include <mutex>

#include "qubo_internal.h"

namespace qgb {
namespace {

static __device__ __align__(256) unsigned char g_no_alloc_scratch[QUBO_NO_ALLOC_SCRATCH_BYTES];

using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);

struct ScratchSlot {
  unsigned long long ctx_id = 0;  // id of the context the address belongs to (0: none yet)
  void* ptr = nullptr;
};

std::mutex g_setup_mu;
ScratchSlot g_slot[64];  // per device
CtxGetCurrentFn g_ctx_get_current = nullptr;
CtxGetIdFn g_ctx_get_id = nullptr;

// The driver's context queries, through the runtime (no link-time dependency on the driver).
int driver_entry_points() {
  if (g_ctx_get_current && g_ctx_get_id) return QUBO_OK;
  void* f1 = nullptr;
  void* f2 = nullptr;
  cudaDriverEntryPointQueryResult q1 = cudaDriverEntryPointSymbolNotFound, q2 = cudaDriverEntryPointSymbolNotFound;
  cudaError_t e = cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f1, 12000, cudaEnableDefault, &q1);
  if (e != cudaSuccess || q1 != cudaDriverEntryPointSuccess || !f1)
    return record_cuda_error(e != cudaSuccess ? e : cudaErrorSymbolNotFound, "driver entry point cuCtxGetCurrent");
  e = cudaGetDriverEntryPointByVersion("cuCtxGetId", &f2, 12000, cudaEnableDefault, &q2);
  if (e != cudaSuccess || q2 != cudaDriverEntryPointSuccess || !f2)
    return record_cuda_error(e != cudaSuccess ? e : cudaErrorSymbolNotFound, "driver entry point cuCtxGetId");
  g_ctx_get_current = reinterpret_cast<CtxGetCurrentFn>(f1);
  g_ctx_get_id = reinterpret_cast<CtxGetIdFn>(f2);
  return QUBO_OK;
}

// Unique id of the calling thread's current context; 0 when none is current yet.
int current_context_id(unsigned long long* id) {
  *id = 0;
  CUcontext ctx = nullptr;
  if (g_ctx_get_current(&ctx) != CUDA_SUCCESS) return record_cuda_error(cudaErrorContextIsDestroyed, "cuCtxGetCurrent");
  if (ctx && g_ctx_get_id(ctx, id) != CUDA_SUCCESS) return record_cuda_error(cudaErrorContextIsDestroyed, "cuCtxGetId");
  return QUBO_OK;
}

// Device address of the scratch array in the current context of device `dev` (which must be
// current). In host code the array's name is only a stand-in, so the address is looked up with
// cudaGetSymbolAddress once per context.
int scratch_address(int dev, void** out) {
  if (dev < 0 || dev >= 64) return QUBO_ERR_ARG;
  std::lock_guard<std::mutex> lk(g_setup_mu);
  int st = driver_entry_points();
  if (st) return st;
  unsigned long long id = 0;
  if ((st = current_context_id(&id))) return st;
  ScratchSlot& s = g_slot[dev];
  if (id == 0 || s.ctx_id != id || !s.ptr) {
    void* ptr = nullptr;
    // With no context current yet, this call initialises the device's primary context.
    cudaError_t e = cudaGetSymbolAddress(&ptr, g_no_alloc_scratch);
    if (e != cudaSuccess || ptr == nullptr)
      return record_cuda_error(e != cudaSuccess ? e : cudaErrorInvalidSymbol, "cudaGetSymbolAddress(scratch)");
    if (id == 0 && (st = current_context_id(&id))) return st;
    s.ctx_id = id;
    s.ptr = ptr;
  }
  *out = s.ptr;
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
  if (abort_requested()) return QUBO_ERR_ABORTED;
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
