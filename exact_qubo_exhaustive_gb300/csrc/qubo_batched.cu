// Batched mode: many independent QUBO instances of equal size, one thread block per instance
// (independent subproblems, §III-C1; one problem per block). Each block folds its instance,
// builds the energy-component cache in shared memory (§II-C), walks every state with the same
// register walker as the single-problem kernel, records per-(warp, segment) minima, and then
// re-walks only the segments whose minimum equals the instance minimum to find the lowest
// rank and the tie count.
#include <cstring>

#include "qubo_walk.cuh"

namespace qgb {

namespace {
constexpr int kBatchMaxN = 25;
constexpr int kBatchSegs = 32;  // segments per instance walk

__device__ __forceinline__ int fold_entry(const int32_t* Q, int n, int i, int j, long long* u) {
  long long v = 0;
  if (j == i) v = Q[i * n + i];
  else if (j > i) v = (long long)Q[i * n + j] + (long long)Q[j * n + i];
  *u = v;
  return 0;
}

// Direct value of M[v][j] and E_cached(j) from the folded triangle in shared memory.
__device__ __forceinline__ int m_entry(const int* sU, int n, int v, int j, int C) {
  int acc = 0;
  for (int b = 0; b < C; ++b)
    if ((j >> b) & 1) acc += sU[v * n + (n - 1 - b)];
  return acc;
}
__device__ __forceinline__ int ec_entry(const int* sU, int n, int j, int C) {
  int acc = 0;
  for (int b1 = C - 1; b1 >= 0; --b1) {
    if (!((j >> b1) & 1)) continue;
    const int a = n - 1 - b1;
    for (int b2 = b1; b2 >= 0; --b2)
      if ((j >> b2) & 1) acc += sU[a * n + (n - 1 - b2)];
  }
  return acc;
}

// Running energies and register rows of thread t (columns of the fast layout), directly.
template <class W>
__device__ __forceinline__ void direct_init(W& wk, const int* sU, int n, int C, int nthreads, int t) {
  wk.s = 0;
  wk.cnt = 0;
  wk.rmin = ~0ull;
  wk.kmin = ~0ull;
  wk.valid = true;
  wk.col0 = 0;
#pragma unroll
  for (int jj = 0; jj < kFastCPT; ++jj) {
    const int j = column_of<kFastCPT>(t, nthreads, jj);
    wk.V[jj] = ec_entry(sU, n, j, C);
#pragma unroll
    for (int a = 0; a < kFastR; ++a) wk.Row[a][jj] = m_entry(sU, n, n - C - 1 - a, j, C);
  }
}

__global__ void __launch_bounds__(256, 1) batched_kernel(int n, int C, const int32_t* __restrict__ Qall,
                                                         qubo_result* __restrict__ out) {
  extern __shared__ __align__(16) int4 smem4[];
  __shared__ int sL[64];
  __shared__ int s_segmin[8 * kBatchSegs];
  __shared__ unsigned long long s_sum, s_cnt, s_rmin;
  __shared__ int s_best;
  __shared__ int s_ntied;
  __shared__ unsigned short s_tied[8 * kBatchSegs];

  const int tid = threadIdx.x, nthreads = blockDim.x;
  const int lane = tid & 31, warp = tid >> 5, nwarps = nthreads >> 5;
  const int w = n - C;
  const int ncols = 1 << C;
  const int nq = ncols >> 2;
  const int ndyn = w - kFastR;
  const int64_t niter = walk_iterations<kFastR>(w);
  const int64_t per = niter / kBatchSegs;

  // shared memory: [dyn rows: ndyn * nq int4][T: 2^w int][U: n*n int]
  int4* rows4 = smem4;
  int* sT = reinterpret_cast<int*>(rows4 + (size_t)ndyn * nq);
  int* sU = sT + (1 << w);

  const int32_t* Q = Qall + (size_t)blockIdx.x * n * n;
  if (tid == 0) {
    s_sum = 0;
    s_cnt = 0;
    s_rmin = ~0ull;
    s_ntied = 0;
  }
  if (tid < 64) sL[tid] = 0;  // no fixed variables: all linear terms are zero
  __syncthreads();
  unsigned long long local = 0;
  for (int idx = tid; idx < n * n; idx += nthreads) {
    long long u;
    fold_entry(Q, n, idx / n, idx % n, &u);
    local += (unsigned long long)(u < 0 ? -u : u);
    sU[idx] = (int)u;
  }
  atomicAdd(&s_sum, local);
  __syncthreads();
  if (s_sum > (unsigned long long)kMaxAbsSum) {
    if (tid == 0) {
      qubo_result r;
      r.status = QUBO_ERR_RANGE;
      r.reserved = 0;
      r.min_energy = 0.0;
      r.argmin_rank = 0;
      r.tie_count = 0;
      out[blockIdx.x] = r;
    }
    return;
  }
  // walked rows a >= R and the Gray-ordered walked energies
  for (int idx = tid; idx < ndyn * nq; idx += nthreads) {
    const int rr = idx / nq, q = idx - rr * nq;
    const int v = n - C - 1 - (kFastR + rr);
    int4 m;
    m.x = m_entry(sU, n, v, 4 * q + 0, C);
    m.y = m_entry(sU, n, v, 4 * q + 1, C);
    m.z = m_entry(sU, n, v, 4 * q + 2, C);
    m.w = m_entry(sU, n, v, 4 * q + 3, C);
    rows4[idx] = m;
  }
  for (int i = tid; i < (1 << w); i += nthreads) {
    const unsigned g = (unsigned)(i ^ (i >> 1));
    int acc = 0;
    for (int a = 0; a < w; ++a) {
      if (!((g >> a) & 1u)) continue;
      const int va = n - C - 1 - a;
      for (int b = a; b < w; ++b)
        if ((g >> b) & 1u) acc += sU[(n - C - 1 - b) * n + va];
    }
    sT[i] = acc;
  }
  __syncthreads();

  WalkCtx c;
  c.n = n;
  c.C = C;
  c.F = 0;
  c.w = w;
  c.nthreads = nthreads;
  c.thread = tid;
  c.sL = sL;
  c.rows4 = rows4;
  c.rows1 = nullptr;
  c.T = sT;
  c.t_global = false;

  // ---- minimum pass, one segment at a time (the walk continues across segments)
  {
    Walker<kFastCPT, kFastR, kModeMin> W;
    direct_init(W, sU, n, C, nthreads, tid);
    for (int seg = 0; seg < kBatchSegs; ++seg) {
      W.aux = kIntInf;
      W.walk(c, seg * per, (seg + 1) * per, niter, 0, nullptr, 0);
      int best = W.aux + W.s;
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) best = min(best, __shfl_xor_sync(0xffffffffu, best, off));
      if (lane == 0) s_segmin[warp * kBatchSegs + seg] = best;
    }
  }
  __syncthreads();
  if (tid == 0) {
    int b = kIntInf;
    for (int k = 0; k < nwarps * kBatchSegs; ++k) b = min(b, s_segmin[k]);
    s_best = b;
    int nt = 0;
    for (int k = 0; k < nwarps * kBatchSegs; ++k)
      if (s_segmin[k] == b) s_tied[nt++] = (unsigned short)k;
    s_ntied = nt;
  }
  __syncthreads();
  const int best = s_best;

  // ---- resolve: each tied (warp, segment) pair, split into its iterations, spread over warps
  {
    const int nitems = s_ntied * (int)per;
    for (int item = warp; item < nitems; item += nwarps) {
      const int pair = s_tied[item / (int)per];
      const int tw = pair / kBatchSegs, seg = pair % kBatchSegs;
      const int64_t it0 = seg * per + (item % (int)per);
      WalkCtx cw = c;
      cw.thread = tw * 32 + lane;  // emulate the columns of warp tw
      Walker<kFastCPT, kFastR, kModeTiesInt> W;
      direct_init(W, sU, n, C, nthreads, cw.thread);
      W.seek(cw, it0);
      W.aux = best - W.s;
      W.walk(cw, it0, it0 + 1, it0 + 1, 0, nullptr, 0);
      uint64_t cnt = W.cnt, rmin = W.rmin;
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) {
        cnt += __shfl_xor_sync(0xffffffffu, cnt, off);
        const uint64_t r2 = __shfl_xor_sync(0xffffffffu, rmin, off);
        rmin = r2 < rmin ? r2 : rmin;
      }
      if (lane == 0 && cnt) {
        atomicAdd(&s_cnt, (unsigned long long)cnt);
        atomicMin(&s_rmin, (unsigned long long)rmin);
      }
    }
  }
  __syncthreads();
  if (tid == 0) {
    qubo_result r;
    r.status = QUBO_OK;
    r.reserved = 0;
    r.min_energy = (double)best;
    r.argmin_rank = s_rmin;
    r.tie_count = s_cnt;
    out[blockIdx.x] = r;
  }
}
}  // namespace

bool plan_batched(int batch, int n, BatchPlan* bp) {
  if (batch < 1 || n < 14 || n > kBatchMaxN) return false;
  // cache bits: 2^C columns = threads * 16; walked w = n - C needs w >= R + 1 + log2(segments)
  int C = n >= 24 ? 11 : n - (kFastR + 1 + 5);
  if (C > 12) C = 12;
  if (C < 9) C = 9;
  const int w = n - C;
  if (w < kFastR + 1 + 5) return false;  // at least one iteration per segment
  bp->batch = batch;
  bp->n = n;
  bp->C = C;
  bp->w = w;
  bp->threads = (1 << C) / kFastCPT;
  bp->smem_bytes = ((size_t)(w - kFastR) << (C + 2)) + ((size_t)1 << (w + 2)) + (size_t)n * n * 4;
  const DevInfo& di = device_info();
  if (bp->smem_bytes + 4096 > di.smem_optin) return false;
  return true;
}

size_t batched_workspace_bytes(const BatchPlan& bp) { return 256; }

cudaError_t run_batched(const BatchPlan& bp, const void* d_Q, void* d_ws, qubo_result* res, cudaStream_t stream,
                        int* launches) {
  (void)d_ws;
  cudaError_t e = cudaFuncSetAttribute(batched_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bp.smem_bytes);
  if (e != cudaSuccess) return e;
  batched_kernel<<<bp.batch, bp.threads, bp.smem_bytes, stream>>>(bp.n, bp.C, static_cast<const int32_t*>(d_Q), res);
  if (launches) *launches = 1;
  return cudaGetLastError();
}

}  // namespace qgb
