// Tensor-core minimum pass (sm_103a, tcgen05 + tensor memory).
//
// The chunk energies of the prefix-suffix decomposition are a matrix product
// (Terastate-per-second QUBO Brute-Force on a Single GPU, §II-C eq. 8):
//     E(C_xp) = E_p(x_p) 1 + x_p M_int + E_s(U_B).
// Here one tcgen05.mma computes that product for a 128 x 256 tile of states at once:
//   rows    = the 128 assignments of the 7 lowest walked variables (the MMA's M),
//   columns = the 256 assignments of the 8 cached variables (the MMA's N),
//   K = 16  = 7 row variables x 2 pieces + 1 bias x 2 pieces.
// Every integer operand v is split into f16-exact pieces v = lo + 2048 hi (lo in [-1024, 1023],
// |hi| <= 2048); A carries the row bits as x and 2048 x, so the fp32 accumulator receives
//     D[r][j] = sum_a x_a(r) M_int[a][j] + V[j]
// exactly (every partial sum is an integer below 2^23 when sum |U_ij| <= 2^21). V[j] (the
// cached self energy, the unit's linear terms and the interaction with the remaining walked
// variables) is the bias row; the remaining walked variables are visited in Gray order (§III-B,
// eq. 9), so each step adds one row of M_int to V on the CUDA cores and issues one MMA.
// The accumulator lives in tensor memory (two buffers: the tensor core fills one while the CUDA
// cores reduce the other with 3-input integer minima on the accumulator bits, which the bias
// offset kTcOffset keeps non-negative: half an ALU instruction per state); the
// walked self energy of each row, in Gray order (§IV-B.3), is added once per row after the
// column minimum.
#include <cuda_fp16.h>

#include "qubo_search_kernel.cuh"
#include "qubo_tc.cuh"

namespace qgb {

namespace {
constexpr uint32_t kTmemCols = 512;            // two 128 x 256 fp32 accumulators
// Added to every column bias: with sum |U| <= 2^21 every accumulator value D = (partial energy)
// + 2^21 lies in [0, 2^22], a non-negative float whose bit pattern orders like its value, so the
// column minimum runs as 3-input integer minima on the raw accumulator bits.
constexpr int kTcOffset = 1 << 21;
static_assert(kTcMaxAbsSum <= kTcOffset, "accumulators must stay non-negative");
constexpr uint32_t kIdesc = tc::idesc_f16_f32(128, 256);
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s: an MMA takes ~0.1 us

// The same split for an fp32 value holding an integer |v| <= 2^22 (exact): round(v / 2048)
// by the 1.5 * 2^23 rounding constant, then lo = v - 2048 hi exactly; one packing conversion.
__device__ __forceinline__ uint32_t pack_pieces_f(float v) {
  const float hi = __fadd_rn(__fmaf_rn(v, 1.0f / 2048.0f, 12582912.0f), -12582912.0f);
  const float lo = __fmaf_rn(-2048.0f, hi, v);
  const __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}

__device__ __forceinline__ uint32_t pack_pieces(int v) {
  const int hi = (v + 1024) >> 11;  // arithmetic shift: round to nearest multiple of 2048
  const int lo = v - hi * 2048;     // in [-1024, 1023]
  const __half2 h = __halves2half2(__int2half_rn(lo), __int2half_rn(hi));
  return *reinterpret_cast<const uint32_t*>(&h);
}
}  // namespace

// ------------------------------------------------------------------------------------------------
// Tables of the tensor-core split (cached C = 8, row bits 7, walked w8 = n - F - 8):
//   M8[v][j] = sum_{cached b} U[v][b] x_b(j), v < n - 8      (M_int rows)
//   E8[j]    = cached self energy                            (E(U_B))
//   T8[i * 128 + r] = walked self energy at walked assignment (gray(i) << 7) | r
// Walked position a drives variable n - 9 - a.
// ------------------------------------------------------------------------------------------------
__global__ void tc_tables_kernel(int n, int w8, const DevHeader* __restrict__ hdr, const int32_t* __restrict__ U,
                                 int32_t* M8, int32_t* E8, int32_t* T8) {
  if (hdr->status != QUBO_OK || hdr->abs_sum > kTcMaxAbsSum) return;
  const uint64_t nM = (uint64_t)(n - kTcC) << kTcC;
  const uint64_t nE = 1u << kTcC;
  const uint64_t nT = (uint64_t)1 << w8;
  const uint64_t total = nM + nE + nT;
  for (uint64_t idx = blockIdx.x * (uint64_t)blockDim.x + threadIdx.x; idx < total;
       idx += (uint64_t)gridDim.x * blockDim.x) {
    if (idx < nM) {
      const int v = (int)(idx >> kTcC), j = (int)(idx & 255);
      int acc = 0;
      for (int b = 0; b < kTcC; ++b)
        if ((j >> b) & 1) acc += U[v * n + (n - 1 - b)];
      M8[idx] = acc;
    } else if (idx < nM + nE) {
      const int j = (int)(idx - nM);
      int acc = 0;
      for (int b1 = kTcC - 1; b1 >= 0; --b1) {
        if (!((j >> b1) & 1)) continue;
        const int a = n - 1 - b1;
        for (int b2 = b1; b2 >= 0; --b2)
          if ((j >> b2) & 1) acc += U[a * n + (n - 1 - b2)];
      }
      E8[j] = acc;
    } else {
      const uint64_t t = idx - nM - nE;
      const uint64_t i = t >> 7, r = t & 127;
      const uint64_t gw = ((i ^ (i >> 1)) << 7) | r;
      int acc = 0;
      for (int a = 0; a < w8; ++a) {
        if (!((gw >> a) & 1u)) continue;
        const int va = n - kTcC - 1 - a;
        for (int b = a; b < w8; ++b)
          if ((gw >> b) & 1u) acc += U[(n - kTcC - 1 - b) * n + va];
      }
      T8[t] = acc;
    }
  }
}

// ------------------------------------------------------------------------------------------------
// Minimum pass: persistent grid over units (fixed prefixes, §III-C1), one block per SM, 8 warps,
// two per SM sub-partition. Thread t owns column t of the bias row and accumulator row
// 32 (w % 4) + lane over columns 128 (w / 4) .. +127 (warp w reads its sub-partition's
// tensor-memory lanes). Per tile i every warp waits for "full i", loads its 128 accumulator
// values and signals "empty i"; lane 0 of warp 1 (the issuer) then waits until every warp has
// done so and issues the MMA of tile i + 2 into that accumulator, before its own reduction. After
// reducing, each thread writes its bias of tile i + 3 into the B buffer the MMA of tile i has
// released (three B buffers, two accumulators). All waits spin on the mbarrier phase (a suspended
// waiter resumes late) and are bounded in time.
// ------------------------------------------------------------------------------------------------
namespace {
constexpr int kWarps = 8;
constexpr int kBlock = kWarps * 32;
constexpr int kIssuerWarp = 1;
}  // namespace

__global__ void __launch_bounds__(kBlock, 1) tc_min_kernel(const KParams p, int w8, const int32_t* __restrict__ M8,
                                                             const int32_t* __restrict__ E8,
                                                             const int32_t* __restrict__ T8) {
  extern __shared__ __align__(1024) unsigned char smem[];
  __shared__ int sL[64];
  __shared__ int s_red[kWarps];
  __shared__ __align__(8) uint64_t s_full[2];
  __shared__ __align__(8) uint64_t s_empty[2];
  __shared__ uint32_t s_tmem;
  __shared__ volatile int s_abort;

  if (p.hdr->status != QUBO_OK || p.hdr->abs_sum > kTcMaxAbsSum) return;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int n = p.n, F = p.F;
  const int nh = w8 - kTcRowBits;  // Gray-walked (high) variables
  unsigned char* sA = smem;
  unsigned char* sBb = smem + 4096;                               // three 8 KB B buffers
  float* sMh = reinterpret_cast<float*>(smem + 4096 + 3 * 8192);  // [nh][256], exact integers

  // ---- once per block: A (row bits and bias in pieces), the constant rows of B, the walked rows
  for (int idx = tid; idx < 128 * 16; idx += kBlock) {
    const int r = idx >> 4, k = idx & 15, a = k >> 1;
    const int x = (a < kTcRowBits) ? ((r >> a) & 1) : 1;
    const __half h = __float2half_rn((k & 1) ? 2048.0f * x : (float)x);
    *reinterpret_cast<__half*>(sA + tc::operand_offset(r, k)) = h;
  }
  for (int idx = tid; idx < 256 * kTcRowBits; idx += kBlock) {
    const int j = idx & 255, a = idx >> 8;
    const int v = n - kTcC - 1 - a;
    const uint32_t pk = pack_pieces(M8[(size_t)v * 256 + j]);
#pragma unroll
    for (int b = 0; b < 3; ++b) *reinterpret_cast<uint32_t*>(sBb + b * 8192 + tc::operand_offset(j, 2 * a)) = pk;
  }
  for (int idx = tid; idx < nh * 256; idx += kBlock) {
    const int h = idx >> 8, j = idx & 255;
    sMh[idx] = (float)M8[(size_t)(n - kTcC - 1 - (kTcRowBits + h)) * 256 + j];
  }
  if (warp == 0) tc::tmem_alloc(tc::smem_addr(&s_tmem), kTmemCols);
  if (tid == 0) {
    tc::mbar_init(tc::smem_addr(&s_full[0]), 1);
    tc::mbar_init(tc::smem_addr(&s_full[1]), 1);
    tc::mbar_init(tc::smem_addr(&s_empty[0]), kWarps);
    tc::mbar_init(tc::smem_addr(&s_empty[1]), kWarps);
    tc::fence_mbar_init();
    s_abort = 0;
  }
  tc::fence_async_smem();
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = s_tmem;
  const uint64_t descA = tc::smem_desc(tc::smem_addr(sA));
  const uint32_t sB_addr = tc::smem_addr(sBb);
  const uint32_t full0 = tc::smem_addr(&s_full[0]), full1 = tc::smem_addr(&s_full[1]);
  const uint32_t empty0 = tc::smem_addr(&s_empty[0]), empty1 = tc::smem_addr(&s_empty[1]);
  const bool is_issuer = (warp == kIssuerWarp && lane == 0);

  const int col = tid;  // bias column
  const int quarter = warp & 3, colhalf = warp >> 2;
  const int row = 32 * quarter + lane;
  const uint32_t tl = (uint32_t)(32 * quarter) << 16;
  const int64_t ntiles = (int64_t)1 << nh;
  uint64_t gtile = 0;
  uint32_t gslot = 0;  // gtile mod 3: the B buffer of the unit's first tile
  int failed = 0;

  auto issue = [&](uint64_t gt, uint32_t bslot) {
    tc::mma_f16(tmem + (uint32_t)(gt & 1) * 256u, descA, tc::smem_desc(sB_addr + bslot * 8192u), kIdesc, 0);
    tc::mma_commit((gt & 1) ? full1 : full0);
  };
  // Bias of step i + 1 from step i: Gray flip of high variable ctz(i + 1).
  auto flip = [&](float v, int64_t i) {
    const int h = __ffsll((long long)(i + 1)) - 1;
    const uint64_t gi = (uint64_t)i ^ ((uint64_t)i >> 1);
    const float mv = sMh[h * 256 + col];
    return ((gi >> h) & 1u) ? __fadd_rn(v, -mv) : __fadd_rn(v, mv);
  };

  for (uint64_t u = p.unit_begin + blockIdx.x; u < p.unit_end; u += gridDim.x) {
    const uint64_t g = u / p.upg;
    const uint64_t P = p.gbase[g] + (u - g * p.upg);
    __syncthreads();  // the previous unit is finished by every warp
    unit_linear_terms(p.U, n, F, P, sL, tid, (int)blockDim.x);
    __syncthreads();
    int s = 0;
    for (int f = 0; f < F; ++f) s += sL[f];
    int Lrow = 0;
#pragma unroll
    for (int a = 0; a < kTcRowBits; ++a)
      if ((row >> a) & 1) Lrow += sL[n - kTcC - 1 - a];
    // bias of steps 0, 1, 2 into their B buffers
    int v0 = E8[col];
#pragma unroll
    for (int b = 0; b < kTcC; ++b)
      if ((col >> b) & 1) v0 += sL[n - 1 - b];
    float Vn = (float)(v0 + kTcOffset);
    {
      uint32_t slot = gslot;
      for (int64_t i = 0; i < 3 && i < ntiles; ++i) {
        if (i > 0) Vn = flip(Vn, i - 1);
        *reinterpret_cast<uint32_t*>(sBb + slot * 8192 + tc::operand_offset(col, 14)) = pack_pieces_f(Vn);
        slot = (slot == 2) ? 0 : slot + 1;
      }
    }
    tc::fence_async_smem();
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    if (is_issuer) {
      issue(gtile, gslot);
      if (ntiles > 1) issue(gtile + 1, gslot == 2 ? 0 : gslot + 1);
    }

    int best = kIntInf;
    int t_cur = __ldg(&T8[row]);
    uint32_t slot = gslot;  // B buffer of tile i; tile i + 2 uses slot + 2, tile i + 3 reuses slot
    for (int64_t i = 0; i < ntiles; ++i) {
      const uint64_t gt = gtile + (uint64_t)i;
      const int buf = (int)(gt & 1);
      const int t_next = (i + 1 < ntiles) ? __ldg(&T8[(size_t)(i + 1) * 128 + row]) : 0;
      const bool ok = tc::mbar_spin(buf ? full1 : full0, (uint32_t)((gt >> 1) & 1), kWaitLimitNs, &s_abort);
      if (!__all_sync(0xffffffffu, ok)) {
        failed = 1;
        s_abort = 1;
        break;
      }
      tc::fence_after_sync();
      uint32_t v[128];
      tc::tmem_load128(tmem + tl + (uint32_t)buf * 256u + 128u * (uint32_t)colhalf, v);
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(buf ? empty1 : empty0);
      if (is_issuer && i + 2 < ntiles) {
        // every warp has read tile i out of this accumulator: refill it with tile i + 2
        if (tc::mbar_spin(buf ? empty1 : empty0, (uint32_t)((gt >> 1) & 1), kWaitLimitNs, &s_abort)) {
          tc::fence_after_sync();
          issue(gt + 2, slot == 0 ? 2 : slot - 1);
        } else {
          failed = 1;
          s_abort = 1;
        }
      }
      __syncwarp();
      // 3-input integer minima on the bit patterns (non-negative floats below 2^31 as integers
      // order like their values): 8 independent chains, chain k over v[k + 8 j], j = 0..15, in
      // 7 three-input and 1 two-input minima; about one ALU instruction per two states
      int m[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        int a = __vimin3_s32((int)v[k], (int)v[k + 8], (int)v[k + 16]);
#pragma unroll
        for (int j = 3; j < 15; j += 2) a = __vimin3_s32(a, (int)v[k + 8 * j], (int)v[k + 8 * j + 8]);
        m[k] = min(a, (int)v[k + 120]);
      }
      const int mb = min(__vimin3_s32(m[0], m[1], m[2]), __vimin3_s32(m[3], m[4], __vimin3_s32(m[5], m[6], m[7])));
      const int rmin = __float2int_rn(__int_as_float(mb)) - kTcOffset;
      best = min(best, rmin + t_cur + Lrow + s);
      if (i + 1 < ntiles) {  // offset of the next tile: its Gray flip's linear term
        const int h = __ffsll((long long)(i + 1)) - 1;
        const uint64_t gi = (uint64_t)i ^ ((uint64_t)i >> 1);
        const int lv = sL[n - kTcC - 1 - (kTcRowBits + h)];
        s += ((gi >> h) & 1u) ? -lv : lv;
      }
      if (i + 3 < ntiles) {  // bias of step i + 3 into the B buffer the MMA of tile i released
        Vn = flip(Vn, i + 2);
        *reinterpret_cast<uint32_t*>(sBb + slot * 8192 + tc::operand_offset(col, 14)) = pack_pieces_f(Vn);
        tc::fence_async_smem();
      }
      slot = (slot == 2) ? 0 : slot + 1;
      t_cur = t_next;
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) best = min(best, __shfl_xor_sync(0xffffffffu, best, off));
    if (lane == 0) s_red[warp] = best;
    gtile += (uint64_t)ntiles;
    gslot = (uint32_t)((gslot + (uint64_t)ntiles) % 3);
    tc::fence_before_sync();
    failed = __syncthreads_or(failed);
    tc::fence_after_sync();
    if (failed) break;
    if (tid == 0) {
      int b = s_red[0];
      for (int k = 1; k < kWarps; ++k) b = min(b, s_red[k]);
      p.unit_min[u] = b;
    }
  }
  if (failed && tid == 0) atomicExch(&p.hdr->status, QUBO_ERR_CUDA);
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 0) tc::tmem_dealloc(tmem, kTmemCols);
}

size_t tc_smem_bytes(int w8) {
  const size_t used = 4096 + 3 * 8192 + ((size_t)(w8 - kTcRowBits) << 10);
  // at least 120 KB: one block per SM, so the block owns all 512 tensor-memory columns
  return used < (size_t)120 * 1024 ? (size_t)120 * 1024 : used;
}

cudaError_t launch_tc_search(const KParams& p, int w8, const int32_t* M8, const int32_t* E8, const int32_t* T8,
                             int blocks, cudaStream_t s) {
  const size_t smem = tc_smem_bytes(w8);
  cudaError_t e = cudaFuncSetAttribute(tc_min_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  tc_min_kernel<<<blocks, kBlock, smem, s>>>(p, w8, M8, E8, T8);
  return cudaGetLastError();
}

cudaError_t launch_tc_tables(int n, int w8, const DevHeader* hdr, const int32_t* U, int32_t* M8, int32_t* E8,
                             int32_t* T8, cudaStream_t s) {
  const uint64_t work = ((uint64_t)(n - kTcC) << kTcC) + 256 + ((uint64_t)1 << w8);
  const int blocks = (int)((work + 255) / 256 < 8192 ? (work + 255) / 256 : 8192);
  tc_tables_kernel<<<blocks, 256, 0, s>>>(n, w8, hdr, U, M8, E8, T8);
  return cudaGetLastError();
}

}  // namespace qgb
