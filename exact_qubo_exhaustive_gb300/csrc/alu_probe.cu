// ALU throughput microbenchmark used to state the roofline of the enumeration kernels:
// 16 independent chains of one operation per thread, 8 blocks of 256 threads per SM, timed with
// CUDA events; the SM clock is read inside the kernel as clock64 ticks per globaltimer ns. Each
// loop iteration repeats the 16 operations kUnroll times, so the loop's own counter, compare and
// branch (3 instructions) cost under 3 % of the issue slots instead of the 16 % they cost with
// one repetition, which would cap a full-rate operation at 16 / 19 of the issue limit.
#include <vector>

#include "qubo_internal.h"

namespace qgb {
namespace {
constexpr int kChains = 16;
constexpr int kUnroll = 8;

template <int KIND>
__global__ void __launch_bounds__(256) alu_probe_kernel(int iters, int seed, int* out, unsigned long long* clk) {
  const unsigned one = (unsigned)(seed > 0 ? 1 : 2);  // 1 at run time (seed is 1), unknown to the compiler
  const int big = seed > 0 ? 0x7fffffff : 0;          // INT_MAX at run time, unknown to the compiler
  // kinds 10..15: adds in forms the compiler cannot merge or cancel (a fused add-min against an
  // opaque bound on the ALU, an integer multiply-add by an opaque one on the FMA pipe, fp32 adds),
  // alone and mixed; the first kFp chains are fp32 adds, the next kMad multiply-adds, the rest
  // add-mins
  constexpr int kFp = KIND == 12 ? 11 : (KIND == 14 ? 10 : (KIND == 15 ? 12 : 0));
  constexpr int kMad = KIND == 11 ? kChains : (KIND == 13 ? 8 : 0);
  int a[kChains];
  float f[kChains];
  float rinv[kChains];  // kind 16: loop-invariant addends
  unsigned long long f2[kChains];  // kind 9: pairs of fp32 in one 64-bit register
#pragma unroll
  for (int k = 0; k < kChains; ++k) {
    a[k] = (threadIdx.x * 7 + k * 13 + seed) & 1023;
    f[k] = (float)a[k] * 0.5f;
    rinv[k] = (float)((k * 37 + seed) & 63);
    f2[k] = 0;
    if constexpr (KIND == 9 || KIND >= 17) {  // only these kinds carry packed pairs
      const float lo = f[k], hi = f[k] + 1.0f;
      asm("mov.b64 %0, {%1, %2};" : "=l"(f2[k]) : "f"(lo), "f"(hi));
    }
  }
  const unsigned long long c0 = clock64();
  unsigned long long g0;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(g0));
#pragma unroll 1
  for (int it = 0; it < iters; ++it) {
#pragma unroll
    for (int kk = 0; kk < kChains * kUnroll; ++kk) {
      const int k = kk % kChains;
      const int x = a[(k + 1) % kChains], y = a[(k + 2) % kChains];
      if (KIND == 0) a[k] = a[k] + x;
      if (KIND == 1) a[k] = min(a[k], x);
      if (KIND == 2) a[k] = __vimin3_s32(a[k], x, y);
      if (KIND == 3) a[k] = __viaddmin_s32(a[k], x, y);
      if (KIND == 4) f[k] = __fadd_rn(f[k], f[(k + 1) % kChains]);
      if (KIND == 5) f[k] = fminf(f[k], f[(k + 1) % kChains]);
      if (KIND == 6) a[k] = (int)__vimin3_u16x2((unsigned)a[k], (unsigned)x, (unsigned)y);
      if (KIND == 7) a[k] = (int)__viaddmin_u16x2((unsigned)a[k], (unsigned)x, (unsigned)y);
      if (KIND == 9) asm("add.rn.f32x2 %0, %0, %1;" : "+l"(f2[k]) : "l"(f2[(k + 1) % kChains]));
      if constexpr (KIND == 17 || KIND == 18) {
        // fp32x2 adds on the first kPairChains chains (two adds per instruction, FMA pipes) and
        // fused add-mins against an opaque INT_MAX on the rest (ALU): the mix a walk could use
        constexpr int kPairChains = KIND == 17 ? 12 : 10;
        if (k < kPairChains) {
          if ((k & 1) == 0) asm("add.rn.f32x2 %0, %0, %1;" : "+l"(f2[k >> 1]) : "l"(f2[8 + (k >> 1)]));
        } else {
          a[k] = __viaddmin_s32(a[k], x, big);
        }
      } else if constexpr (KIND == 16) {
        // fp32 adds of loop-invariant addends into 16 accumulators, alternating add and subtract:
        // the pattern of the walk's column updates (V[j] +-= Row[a][j])
        f[k] = (k & 1) ? __fsub_rn(f[k], rinv[k]) : __fadd_rn(f[k], rinv[k]);
      } else if constexpr (KIND >= 10) {
        if (k < kFp) {
          f[k] = __fadd_rn(f[k], f[(k + 1) % kFp]);
        } else if (k < kFp + kMad) {
          asm("mad.lo.s32 %0, %1, %2, %0;" : "+r"(a[k]) : "r"(x), "r"((int)one));
        } else {
          a[k] = __viaddmin_s32(a[k], x, big);
        }
      }
      if (KIND == 8) {
        // int32 adds, half of them as multiply-adds by a run-time one, so that the ALU and the
        // FMA pipe's integer multiply-add unit share them
        if (k & 1) {
          asm("mad.lo.u32 %0, %1, %2, %0;" : "+r"(a[k]) : "r"(x), "r"(one));
        } else {
          a[k] = a[k] + x;
        }
      }
    }
  }
  const unsigned long long c1 = clock64();
  unsigned long long g1;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(g1));
  int s = 0;
#pragma unroll
  for (int k = 0; k < kChains; ++k) {
    s += a[k] + (int)f[k];
    if constexpr (KIND == 9 || KIND >= 17) {
      float lo, hi;
      asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(f2[k]));
      s += (int)lo + (int)hi;
    }
  }
  out[blockIdx.x * blockDim.x + threadIdx.x] = s;
  if (threadIdx.x == 0) {
    clk[2 * blockIdx.x] = c1 - c0;
    clk[2 * blockIdx.x + 1] = g1 - g0;
  }
}

template <int KIND>
cudaError_t launch(int blocks, int iters, int* out, unsigned long long* clk) {
  alu_probe_kernel<KIND><<<blocks, 256>>>(iters, 1, out, clk);
  return cudaGetLastError();
}
}  // namespace

cudaError_t run_alu_probe(int kind, int iters, double* ops_per_s, double* sm_mhz) {
  const DevInfo& di = device_info();
  const int blocks = di.sms * 8;
  int* out = nullptr;
  unsigned long long* clk = nullptr;
  cudaError_t e = cudaMalloc(&out, (size_t)blocks * 256 * 4);
  if (e != cudaSuccess) return e;
  e = cudaMalloc(&clk, (size_t)blocks * 16);
  if (e != cudaSuccess) {
    cudaFree(out);
    return e;
  }
  auto go = [&](int it) -> cudaError_t {
    switch (kind) {
      case 0: return launch<0>(blocks, it, out, clk);
      case 1: return launch<1>(blocks, it, out, clk);
      case 2: return launch<2>(blocks, it, out, clk);
      case 3: return launch<3>(blocks, it, out, clk);
      case 4: return launch<4>(blocks, it, out, clk);
      case 5: return launch<5>(blocks, it, out, clk);
      case 6: return launch<6>(blocks, it, out, clk);
      case 7: return launch<7>(blocks, it, out, clk);
      case 8: return launch<8>(blocks, it, out, clk);
      case 9: return launch<9>(blocks, it, out, clk);
      case 10: return launch<10>(blocks, it, out, clk);
      case 11: return launch<11>(blocks, it, out, clk);
      case 12: return launch<12>(blocks, it, out, clk);
      case 13: return launch<13>(blocks, it, out, clk);
      case 14: return launch<14>(blocks, it, out, clk);
      case 15: return launch<15>(blocks, it, out, clk);
      case 16: return launch<16>(blocks, it, out, clk);
      case 17: return launch<17>(blocks, it, out, clk);
      default: return launch<18>(blocks, it, out, clk);
    }
  };
  cudaEvent_t e0 = nullptr, e1 = nullptr;
  float ms = 0.f;
  std::vector<unsigned long long> h((size_t)blocks * 2);
  if ((e = go(64)) != cudaSuccess) goto done;  // warm-up
  if ((e = cudaDeviceSynchronize()) != cudaSuccess) goto done;
  cudaEventCreate(&e0);
  cudaEventCreate(&e1);
  cudaEventRecord(e0);
  if ((e = go(iters)) != cudaSuccess) goto done;
  cudaEventRecord(e1);
  if ((e = cudaEventSynchronize(e1)) != cudaSuccess) goto done;
  cudaEventElapsedTime(&ms, e0, e1);
  if ((e = cudaMemcpy(h.data(), clk, (size_t)blocks * 16, cudaMemcpyDeviceToHost)) != cudaSuccess) goto done;
  {
    double cy = 0, ns = 0;
    for (int b = 0; b < blocks; ++b) {
      cy += (double)h[2 * b];
      ns += (double)h[2 * b + 1];
    }
    *sm_mhz = ns > 0 ? cy / ns * 1e3 : 0.0;
    // kind 9 performs two fp32 adds per instruction
    *ops_per_s = (double)blocks * 256.0 * iters * kChains * kUnroll * (kind == 9 ? 2 : 1) / (ms * 1e-3);
  }
done:
  if (e0) cudaEventDestroy(e0);
  if (e1) cudaEventDestroy(e1);
  cudaFree(out);
  cudaFree(clk);
  return e;
}

}  // namespace qgb
