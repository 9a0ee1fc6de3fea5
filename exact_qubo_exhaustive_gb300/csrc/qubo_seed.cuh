// Greedy one-flip descent on the int32 image of U, one warp per descent: the energy it reaches is
// an energy some state attains, which the bounded minimum passes take as a starting best (any
// attained energy is a valid threshold: it is never below the minimum). It decides nothing else;
// the walk still visits every state.
#pragma once

#include <cstdint>

namespace qgb {

constexpr int kSeedMaxN = 62;

// sU: the symmetric n x n image (sU[i][j] = U[min(i,j)][max(i,j)]), shared memory. The start
// state is a SplitMix64-style hash of `seed`; with F > 0 its first F variables are fixed to the
// unit prefix base + (hash mod upg) and only the others flip. Lane l holds the fields of
// variables l and l + 32, g[v] = U_vv + sum over set u != v of U(u, v) (the energy change when x_v
// goes from 0 to 1); each step flips the free variable of the most negative change (the lowest
// index among equals) until none lowers the energy. Called by all 32 lanes; returns the energy.
__device__ __forceinline__ int32_t warp_descent(const int32_t* sU, int n, int F, uint64_t base, uint64_t upg,
                                                uint64_t seed) {
  const int lane = threadIdx.x & 31;
  uint64_t z = (seed + 1) * 0x9E3779B97F4A7C15ull;
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  uint64_t x = z ^ (z >> 31);
  if (F > 0) {  // the prefix: a unit of the group (bit F - 1 - f of P is variable f)
    const uint64_t P = base + (z % upg);
    for (int f = 0; f < F; ++f) x = (x & ~((uint64_t)1 << f)) | (((P >> (F - 1 - f)) & 1u) << f);
  }
  const int v0 = lane, v1 = lane + 32;
  const bool h0 = v0 < n, h1 = v1 < n;
  const bool f0 = h0 && v0 >= F, f1 = h1 && v1 >= F;  // free to flip
  int32_t g0 = h0 ? sU[v0 * n + v0] : 0, g1 = h1 ? sU[v1 * n + v1] : 0;
  for (int u = 0; u < n; ++u) {
    if (!((x >> u) & 1u)) continue;
    if (h0 && u != v0) g0 += sU[u * n + v0];
    if (h1 && u != v1) g1 += sU[u * n + v1];
  }
  // 2 E(x) = sum over set v of (g[v] + U_vv)
  long long twice = 0;
  if (h0 && ((x >> v0) & 1u)) twice += (long long)g0 + sU[v0 * n + v0];
  if (h1 && ((x >> v1) & 1u)) twice += (long long)g1 + sU[v1 * n + v1];
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) twice += __shfl_xor_sync(0xffffffffu, twice, off);
  int32_t e = (int32_t)(twice / 2);
  for (int it = 0; it < 4 * n; ++it) {  // each flip lowers E, so this ends long before the cap
    // key: (change + 2^31) in the high word, the variable in the low word; the least key wins
    unsigned long long key = ~0ull;
    if (f0) {
      const int32_t d = ((x >> v0) & 1u) ? -g0 : g0;
      key = ((unsigned long long)((long long)d + 0x80000000ll) << 32) | (unsigned)v0;
    }
    if (f1) {
      const int32_t d = ((x >> v1) & 1u) ? -g1 : g1;
      const unsigned long long k1 = ((unsigned long long)((long long)d + 0x80000000ll) << 32) | (unsigned)v1;
      key = k1 < key ? k1 : key;
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      const unsigned long long o = __shfl_xor_sync(0xffffffffu, key, off);
      key = o < key ? o : key;
    }
    const int32_t best = (int32_t)((long long)(key >> 32) - 0x80000000ll);
    if (best >= 0) break;  // a local minimum: no single flip lowers E
    const int bv = (int)(key & 0xffffffffu);
    const int32_t sg = ((x >> bv) & 1u) ? -1 : 1;
    x ^= (uint64_t)1 << bv;
    e += best;
    if (h0 && v0 != bv) g0 += sg * sU[bv * n + v0];
    if (h1 && v1 != bv) g1 += sg * sU[bv * n + v1];
  }
  return e;
}

}  // namespace qgb
