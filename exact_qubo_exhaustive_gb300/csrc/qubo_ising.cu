// Ising input (J, h) converted exactly to the QUBO form, then searched like any QUBO.
//
// Terastate-per-second QUBO Brute-Force on a Single GPU, §I: the Ising energy with spins
// s in {-1, +1} and the QUBO energy with bits x in {0, 1} are the same problem under s = 2x - 1.
// The input convention (the plainest one consistent with the QUBO entry points, which sum over
// all i, j): H(s) = sum_{i,j} J_ij s_i s_j + sum_i h_i s_i. Only J_ij + J_ji matters for i != j,
// and J_ii s_i s_i = J_ii is a constant. With K_ij = J_ij + J_ji (i < j) and s = 2x - 1:
//   H = sum_{i<j} 4 K_ij x_i x_j + sum_i (2 h_i - 2 sum_{j != i} K_ij) x_i + C,
//   C = sum_{i<j} K_ij - sum_i h_i + sum_i J_ii,
// so Q is upper triangular with Q_ij = 4 K_ij (i < j), Q_ii = 2 h_i - 2 sum_{j != i} K_ij, and
// H(s) = E_Q(x) + C. The conversion runs on the host in int64 (exact; int32 output is
// range-checked) or in fp64.
#include <cmath>
#include <cstring>
#include <vector>

#include "qubo_internal.h"

namespace {

template <typename T>
double at(const void* p, size_t i) {
  return static_cast<double>(static_cast<const T*>(p)[i]);
}

// int32 input: exact in int64.
int convert_int(int n, const int32_t* J, const int32_t* h, int64_t* Q, int64_t* C) {
  std::memset(Q, 0, sizeof(int64_t) * (size_t)n * n);
  int64_t c = 0;
  std::vector<int64_t> row(n, 0);  // sum_{j != i} K_ij
  for (int i = 0; i < n; ++i) {
    c += J[(size_t)i * n + i];
    for (int j = i + 1; j < n; ++j) {
      const int64_t k = (int64_t)J[(size_t)i * n + j] + (int64_t)J[(size_t)j * n + i];
      Q[(size_t)i * n + j] = 4 * k;
      row[i] += k;
      row[j] += k;
      c += k;
    }
  }
  for (int i = 0; i < n; ++i) {
    const int64_t hi = h ? h[i] : 0;
    Q[(size_t)i * n + i] = 2 * hi - 2 * row[i];
    c -= hi;
  }
  *C = c;
  return QUBO_OK;
}

// fp32 / fp64 input: the same formulas in fp64, summed in a fixed order (j ascending).
int convert_fp(int n, const void* J, const void* h, int dtype, double* Q, double* C) {
  auto Jat = [&](size_t i) { return dtype == QUBO_FP64 ? at<double>(J, i) : at<float>(J, i); };
  auto hat = [&](int i) { return h ? (dtype == QUBO_FP64 ? at<double>(h, i) : at<float>(h, i)) : 0.0; };
  for (size_t i = 0; i < (size_t)n * n; ++i)
    if (!std::isfinite(Jat(i))) return QUBO_ERR_NONFINITE;
  for (int i = 0; i < n; ++i)
    if (!std::isfinite(hat(i))) return QUBO_ERR_NONFINITE;
  std::memset(Q, 0, sizeof(double) * (size_t)n * n);
  double c = 0.0;
  for (int i = 0; i < n; ++i) c += Jat((size_t)i * n + i);
  for (int i = 0; i < n; ++i)
    for (int j = i + 1; j < n; ++j) {
      const double k = Jat((size_t)i * n + j) + Jat((size_t)j * n + i);
      Q[(size_t)i * n + j] = 4.0 * k;
      c += k;
    }
  for (int i = 0; i < n; ++i) {
    double r = 0.0;
    for (int j = 0; j < n; ++j) {
      if (j == i) continue;
      r += (j > i) ? Jat((size_t)i * n + j) + Jat((size_t)j * n + i) : Jat((size_t)j * n + i) + Jat((size_t)i * n + j);
    }
    Q[(size_t)i * n + i] = 2.0 * hat(i) - 2.0 * r;
    c -= hat(i);
  }
  *C = c;
  for (size_t i = 0; i < (size_t)n * n; ++i)
    if (!std::isfinite(Q[i])) return QUBO_ERR_NONFINITE;
  return std::isfinite(c) ? QUBO_OK : QUBO_ERR_NONFINITE;
}

}  // namespace

extern "C" {

int qubo_ising_to_qubo(int n, const void* J, const void* h, int dtype, void* out_Q, double* out_offset) {
  if (n < 1 || n > 62 || !J || !out_Q || !out_offset || !qgb::valid_dtype(dtype)) return QUBO_ERR_ARG;
  if (dtype == QUBO_INT32) {
    std::vector<int64_t> Q((size_t)n * n);
    int64_t c = 0;
    convert_int(n, static_cast<const int32_t*>(J), static_cast<const int32_t*>(h), Q.data(), &c);
    for (int64_t v : Q)
      if (v < INT32_MIN || v > INT32_MAX) return QUBO_ERR_RANGE;
    int32_t* out = static_cast<int32_t*>(out_Q);
    for (size_t i = 0; i < Q.size(); ++i) out[i] = (int32_t)Q[i];
    *out_offset = (double)c;  // |c| < 2^53: exact
    return QUBO_OK;
  }
  double c = 0.0;
  const int st = convert_fp(n, J, h, dtype, static_cast<double*>(out_Q), &c);
  if (st) return st;
  *out_offset = c;
  return QUBO_OK;
}

int qubo_solve_ising(int n, const void* J, const void* h, int dtype, int k_prefix, int cache_bits, double* out_min_H,
                     int8_t* out_argmin_s, uint64_t* out_tie_count) {
  if (n < 1 || n > 62 || !J || !out_min_H || !out_argmin_s || !out_tie_count || !qgb::valid_dtype(dtype))
    return QUBO_ERR_ARG;
  const bool integer = dtype == QUBO_INT32;
  std::vector<unsigned char> Q((size_t)n * n * (integer ? 4 : 8));
  double offset = 0.0;
  int st = qubo_ising_to_qubo(n, J, h, dtype, Q.data(), &offset);
  if (st) return st;
  double e = 0.0;
  std::vector<uint8_t> x(n);
  uint64_t ties = 0;
  st = qubo_solve(n, Q.data(), integer ? QUBO_INT32 : QUBO_FP64, k_prefix, cache_bits, &e, x.data(), &ties);
  if (st) return st;
  *out_min_H = e + offset;
  for (int i = 0; i < n; ++i) out_argmin_s[i] = (int8_t)(2 * x[i] - 1);
  *out_tie_count = ties;
  return QUBO_OK;
}

}  // extern "C"
