// Slice-granular checkpoint / resume for long searches (host runtime).
//
// Terastate-per-second QUBO Brute-Force on a Single GPU, §III-C1 and §IV-C: fixing the first
// k_prefix variables splits the search into independent slices whose results combine by
// (lowest energy; among equal energies the lowest rank and the summed tie count). A long run
// (the paper's Table IV goes to N = 55) is therefore a loop over slice chunks that can stop
// after any chunk and resume from a small record. The record lives in a fixed binary file
// (little-endian, see CheckpointFile) rewritten atomically after every chunk.
#include <algorithm>
#include <chrono>
#include <cstddef>
#include <cstdio>
#include <cstring>
#include <string>
#include <vector>

#include "qubo_internal.h"

namespace {

constexpr char kMagic[8] = {'Q', 'U', 'B', 'O', 'C', 'K', 'P', '1'};

// On-disk record (88 bytes). `checksum` is the FNV-1a hash of the preceding bytes.
struct CheckpointFile {
  char magic[8];
  uint32_t version;
  int32_t n, dtype, k_prefix;
  uint64_t q_hash;
  uint64_t next_slice, total_slices;
  int32_t have, pad;
  double best_e;
  uint64_t best_rank, ties;
  uint64_t checksum;
};
static_assert(sizeof(CheckpointFile) == 88, "checkpoint layout");

uint64_t fnv1a(const void* data, size_t bytes) {
  const unsigned char* p = static_cast<const unsigned char*>(data);
  uint64_t h = 0xcbf29ce484222325ull;  // FNV-1a 64-bit offset basis
  for (size_t i = 0; i < bytes; ++i) {
    h ^= p[i];
    h *= 0x100000001b3ull;  // FNV 64-bit prime
  }
  return h;
}

uint64_t record_checksum(const CheckpointFile& c) { return fnv1a(&c, offsetof(CheckpointFile, checksum)); }

// 0: read and valid; 1: no file; QUBO_ERR_CHECKPOINT: unreadable or corrupt.
int read_file(const char* path, CheckpointFile* c) {
  FILE* f = std::fopen(path, "rb");
  if (!f) return 1;
  CheckpointFile r;
  const size_t got = std::fread(&r, 1, sizeof(r), f);
  const bool extra = std::fgetc(f) != EOF;
  std::fclose(f);
  if (got != sizeof(r) || extra || std::memcmp(r.magic, kMagic, 8) != 0 || r.version != 1 ||
      r.checksum != record_checksum(r) || r.next_slice > r.total_slices)
    return QUBO_ERR_CHECKPOINT;
  *c = r;
  return 0;
}

int write_file(const char* path, CheckpointFile c) {
  c.checksum = record_checksum(c);
  std::string tmp = std::string(path) + ".tmp";
  FILE* f = std::fopen(tmp.c_str(), "wb");
  if (!f) return QUBO_ERR_CHECKPOINT;
  const bool ok = std::fwrite(&c, 1, sizeof(c), f) == sizeof(c) && std::fflush(f) == 0;
  if (std::fclose(f) != 0 || !ok || std::rename(tmp.c_str(), path) != 0) {
    std::remove(tmp.c_str());
    return QUBO_ERR_CHECKPOINT;
  }
  return QUBO_OK;
}

uint64_t rank_of(const uint8_t* x, int n) {
  uint64_t r = 0;
  for (int i = 0; i < n; ++i) r = (r << 1) | (x[i] & 1u);
  return r;
}

}  // namespace

extern "C" {

uint64_t qubo_fnv1a64(const void* data, size_t bytes) { return data ? fnv1a(data, bytes) : 0; }

int qubo_checkpoint_read(const char* path, int* out_n, int* out_dtype, int* out_k_prefix, uint64_t* out_q_hash,
                         uint64_t* out_next_slice, uint64_t* out_total_slices, int* out_have, double* out_min_energy,
                         uint64_t* out_argmin_rank, uint64_t* out_tie_count) {
  if (!path || !out_n || !out_dtype || !out_k_prefix || !out_q_hash || !out_next_slice || !out_total_slices ||
      !out_have || !out_min_energy || !out_argmin_rank || !out_tie_count)
    return QUBO_ERR_ARG;
  CheckpointFile c;
  const int st = read_file(path, &c);
  if (st) return QUBO_ERR_CHECKPOINT;  // a missing file is an error here too
  *out_n = c.n;
  *out_dtype = c.dtype;
  *out_k_prefix = c.k_prefix;
  *out_q_hash = c.q_hash;
  *out_next_slice = c.next_slice;
  *out_total_slices = c.total_slices;
  *out_have = c.have;
  *out_min_energy = c.best_e;
  *out_argmin_rank = c.best_rank;
  *out_tie_count = c.ties;
  return QUBO_OK;
}

int qubo_solve_checkpointed(int n, const void* Q, int dtype, int k_prefix, int cache_bits, uint64_t slices_per_chunk,
                            const char* checkpoint_path, double time_budget_s, double* out_min_energy,
                            uint8_t* out_argmin_x, uint64_t* out_tie_count, uint64_t* out_slices_done) {
  if (n < 2 || n > 62 || !Q || !qgb::valid_dtype(dtype) || k_prefix < 1 || k_prefix >= n || !checkpoint_path ||
      !out_min_energy || !out_argmin_x || !out_tie_count || !out_slices_done)
    return QUBO_ERR_ARG;
  const auto t0 = std::chrono::steady_clock::now();
  const uint64_t total = (uint64_t)1 << k_prefix;
  const uint64_t qhash = fnv1a(Q, (size_t)n * n * qgb::dtype_bytes(dtype));
  CheckpointFile c;
  int st = read_file(checkpoint_path, &c);
  if (st == QUBO_ERR_CHECKPOINT) return st;
  if (st == 0) {
    if (c.n != n || c.dtype != dtype || c.k_prefix != k_prefix || c.q_hash != qhash || c.total_slices != total)
      return QUBO_ERR_CHECKPOINT;
  } else {
    std::memset(&c, 0, sizeof(c));
    std::memcpy(c.magic, kMagic, 8);
    c.version = 1;
    c.n = n;
    c.dtype = dtype;
    c.k_prefix = k_prefix;
    c.q_hash = qhash;
    c.total_slices = total;
  }
  uint64_t chunk = slices_per_chunk;
  if (chunk == 0) {
    const int per_slice_bits = n - k_prefix;  // states per slice = 2^(n - k_prefix)
    chunk = per_slice_bits >= 44 ? 1 : ((uint64_t)1 << (44 - per_slice_bits));
  }
  std::vector<uint8_t> x(n);
  bool ran = false;
  while (c.next_slice < total) {
    if (ran && time_budget_s > 0 &&
        std::chrono::duration<double>(std::chrono::steady_clock::now() - t0).count() >= time_budget_s)
      break;
    const uint64_t cnt = std::min<uint64_t>(chunk, total - c.next_slice);
    double e = 0.0;
    uint64_t t = 0;
    st = qubo_solve_slice_range(n, Q, dtype, k_prefix, cache_bits, c.next_slice, cnt, &e, x.data(), &t);
    if (st) return st;  // the file still holds the last completed chunk
    const uint64_t r = rank_of(x.data(), n);
    if (!c.have || e < c.best_e) {
      c.best_e = e;
      c.best_rank = r;
      c.ties = t;
      c.have = 1;
    } else if (e == c.best_e) {
      c.best_rank = r < c.best_rank ? r : c.best_rank;
      c.ties += t;
    }
    c.next_slice += cnt;
    if ((st = write_file(checkpoint_path, c))) return st;
    ran = true;
  }
  if (c.have) {
    *out_min_energy = c.best_e;
    for (int i = 0; i < n; ++i) out_argmin_x[i] = (uint8_t)((c.best_rank >> (n - 1 - i)) & 1u);
    *out_tie_count = c.ties;
  }
  *out_slices_done = c.next_slice;
  return c.next_slice == total ? QUBO_OK : QUBO_INCOMPLETE;
}

}  // extern "C"
