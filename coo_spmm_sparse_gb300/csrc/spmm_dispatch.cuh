// Batch-width / team-size dispatch of the segmented kernels.  Each launcher
// is instantiated in its own translation unit so the three families compile
// in parallel.
#pragma once

#include <mutex>
#include <unordered_map>

#include "spmm_kernels.cuh"

namespace snack {

// Lanes per entry for a slice width.  One 16-byte vector per lane, and the
// G lanes of a group read an entry's whole dense row (up to one 128-byte
// line) in ONE instruction: the L1 data pipe spends a wavefront per
// (instruction, line), so splitting a row over several instructions costs
// proportionally more.  BW = 64 (two lines) uses 8 lanes x 2 vectors.
constexpr int lanes_for(int bw) { return bw <= 4 ? 1 : (bw >= 32 ? 8 : bw / 4); }

// Resident blocks per SM of a kernel instantiation (queried once per kernel).
inline int resident_blocks(const void *kern) {
  static std::mutex mu;
  static std::unordered_map<const void *, int> cache;
  std::lock_guard<std::mutex> lock(mu);
  auto it = cache.find(kern);
  if (it != cache.end()) return it->second;
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, 256, 0) != cudaSuccess || n < 1) n = 1;
  cache.emplace(kern, n);
  return n;
}

inline int sm_count() {
  static int cached[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) dev = 0;
  if (cached[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1)
      n = 1;
    cached[dev] = n;
  }
  return cached[dev];
}

// Persistent launch: no more blocks than can be resident at once.
template <typename Args, typename Kern>
inline cudaError_t launch_teams(Kern kern, const Args &a, int lps, cudaStream_t s) {
  if (a.nseg == 0) return cudaSuccess;
  const int64_t need = (a.nseg * (int64_t)lps + 255) / 256;
  const int64_t cap = (int64_t)sm_count() * resident_blocks(reinterpret_cast<const void *>(kern));
  const int64_t grid = need < cap ? need : cap;
  kern<<<(unsigned)grid, 256, 0, s>>>(a);
  return cudaGetLastError();
}

#define SNACK_TEAM_CASES(KERNEL, BW, ...)                                              \
  switch (p.lanes < lanes_for(BW) ? lanes_for(BW) : p.lanes) {                         \
    case 4:                                                                            \
      return launch_teams(KERNEL<BW, lanes_for(BW), (lanes_for(BW) > 4 ? lanes_for(BW) : 4) __VA_ARGS__>, a, (lanes_for(BW) > 4 ? lanes_for(BW) : 4), s); \
    case 8:                                                                            \
      return launch_teams(KERNEL<BW, lanes_for(BW), 8 __VA_ARGS__>, a, 8, s);          \
    case 16:                                                                           \
      return launch_teams(KERNEL<BW, lanes_for(BW), 16 __VA_ARGS__>, a, 16, s);        \
    case 32:                                                                           \
      return launch_teams(KERNEL<BW, lanes_for(BW), 32 __VA_ARGS__>, a, 32, s);        \
    default:                                                                           \
      return cudaErrorInvalidValue;                                                    \
  }

#define SNACK_WIDTH_CASES(KERNEL, ...)              \
  switch (p.bw) {                                   \
    case 1: SNACK_TEAM_CASES(KERNEL, 1, __VA_ARGS__)   \
    case 2: SNACK_TEAM_CASES(KERNEL, 2, __VA_ARGS__)   \
    case 4: SNACK_TEAM_CASES(KERNEL, 4, __VA_ARGS__)   \
    case 8: SNACK_TEAM_CASES(KERNEL, 8, __VA_ARGS__)   \
    case 16: SNACK_TEAM_CASES(KERNEL, 16, __VA_ARGS__) \
    case 32: SNACK_TEAM_CASES(KERNEL, 32, __VA_ARGS__) \
    case 64: SNACK_TEAM_CASES(KERNEL, 64, __VA_ARGS__) \
    default:                                        \
      return cudaErrorInvalidValue;                 \
  }

}  // namespace snack
