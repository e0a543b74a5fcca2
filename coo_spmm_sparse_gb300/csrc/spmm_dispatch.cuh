// Batch-width / team-size dispatch of the segmented kernels.  Each launcher
// is instantiated in its own translation unit so the three families compile
// in parallel.
#pragma once

#include "spmm_kernels.cuh"

namespace snack {

// Lanes per entry for a slice width: 16-byte vectors, and at least one full
// 32-byte sector per group once the slice is 8 floats or wider.
constexpr int lanes_for(int bw) { return bw <= 4 ? 1 : (bw <= 16 ? 2 : 4); }

template <typename Args, typename Kern>
inline cudaError_t launch_teams(Kern kern, const Args &a, int lps, cudaStream_t s) {
  if (a.nseg == 0) return cudaSuccess;
  const int64_t threads = a.nseg * (int64_t)lps;
  const int64_t grid = (threads + 255) / 256;
  if (grid > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  kern<<<(unsigned)grid, 256, 0, s>>>(a);
  return cudaGetLastError();
}

#define SNACK_TEAM_CASES(KERNEL, BW, ...)                                              \
  switch (p.lanes) {                                                                   \
    case 4:                                                                            \
      return launch_teams(KERNEL<BW, lanes_for(BW), 4 __VA_ARGS__>, a, 4, s);          \
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
