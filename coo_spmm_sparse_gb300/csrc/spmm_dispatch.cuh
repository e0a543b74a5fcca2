// Launch helpers for the segmented kernels: persistent grid sizing and
// programmatic dependent launch.  Each kernel family is instantiated for the
// seven slice widths in its own translation unit, so they compile in
// parallel.
#pragma once

#include <map>
#include <mutex>
#include <utility>

#include "spmm_kernels.cuh"

namespace snack {

// Resident blocks per SM of a kernel (queried once per device and kernel).
inline int resident_blocks(const void *kern) {
  static std::mutex mu;
  static std::map<std::pair<int, const void *>, int> cache;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) dev = 0;
  const std::pair<int, const void *> key(dev, kern);
  std::lock_guard<std::mutex> lock(mu);
  auto it = cache.find(key);
  if (it != cache.end()) return it->second;
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, 256, 0) != cudaSuccess || n < 1) n = 1;
  cache.emplace(key, n);
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

// Blocks of a persistent grid: no more than can be resident at once.
template <typename K>
inline int64_t resident_capacity(K kern) {
  return (int64_t)sm_count() * resident_blocks(reinterpret_cast<const void *>(kern));
}

// Launch with 256 threads.  pdl: the launch may begin while the previous
// kernel on the stream is still running; the kernel's griddep_wait() holds
// it until that kernel has completed and its writes are visible.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_ex(void (*kern)(KArgs...), dim3 grid, bool pdl, cudaStream_t s,
                             Args &&...args) {
  if (grid.x < 1 || grid.y < 1) return cudaSuccess;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(256);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

template <typename... KArgs, typename... Args>
inline cudaError_t launch_ex(void (*kern)(KArgs...), int64_t grid, bool pdl, cudaStream_t s,
                             Args &&...args) {
  if (grid < 1) return cudaSuccess;
  if (grid > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  return launch_ex(kern, dim3((unsigned)grid), pdl, s, std::forward<Args>(args)...);
}

// Team sizes are compiled for 8, 16 and 32 lanes.
inline int team_lanes(const Plan &p) {
  int l = p.lanes < lanes_for(p.bw) ? lanes_for(p.bw) : p.lanes;
  return l < 8 ? 8 : (l > 32 ? 32 : l);
}

#define SNACK_BW_SWITCH(bw, CALL) \
  switch (bw) {                   \
    case 1: CALL(1)               \
    case 2: CALL(2)               \
    case 4: CALL(4)               \
    case 8: CALL(8)               \
    case 16: CALL(16)             \
    case 32: CALL(32)             \
    case 64: CALL(64)             \
    default:                      \
      return cudaErrorInvalidValue; \
  }

// The same with the wide slices of the handle path (128, 256).
#define SNACK_BW_SWITCH_WIDE(bw, CALL) \
  switch (bw) {                        \
    case 128: CALL(128)                \
    case 256: CALL(256)                \
    default:                           \
      SNACK_BW_SWITCH(bw, CALL)        \
  }

// Team size one step down from L for slice width W (L itself if none).
constexpr int half_team(int W, int L) {
  return (L / 2 >= 8 && L / 2 >= lanes_for(W)) ? L / 2 : L;
}

inline int64_t teams_of(const SpmmArgs &a) { return a.nseg * a.nsub; }
inline int64_t teams_of(const SddmmArgs &a) { return a.nseg * a.nsub; }

// Grid rows: SpMM batch sub-slices run as gridDim.y (the segment loop then
// stays the same); the SDDMM's entry sub-ranges are part of its team index.
inline int grid_rows(const SpmmArgs &a) { return a.nsub; }
inline int grid_rows(const SddmmArgs &) { return 1; }

// Persistent grid of `cap` resident blocks for `teams` teams of L lanes,
// `rows` grid rows sharing them.
inline dim3 one_wave_grid(int64_t teams, int L, int64_t cap, int rows) {
  const int64_t per_row = (teams / rows * L + 255) / 256;
  int64_t cap_row = cap / rows;
  if (cap_row < 1) cap_row = 1;
  return dim3((unsigned)(per_row < cap_row ? per_row : cap_row), (unsigned)rows);
}

// Whether halving the team may pay: only while a half-size team still walks
// an average segment in at most four steps (two quads of four entries per
// group per step).  On long segments the doubled walk costs more than the
// second wave it avoids (10000x10000 @95% batch 32 forward 66.3 -> 60.2 us
// without halving), on short ones the halving wins (8192x8192 Zipf-row
// batch 16 forward 24.5 -> 22.6 us with it).
inline bool may_halve(const Plan &p, int LH) {
  return p.mean_len <= 4.0 * 8.0 * LH / lanes_for(p.bw);
}

// Launch `k` (teams of L lanes) on a persistent grid, unless the segments
// overflow one wave of resident teams by less than what `kh` (teams of LH
// = half_team lanes) can hold at once: then the last segments would run as
// a second wave behind their teams' first ones, so `kh` runs instead with
// every segment resident from the start (if halve_ok).
template <typename K, typename KH, typename A>
inline cudaError_t launch_one_wave(K k, int L, KH kh, int LH, bool halve_ok, A a, bool pdl,
                                   cudaStream_t s) {
  const int64_t cap = resident_capacity(k);
  const int64_t teams = teams_of(a);
  const int rows = grid_rows(a);
  if (LH < L && halve_ok) {
    const int64_t cap_h = resident_capacity(kh);
    if (teams > cap * (256 / L) && teams <= cap_h * (256 / LH)) {
      a.lps = LH;
      return launch_ex(kh, one_wave_grid(teams, LH, cap_h, rows), pdl, s, a);
    }
  }
  a.lps = L;
  return launch_ex(k, one_wave_grid(teams, L, cap, rows), pdl, s, a);
}

// CALL2(W, L) for the slice width and team size of a plan.
#define SNACK_BW_LPS_SWITCH(bw, lps, CALL2)                                   \
  switch (bw * 64 + lps) {                                                    \
    case 1 * 64 + 8: CALL2(1, 8) case 1 * 64 + 16: CALL2(1, 16)               \
    case 1 * 64 + 32: CALL2(1, 32) case 2 * 64 + 8: CALL2(2, 8)               \
    case 2 * 64 + 16: CALL2(2, 16) case 2 * 64 + 32: CALL2(2, 32)             \
    case 4 * 64 + 8: CALL2(4, 8) case 4 * 64 + 16: CALL2(4, 16)               \
    case 4 * 64 + 32: CALL2(4, 32) case 8 * 64 + 8: CALL2(8, 8)               \
    case 8 * 64 + 16: CALL2(8, 16) case 8 * 64 + 32: CALL2(8, 32)             \
    case 16 * 64 + 8: CALL2(16, 8) case 16 * 64 + 16: CALL2(16, 16)           \
    case 16 * 64 + 32: CALL2(16, 32) case 32 * 64 + 8: CALL2(32, 8)           \
    case 32 * 64 + 16: CALL2(32, 16) case 32 * 64 + 32: CALL2(32, 32)         \
    case 64 * 64 + 8: CALL2(64, 8) case 64 * 64 + 16: CALL2(64, 16)           \
    case 64 * 64 + 32: CALL2(64, 32) case 128 * 64 + 16: CALL2(128, 16)       \
    case 128 * 64 + 32: CALL2(128, 32) case 256 * 64 + 32: CALL2(256, 32)     \
    default:                                                                  \
      return cudaErrorInvalidValue;                                           \
  }

}  // namespace snack
