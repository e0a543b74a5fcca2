// Forward SpMM Y = X W^T over the row segmentation.
#include "spmm_dispatch.cuh"

namespace snack {

cudaError_t launch_spmm_rows(const Plan &p, const SpmmArgs &args, bool pdl, cudaStream_t s) {
  if (args.nseg == 0) return cudaSuccess;
  SpmmArgs a = args;
  a.lps = team_lanes(p);
#define SNACK_CALL(W, L)                                                                  \
  return launch_one_wave(spmm_segments<W, L, false>, L, spmm_segments<W, half_team(W, L), false>, \
                         half_team(W, L), may_halve(p, half_team(W, L)), a, pdl, s);
  SNACK_BW_LPS_SWITCH(p.bw, a.lps, SNACK_CALL)
#undef SNACK_CALL
}

cudaError_t launch_split_sums(int bw, const SpmmArgs &a, int64_t nsplit, int max_parts,
                              bool pdl, cudaStream_t s) {
  if (nsplit == 0) return cudaSuccess;
  if (bw < 1 || bw > kMaxSlice) return cudaErrorInvalidValue;
  const int tpl = bw / (bw >= 4 ? 4 : bw);  // threads over a line's batch rows (split_sum_vec)
  // threads over a line's parts: one while a thread's eight loads cover the
  // longest line, else enough for that (a power of two, the line in a warp)
  int pl = 1;
  while (pl * tpl < 32 && pl * 8 < max_parts) pl *= 2;
  const int64_t threads = nsplit * tpl * pl;
  const int64_t blocks = (threads + 255) / 256;
  switch (bw) {
    case 1: return launch_ex(split_sums<1>, blocks, pdl, s, a, nsplit, pl);
    case 2: return launch_ex(split_sums<2>, blocks, pdl, s, a, nsplit, pl);
    case 4: return launch_ex(split_sums<4>, blocks, pdl, s, a, nsplit, pl);
    case 8: return launch_ex(split_sums<8>, blocks, pdl, s, a, nsplit, pl);
    case 16: return launch_ex(split_sums<16>, blocks, pdl, s, a, nsplit, pl);
    case 32: return launch_ex(split_sums<32>, blocks, pdl, s, a, nsplit, pl);
    case 64: return launch_ex(split_sums<64>, blocks, pdl, s, a, nsplit, pl);
    case 128: return launch_ex(split_sums<128>, blocks, pdl, s, a, nsplit, pl);
    case 256: return launch_ex(split_sums<256>, blocks, pdl, s, a, nsplit, pl);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace snack
