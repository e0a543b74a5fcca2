// Both backward products in one launch: dX over the column segments and dW
// over the row segments share a persistent grid, split in proportion to the
// blocks each part would need on its own.
#include "spmm_dispatch.cuh"

namespace snack {

cudaError_t launch_backward_fused(const Plan &pc, const SpmmArgs &cols_in, const Plan &pr,
                                  const SddmmArgs &rows_in, bool pdl, cudaStream_t s) {
  SpmmArgs cols = cols_in;
  SddmmArgs rows = rows_in;
  // One team size for both parts: the larger of the two plans.
  const int lps = team_lanes(pc) > team_lanes(pr) ? team_lanes(pc) : team_lanes(pr);
  cols.lps = lps;
  rows.lps = lps;
  const int64_t need_c = (cols.nseg * lps + 255) / 256;
  const int64_t need_r = (teams_of(rows) * lps + 255) / 256;
  if (need_c + need_r == 0) return cudaSuccess;
#define SNACK_CALL(W, L)                                                            \
  {                                                                                 \
    auto k = cols.perm ? backward_segments<W, L, true>                             \
                       : backward_segments<W, L, false>;                           \
    const int64_t cap = resident_capacity(k);                                       \
    int64_t gc = need_c, gr = need_r;                                               \
    if (gc + gr > cap) {                                                            \
      gc = (cap * need_c + (need_c + need_r) / 2) / (need_c + need_r);              \
      if (need_c > 0 && gc < 1) gc = 1;                                             \
      if (need_r > 0 && gc > cap - 1) gc = cap - 1;                                 \
      gr = need_r == 0 ? 0 : cap - gc;                                              \
    }                                                                               \
    return launch_ex(k, gc + gr, pdl, s, cols, rows, (int)gc);                      \
  }
  SNACK_BW_LPS_SWITCH(pc.bw, lps, SNACK_CALL)
#undef SNACK_CALL
}

}  // namespace snack
