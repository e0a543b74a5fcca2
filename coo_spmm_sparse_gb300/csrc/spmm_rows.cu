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

}  // namespace snack
