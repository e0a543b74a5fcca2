// Backward-input SpMM dX = dY W over the column segmentation.
#include "spmm_dispatch.cuh"

namespace snack {

cudaError_t launch_spmm_cols(const Plan &p, const SpmmArgs &args, bool pdl, cudaStream_t s) {
  if (args.nseg == 0) return cudaSuccess;
  SpmmArgs a = args;
  a.lps = team_lanes(p);
#define SNACK_CALL(W, L)                                                                  \
  return launch_one_wave(spmm_segments<W, L, true>, L, spmm_segments<W, half_team(W, L), true>, \
                         half_team(W, L), may_halve(p, half_team(W, L)), a, pdl, s);
  SNACK_BW_LPS_SWITCH(p.bw, a.lps, SNACK_CALL)
#undef SNACK_CALL
}

}  // namespace snack
