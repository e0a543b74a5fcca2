// The optimizer step fused into the SDDMM (sddmm_segments<BW, LPS, true>):
// each stored entry's gradient updates its value and optimizer state in
// place instead of being written to dW.  Instantiated in its own translation
// unit so that it compiles in parallel with the plain kernels.
#include "spmm_dispatch.cuh"

namespace snack {

cudaError_t launch_sddmm_step(const Plan &p, const SddmmArgs &args, bool pdl, cudaStream_t s) {
  if (args.nseg == 0) return cudaSuccess;
  SddmmArgs a = args;
  a.lps = team_lanes(p);
#define SNACK_CALL(W, L)                                                                 \
  return launch_one_wave(sddmm_segments<W, L, true>, L, sddmm_segments<W, half_team(W, L), true>, \
                         half_team(W, L), a, pdl, s);
  SNACK_BW_LPS_SWITCH(p.bw, a.lps, SNACK_CALL)
#undef SNACK_CALL
}

}  // namespace snack
