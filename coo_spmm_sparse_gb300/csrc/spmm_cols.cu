// Backward-input SpMM dX = dY W over the column segmentation.
#include "spmm_dispatch.cuh"

namespace snack {

cudaError_t launch_spmm_cols(const Plan &p, const SpmmArgs &args, bool pdl, cudaStream_t s) {
  if (args.nseg == 0) return cudaSuccess;
  SpmmArgs a = args;
  a.lps = team_lanes(p);
  const int64_t need = (a.nseg * a.lps + 255) / 256;
#define SNACK_CALL(W, L)                                        \
  {                                                             \
    auto k = spmm_segments<W, L, true>;                         \
    const int64_t cap = resident_capacity(k);                   \
    return launch_ex(k, need < cap ? need : cap, pdl, s, a);    \
  }
  SNACK_BW_LPS_SWITCH(p.bw, a.lps, SNACK_CALL)
#undef SNACK_CALL
}

}  // namespace snack
