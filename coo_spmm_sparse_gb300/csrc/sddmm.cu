// Backward-weight SDDMM, the dense-operand transposes, and kernel selection.
#include "spmm_dispatch.cuh"

namespace snack {

cudaError_t launch_sddmm(const Plan &p, const SddmmArgs &args, bool pdl, cudaStream_t s) {
  if (args.nseg == 0) return cudaSuccess;
  SddmmArgs a = args;
  a.lps = team_lanes(p);
#define SNACK_CALL(W, L)                                                               \
  return launch_one_wave(sddmm_segments<W, L>, L, sddmm_segments<W, half_team(W, L)>, \
                         half_team(W, L), may_halve(p, half_team(W, L)), a, pdl, s);
  SNACK_BW_LPS_SWITCH(p.bw, a.lps, SNACK_CALL)
#undef SNACK_CALL
}

cudaError_t launch_transpose(const float *src, int64_t ld, int nb, int64_t ncols, float *dst,
                             int bw, cudaStream_t s, bool pdl) {
#define SNACK_CALL(W) \
  return launch_ex(transpose_pad<W>, transpose_tiles<W>(ncols), pdl, s, src, ld, nb, ncols, dst);
  SNACK_BW_SWITCH_WIDE(bw, SNACK_CALL)
#undef SNACK_CALL
}

cudaError_t launch_transpose_pair(const float *a, int64_t a_ld, int64_t a_cols, float *at,
                                  const float *b, int64_t b_ld, int64_t b_cols, float *bt, int nb,
                                  int bw, cudaStream_t s, bool pdl) {
#define SNACK_CALL(W)                                                                      \
  return launch_ex(transpose_pair<W>, transpose_tiles<W>(a_cols) + transpose_tiles<W>(b_cols), \
                   pdl, s, a, a_ld, a_cols, at, b, b_ld, b_cols, bt, nb, transpose_tiles<W>(a_cols));
  SNACK_BW_SWITCH_WIDE(bw, SNACK_CALL)
#undef SNACK_CALL
}

int slice_width(int64_t nb) {
  int w = 1;
  while (w < nb && w < kMaxSlice) w <<= 1;
  return w;
}

int entry_lanes(int bw) { return lanes_for(bw); }

// Team size: a group takes 4 entries per step; aim for about two steps per
// group on an average segment, between 8 and 32 lanes.
Plan choose_plan(const SegTable &t, int64_t nb) {
  return plan_for_width(t, slice_width(nb < kMaxSlice ? nb : kMaxSlice));
}

int plan_team_lanes(const Plan &p) { return team_lanes(p); }

int device_sms() { return sm_count(); }

Plan plan_for_width(const SegTable &t, int bw) {
  Plan p;
  p.bw = bw;
  p.mean_len = t.mean_len;
  const int g = lanes_for(p.bw);
  const double want = t.mean_len / 8.0;
  int npt = 1;
  while (npt < want && npt * g < 32) npt <<= 1;
  int lanes = npt * g;
  if (lanes < 8) lanes = 8;
  if (lanes > 32) lanes = 32;
  p.lanes = lanes;
  return p;
}

}  // namespace snack
