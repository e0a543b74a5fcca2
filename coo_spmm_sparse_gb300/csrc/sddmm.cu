// Backward-weight SDDMM, the dense-operand transpose, and kernel selection.
#include "spmm_dispatch.cuh"

namespace snack {

cudaError_t launch_sddmm(const Plan &p, const SddmmArgs &a, cudaStream_t s) {
  SNACK_WIDTH_CASES(sddmm_segments, )
}

cudaError_t launch_transpose(const float *src, int64_t ld, int nb, int64_t ncols, float *dst,
                             int bw, cudaStream_t s) {
  if (ncols == 0) return cudaSuccess;
  const int64_t grid = (ncols + 31) / 32;
  switch (bw) {
    case 2: transpose_pad<2><<<(unsigned)grid, 256, 0, s>>>(src, ld, nb, ncols, dst); break;
    case 4: transpose_pad<4><<<(unsigned)grid, 256, 0, s>>>(src, ld, nb, ncols, dst); break;
    case 8: transpose_pad<8><<<(unsigned)grid, 256, 0, s>>>(src, ld, nb, ncols, dst); break;
    case 16: transpose_pad<16><<<(unsigned)grid, 256, 0, s>>>(src, ld, nb, ncols, dst); break;
    case 32: transpose_pad<32><<<(unsigned)grid, 256, 0, s>>>(src, ld, nb, ncols, dst); break;
    case 64: transpose_pad<64><<<(unsigned)grid, 256, 0, s>>>(src, ld, nb, ncols, dst); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

int slice_width(int64_t nb) {
  int w = 1;
  while (w < nb && w < kMaxSlice) w <<= 1;
  return w;
}

int entry_lanes(int bw) { return lanes_for(bw); }

// Team size: a group takes 4 entries per step; aim for about two steps per
// group on an average segment, between 4 and 32 lanes.
Plan choose_plan(const SegTable &t, int64_t nb) {
  Plan p;
  p.bw = slice_width(nb < kMaxSlice ? nb : kMaxSlice);
  const int g = lanes_for(p.bw);
  const double want = t.mean_len / 8.0;
  int npt = 1;
  while (npt < want && npt * g < 32) npt <<= 1;
  int lanes = npt * g;
  if (lanes < 4) lanes = 4;
  if (lanes > 32) lanes = 32;
  p.lanes = lanes;
  return p;
}

}  // namespace snack
