// Backward-input SpMM dX = dY W over the column segmentation.
#include "spmm_dispatch.cuh"

namespace snack {

cudaError_t launch_spmm_cols(const Plan &p, const SpmmArgs &a, cudaStream_t s) {
  SNACK_WIDTH_CASES(spmm_segments, , true)
}

}  // namespace snack
