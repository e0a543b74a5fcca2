// Forward SpMM Y = X W^T over the row segmentation.
#include "spmm_dispatch.cuh"

namespace snack {

cudaError_t launch_spmm_rows(const Plan &p, const SpmmArgs &a, cudaStream_t s) {
  SNACK_WIDTH_CASES(spmm_segments, , false)
}

}  // namespace snack
