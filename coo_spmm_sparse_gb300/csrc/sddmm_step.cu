// The optimizer step fused into the SDDMM (sddmm_segments<BW, LPS, true>):
// each stored entry's gradient updates its value and optimizer state in
// place instead of being written to dW.  Instantiated in its own translation
// unit so that it compiles in parallel with the plain kernels.  Also the
// step applied from a gradient already in memory (opt_apply), for slices
// wide enough that the plain SDDMM plus a streaming update beats the fused
// kernel.
#include "spmm_dispatch.cuh"

namespace snack {
namespace {

// Optimizer step of every stored entry from its whole-batch gradient g,
// one quad per thread (the same update arithmetic as the fused kernel).
__global__ void __launch_bounds__(256) opt_apply(const OptArgs o, const float *__restrict__ g,
                                                 int64_t nnz) {
  griddep_wait();
  const int64_t nq = (nnz + 3) / 4;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < nq; i += stride) {
    const int kq = (int)(4 * i);
    const unsigned mask = kq + 4 <= nnz ? 0xfu : (1u << (int)(nnz - kq)) - 1u;
    OptQuad q;
    opt_load(o, kq, mask, q);
    float res[4];
    load4(g + kq, mask, res);
    opt_store(o, kq, q, res);
  }
}

}  // namespace

cudaError_t launch_opt_apply(const OptArgs &o, const float *g, int64_t nnz, bool pdl,
                             cudaStream_t s) {
  if (nnz == 0) return cudaSuccess;
  const int64_t need = ((nnz + 3) / 4 + 255) / 256;
  const int64_t cap = resident_capacity(opt_apply);
  return launch_ex(opt_apply, need < cap ? need : cap, pdl, s, o, g, nnz);
}

cudaError_t launch_sddmm_step(const Plan &p, const SddmmArgs &args, bool pdl, cudaStream_t s) {
  if (args.nseg == 0) return cudaSuccess;
  SddmmArgs a = args;
  a.lps = team_lanes(p);
  // Only slices of 1-4 floats take the fused step (wider ones apply it from
  // the gradient buffer with opt_apply).
#define SNACK_CALL(W, L)                                                                 \
  return launch_one_wave(sddmm_segments<W, L, true>, L, sddmm_segments<W, half_team(W, L), true>, \
                         half_team(W, L), may_halve(p, half_team(W, L)), a, pdl, s);
  switch (p.bw * 64 + a.lps) {
    case 1 * 64 + 8: SNACK_CALL(1, 8)
    case 1 * 64 + 16: SNACK_CALL(1, 16)
    case 1 * 64 + 32: SNACK_CALL(1, 32)
    case 2 * 64 + 8: SNACK_CALL(2, 8)
    case 2 * 64 + 16: SNACK_CALL(2, 16)
    case 2 * 64 + 32: SNACK_CALL(2, 32)
    case 4 * 64 + 8: SNACK_CALL(4, 8)
    case 4 * 64 + 16: SNACK_CALL(4, 16)
    case 4 * 64 + 32: SNACK_CALL(4, 32)
    default: return cudaErrorInvalidValue;
  }
#undef SNACK_CALL
}

}  // namespace snack
