// Segmented kernels with the dense operand resident in shared memory.
//
// At batch slices of 1, 2 or 4 floats the gathered operand row is only 4-16
// bytes, and a warp-wide gather of 32 random rows costs the L1 data pipe
// about one cycle per row (measured with a probe kernel on GB300), which
// makes the L1 the bottleneck of the whole SpMM.  The same random gathers
// from shared memory cost a few bank-conflict wavefronts per 32 rows.  When
// the whole transposed operand fits (lines x slice x 4 bytes <= 192 KB, e.g.
// 10000 x 4 floats), each CTA (1024 threads) copies it once into shared
// memory with cp.async.bulk (completion on an mbarrier, bounded wait), then
// runs the usual segment loop gathering from there.
#include <mutex>
#include <unordered_map>

#include "spmm_dispatch.cuh"

namespace snack {

namespace {

constexpr int kResidentThreads = 1024;
constexpr int64_t kResidentMaxBytes = 192 * 1024;

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// Copy nfl floats from src (global, 16-byte aligned) into dst (this CTA's
// shared memory): bulk copies for the 16-byte multiple, plain loads for the
// last 0-3 floats.  A wait that does not complete within ~2^22 polls sets
// *err and gives up, so the kernel always terminates.
__device__ __forceinline__ void stage_operand(const float *src, int64_t nfl, float *dst,
                                              uint64_t *bar, int *err) {
  const int64_t bulk = nfl & ~int64_t(3);
  if (threadIdx.x == 0) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(1) : "memory");
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  if (threadIdx.x == 0 && bulk > 0) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"((uint32_t)(bulk * 4))
                 : "memory");
    for (int64_t off = 0; off < bulk; off += 8192) {
      const uint32_t n = (uint32_t)((bulk - off < 8192 ? bulk - off : 8192) * 4);
      asm volatile(
          "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
              smem_u32(dst + off)),
          "l"(src + off), "r"(n), "r"(smem_u32(bar))
          : "memory");
    }
  }
  for (int64_t i = bulk + threadIdx.x; i < nfl; i += blockDim.x) dst[i] = src[i];
  if (bulk > 0) {
    for (uint32_t it = 0;; ++it) {
      uint32_t done;
      asm volatile(
          "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], 0;\n"
          " selp.u32 %0, 1, 0, p;\n}\n"
          : "=r"(done)
          : "r"(smem_u32(bar))
          : "memory");
      if (done) break;
      if (it > (1u << 22)) {
        atomicOr(err, 1);
        break;
      }
    }
  }
  __syncthreads();
}

template <int BW, int LPS, bool PERM>
__global__ void __launch_bounds__(kResidentThreads) spmm_resident(const SpmmArgs a, int64_t n_op,
                                                                   int *err) {
  extern __shared__ __align__(128) float op_s[];
  __shared__ uint64_t bar;
  griddep_wait();
  stage_operand(a.src, n_op * BW, op_s, &bar, err);
  spmm_part<BW, LPS, PERM, true>(a, op_s, blockIdx.x, gridDim.x);
}

template <int BW, int LPS>
__global__ void __launch_bounds__(kResidentThreads) sddmm_resident(const SddmmArgs a, int64_t n_op,
                                                                    int *err) {
  extern __shared__ __align__(128) float op_s[];
  __shared__ uint64_t bar;
  griddep_wait();
  stage_operand(a.xt, n_op * BW, op_s, &bar, err);
  sddmm_part<BW, LPS, true>(a, op_s, blockIdx.x, gridDim.x);
}

// Persistent grid for a resident-operand kernel with `smem` bytes.
template <typename K, typename A>
cudaError_t launch_resident(K kern, const A &a, int64_t n_op, int *err, size_t smem, bool pdl,
                            cudaStream_t s) {
  static std::mutex mu;
  static std::unordered_map<const void *, size_t> raised;
  const void *key = reinterpret_cast<const void *>(kern);
  {
    std::lock_guard<std::mutex> lock(mu);
    auto it = raised.find(key);
    if (it == raised.end() || it->second < smem) {
      cudaError_t e =
          cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      if (e != cudaSuccess) return e;
      raised[key] = smem;
    }
  }
  int per_sm = 0;
  cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kResidentThreads, smem);
  if (e != cudaSuccess) return e;
  if (per_sm < 1) return cudaErrorInvalidConfiguration;
  const int64_t need = (a.nseg * a.lps + kResidentThreads - 1) / kResidentThreads;
  const int64_t cap = (int64_t)sm_count() * per_sm;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(need < cap ? need : cap));
  cfg.blockDim = dim3(kResidentThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, a, n_op, err);
}

}  // namespace

// Slices of 1-4 floats whose whole operand fits in 192 KB, on layers of at
// least 2^22 entries whose value bytes cover the staging copies (one operand
// per SM).  Measured on GB300: on smaller layers (e.g. 1 M entries at 10000
// lines, or the 118 k-entry GPT-2 MLP layers) the segment kernels with the
// stream look-ahead are faster, the copies being a large part of the traffic.
bool resident_fits(int bw, int64_t n_op, int64_t nseg, int64_t nnz) {
  return bw <= 4 && n_op * bw * 4 <= kResidentMaxBytes && nseg >= 2 * (int64_t)sm_count() &&
         nnz >= (int64_t(1) << 22) && (int64_t)sm_count() * n_op * bw <= nnz;
}

cudaError_t launch_resident_spmm(bool perm, const Plan &p, const SpmmArgs &args, int64_t n_op,
                                 int *err, bool pdl, cudaStream_t s) {
  if (args.nseg == 0) return cudaSuccess;
  SpmmArgs a = args;
  a.lps = team_lanes(p);
  const size_t smem = (size_t)((n_op * p.bw + 3) & ~int64_t(3)) * 4;
#define SNACK_CALL(W, L)                                                                 \
  return perm ? launch_resident(spmm_resident<W, L, true>, a, n_op, err, smem, pdl, s)  \
              : launch_resident(spmm_resident<W, L, false>, a, n_op, err, smem, pdl, s);
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

cudaError_t launch_resident_sddmm(const Plan &p, const SddmmArgs &args, int64_t n_op, int *err,
                                  bool pdl, cudaStream_t s) {
  if (args.nseg == 0) return cudaSuccess;
  SddmmArgs a = args;
  a.lps = team_lanes(p);
  const size_t smem = (size_t)((n_op * p.bw + 3) & ~int64_t(3)) * 4;
#define SNACK_CALL(W, L) return launch_resident(sddmm_resident<W, L>, a, n_op, err, smem, pdl, s);
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
