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
#include <map>
#include <mutex>
#include <utility>

#include "spmm_dispatch.cuh"

namespace snack {

namespace {

constexpr int kResidentThreads = 1024;
constexpr int64_t kResidentMaxBytes = 192 * 1024;

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// Bounded wait for phase `parity` of the mbarrier at bar: true once it has
// completed, false after `limit` polls (each poll may block for a
// hardware-bounded time).
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity, uint32_t limit) {
  for (uint32_t it = 0; it <= limit; ++it) {
    uint32_t done;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(done)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    if (done) return true;
  }
  return false;
}

// Copy nfl floats from src (global, 16-byte aligned) into dst (this CTA's
// shared memory): bulk copies for the 16-byte multiple, plain loads for the
// last 0-3 floats.  Returns true (for the whole block) when the copy has
// landed.  A wait that does not complete within ~2^22 polls sets *err, waits
// once more (bounded) for the copies still in flight, and returns false:
// the block then skips its work and exits, so the kernel always terminates.
__device__ __forceinline__ bool stage_operand(const float *src, int64_t nfl, float *dst,
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
  bool ok = true;
  if (bulk > 0) ok = mbar_wait(bar, 0, 1u << 22);
  ok = __syncthreads_and(ok);
  if (!ok) {
    if (threadIdx.x == 0) atomicOr(err, 1);
    mbar_wait(bar, 0, 1u << 22);  // let copies still in flight land before the block exits
  }
  __syncthreads();
  return ok;
}

template <int BW, int LPS, bool PERM>
__global__ void __launch_bounds__(kResidentThreads) spmm_resident(const SpmmArgs a, int64_t n_op,
                                                                   int *err) {
  extern __shared__ __align__(128) float op_s[];
  __shared__ uint64_t bar;
  griddep_wait();
  if (!stage_operand(a.src, n_op * BW, op_s, &bar, err)) return;
  spmm_part<BW, LPS, PERM, true>(a, op_s, blockIdx.x, gridDim.x);
}

template <int BW, int LPS>
__global__ void __launch_bounds__(kResidentThreads) sddmm_resident(const SddmmArgs a, int64_t n_op,
                                                                    int *err) {
  extern __shared__ __align__(128) float op_s[];
  __shared__ uint64_t bar;
  griddep_wait();
  if (!stage_operand(a.xt, n_op * BW, op_s, &bar, err)) return;
  sddmm_part<BW, LPS, true>(a, op_s, blockIdx.x, gridDim.x);
}

// Persistent grid for a resident-operand kernel with `smem` bytes.
template <typename K, typename A>
cudaError_t launch_resident(K kern, const A &a, int64_t n_op, int *err, size_t smem, bool pdl,
                            cudaStream_t s) {
  // The shared-memory limit is a per-device attribute of the kernel: the
  // record of limits already raised is keyed by (device, kernel).
  static std::mutex mu;
  static std::map<std::pair<int, const void *>, size_t> raised;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const std::pair<int, const void *> key(dev, reinterpret_cast<const void *>(kern));
  {
    std::lock_guard<std::mutex> lock(mu);
    auto it = raised.find(key);
    if (it == raised.end() || it->second < smem) {
      e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      if (e != cudaSuccess) return e;
      raised[key] = smem;
    }
  }
  int per_sm = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kResidentThreads, smem);
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

// Self-test of the failure path: an mbarrier that expects 16 bytes nobody
// sends, waited on with a short bound; the block records the time-out in
// *err and exits normally.
__global__ void __launch_bounds__(32) wait_selftest(int *err, uint32_t limit) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(&bar)), "r"(1) : "memory");
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  if (threadIdx.x == 0)
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(&bar)),
                 "r"(16u)
                 : "memory");
  const bool ok = __syncthreads_and(mbar_wait(&bar, 0, limit));
  if (threadIdx.x == 0) {
    if (!ok) atomicOr(err, 1);
    asm volatile("mbarrier.inval.shared::cta.b64 [%0];" ::"r"(smem_u32(&bar)) : "memory");
  }
}

}  // namespace

cudaError_t launch_wait_selftest(int *err, cudaStream_t s) {
  wait_selftest<<<1, 32, 0, s>>>(err, 1024u);
  return cudaGetLastError();
}

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
