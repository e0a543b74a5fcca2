// Forward pass for callers that cannot allocate device memory.
//
// snack_forward_csr_static() computes Y = X W^T from CSR arrays the caller
// already holds (row_ptr, col, val) and uses, as its only scratch, a fixed
// array in this file's device memory: no cudaMalloc, cudaFree or allocating
// library call is made, and no handle is needed.  The scratch holds the
// transposed slice of X (in_features x slice width floats); it is rewritten
// in full (padding rows included) by every call, so nothing in it has to
// start at zero.  All calls share the one array: calls whose work overlaps
// on the GPU (different streams, or different host threads) race.
//
// The kernel is a variant of the row-segment forward kernel: one team per
// row taken straight from row_ptr (rows are not split), and index / value
// loads that never read past entry nnz - 1, since caller arrays carry no
// padding.
#include <mutex>
#include <string>

#include "spmm_dispatch.cuh"

namespace snack {

void record_thread_error(const std::string &msg);  // api.cu

namespace {

// Scratch capacity: 2^21 floats = 8 MiB of device memory, held by every GPU
// that loads the library until the process exits.
constexpr int64_t kStaticScratchFloats = int64_t(1) << 21;
__device__ __align__(256) float g_static_scratch[kStaticScratchFloats];

constexpr int kMaxDevices = 64;
constexpr int kStaticSlice = 64;  // widest batch slice this entry point runs
std::mutex g_scratch_mu;
float *g_scratch_addr[kMaxDevices] = {};

struct CsrStaticArgs {
  int64_t nseg;  // rows
  const int32_t *row_ptr;
  const int32_t *col;
  const float *val;
  int64_t nnz;
  const float *src;  // transposed X slice [in][BW] (or X itself for BW = 1)
  float *dst;        // Y, element (b, row) at dst[b * ld + row]
  int64_t ld;
  int nb;
  int lps;
};

__device__ __forceinline__ void load_quad_bounded(const CsrStaticArgs &a, int kb, int (&c)[4],
                                                  float (&w)[4]) {
  if ((int64_t)kb + 3 < a.nnz) {
    const int4 c4 = ld_stream_i4(a.col + kb);
    const float4 v4 = ld_stream_f4(a.val + kb);
    c[0] = c4.x;
    c[1] = c4.y;
    c[2] = c4.z;
    c[3] = c4.w;
    w[0] = v4.x;
    w[1] = v4.y;
    w[2] = v4.z;
    w[3] = v4.w;
  } else {
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const bool in = (int64_t)kb + e < a.nnz;
      c[e] = in ? __ldg(a.col + kb + e) : 0;
      w[e] = in ? __ldg(a.val + kb + e) : 0.f;
    }
  }
}

template <int BW>
__global__ void __launch_bounds__(256) spmm_csr_rows_static(const CsrStaticArgs a) {
  using S = SliceShape<BW>;
  constexpr int VEC = S::VEC, NV = S::NV, G = S::G;
  const int lps = a.lps;  // power of two in [G, 32]
  const int npt = lps / G;
  const int lane = threadIdx.x & 31;
  const int tlane = lane & (lps - 1);
  const int grp = tlane / G;
  const int sub = tlane % G;
  const int64_t teams_per_block = blockDim.x / lps;
  const int64_t stride = (int64_t)gridDim.x * teams_per_block;
  const int64_t my_team = (int64_t)blockIdx.x * teams_per_block + threadIdx.x / lps;
  const int64_t warp_team = (int64_t)blockIdx.x * teams_per_block + (threadIdx.x & ~31) / lps;
  const float *src = a.src + sub * VEC;

  for (int64_t t0 = 0; warp_team + t0 < a.nseg; t0 += stride) {
    const int64_t row = my_team + t0;
    const bool active = row < a.nseg;
    const int k0 = active ? a.row_ptr[row] : 0;
    const int k1 = active ? a.row_ptr[row + 1] : 0;

    float acc[NV][VEC];
#pragma unroll
    for (int v = 0; v < NV; ++v)
#pragma unroll
      for (int i = 0; i < VEC; ++i) acc[v][i] = 0.f;

    for (int kb = (k0 & ~3) + 4 * grp; kb < k1; kb += 4 * npt) {
      int c[1][4];
      float w[1][4];
      bool ok[1][4];
      load_quad_bounded(a, kb, c[0], w[0]);
#pragma unroll
      for (int e = 0; e < 4; ++e) ok[0][e] = kb + e >= k0 && kb + e < k1;
      gather_fma<BW, 1>(src, c, w, ok, acc);
    }

    for (int off = G; off < lps; off <<= 1)
#pragma unroll
      for (int v = 0; v < NV; ++v)
#pragma unroll
        for (int i = 0; i < VEC; ++i) acc[v][i] += __shfl_xor_sync(0xffffffffu, acc[v][i], off);

    if (active && grp == 0) {
#pragma unroll
      for (int v = 0; v < NV; ++v)
#pragma unroll
        for (int i = 0; i < VEC; ++i) {
          const int b = v * G * VEC + sub * VEC + i;
          if (b < a.nb) a.dst[(int64_t)b * a.ld + row] = acc[v][i];
        }
    }
  }
}

cudaError_t launch_csr_rows_static(const Plan &p, const CsrStaticArgs &args, cudaStream_t s) {
  CsrStaticArgs a = args;
  a.lps = team_lanes(p);
  const int64_t need = (a.nseg * a.lps + 255) / 256;
#define SNACK_CALL(W)                                                        \
  {                                                                          \
    auto k = spmm_csr_rows_static<W>;                                        \
    const int64_t cap = resident_capacity(k);                                \
    return launch_ex(k, need < cap ? need : cap, false, s, a);               \
  }
  SNACK_BW_SWITCH(p.bw, SNACK_CALL)
#undef SNACK_CALL
}

snack_status fail(snack_status st, const std::string &msg) {
  record_thread_error(msg);
  return st;
}

bool aligned(const void *p, uintptr_t n) { return (reinterpret_cast<uintptr_t>(p) & (n - 1)) == 0; }

}  // namespace
}  // namespace snack

extern "C" snack_status snack_forward_csr_static(int64_t out_features, int64_t in_features,
                                                 int64_t nnz, const int32_t *row_ptr,
                                                 const int32_t *col, const float *val,
                                                 const float *X, float *Y, int64_t batch,
                                                 void *stream) {
  using namespace snack;
  if (out_features < 1 || in_features < 1 || out_features > 0x7fffffffLL ||
      in_features > 0x7fffffffLL)
    return fail(SNACK_ERR_INVALID_ARG, "out_features and in_features must be in [1, 2^31)");
  if (nnz < 0 || nnz > 0x7fffff00LL) return fail(SNACK_ERR_INVALID_ARG, "nnz out of range");
  if (batch < 1) return fail(SNACK_ERR_INVALID_ARG, "batch must be >= 1");
  if (!row_ptr || !X || !Y || (nnz > 0 && (!col || !val)))
    return fail(SNACK_ERR_INVALID_ARG, "NULL pointer argument");
  if (!aligned(row_ptr, 4) || !aligned(X, 16) || !aligned(Y, 16) ||
      (nnz > 0 && (!aligned(col, 16) || !aligned(val, 16))))
    return fail(SNACK_ERR_INVALID_ARG,
                "col, val, X and Y must be 16-byte aligned, row_ptr 4-byte aligned");
  {
    // At batch 1 the kernel reads X itself while other teams write Y, so an
    // in-place call would silently give wrong rows: refuse overlapping ranges.
    const uintptr_t x0 = reinterpret_cast<uintptr_t>(X), y0 = reinterpret_cast<uintptr_t>(Y);
    const uintptr_t x1 = x0 + (uintptr_t)batch * (uintptr_t)in_features * 4u;
    const uintptr_t y1 = y0 + (uintptr_t)batch * (uintptr_t)out_features * 4u;
    if (x0 < y1 && y0 < x1) return fail(SNACK_ERR_INVALID_ARG, "Y overlaps X");
  }
  const int first_width = slice_width(batch < kStaticSlice ? batch : kStaticSlice);
  if (first_width > 1 && in_features * first_width > kStaticScratchFloats)
    return fail(SNACK_ERR_UNSUPPORTED,
                "in_features x batch slice width (" + std::to_string(in_features) + " x " +
                    std::to_string(first_width) + ") exceeds the static scratch of " +
                    std::to_string(kStaticScratchFloats) + " floats");
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail(SNACK_ERR_CUDA, std::string("cudaGetDevice: ") + cudaGetErrorString(e));
  if (dev < 0 || dev >= kMaxDevices) return fail(SNACK_ERR_UNSUPPORTED, "device index too large");
  float *scratch = nullptr;
  {
    // First call on a device: look up the device address of the scratch
    // array (host code cannot use the symbol itself as a device pointer).
    // The address is kept for the life of the process; a cudaDeviceReset()
    // unloads the module and makes it stale (the header says so).
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (!g_scratch_addr[dev]) {
      void *addr = nullptr;
      e = cudaGetSymbolAddress(&addr, g_static_scratch);
      if (e != cudaSuccess)
        return fail(SNACK_ERR_CUDA, std::string("cudaGetSymbolAddress: ") + cudaGetErrorString(e));
      g_scratch_addr[dev] = static_cast<float *>(addr);
    }
    scratch = g_scratch_addr[dev];
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  SegTable shape;
  shape.mean_len = (double)nnz / (double)out_features;
  for (int64_t b0 = 0; b0 < batch; b0 += kStaticSlice) {
    const int nb = (int)((batch - b0) < kStaticSlice ? (batch - b0) : kStaticSlice);
    const Plan p = choose_plan(shape, nb);
    const float *op = X + b0 * in_features;
    if (p.bw > 1) {
      e = launch_transpose(op, in_features, nb, in_features, scratch, p.bw, s);
      if (e != cudaSuccess)
        return fail(SNACK_ERR_CUDA, std::string("transpose launch: ") + cudaGetErrorString(e));
      op = scratch;
    }
    CsrStaticArgs a;
    a.nseg = out_features;
    a.row_ptr = row_ptr;
    a.col = col;
    a.val = val;
    a.nnz = nnz;
    a.src = op;
    a.dst = Y + b0 * out_features;
    a.ld = out_features;
    a.nb = nb;
    e = launch_csr_rows_static(p, a, s);
    if (e != cudaSuccess)
      return fail(SNACK_ERR_CUDA, std::string("forward launch: ") + cudaGetErrorString(e));
  }
  return SNACK_OK;
}
