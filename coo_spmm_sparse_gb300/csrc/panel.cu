// Column-panel kernels: the dense operand staged in shared memory panel by
// panel, for batch slices of 8-64 floats.
//
// At slices of 8+ floats the segment kernels gather every entry's operand
// row (32-256 bytes) through L1, and the L1 data pipe (one wavefront per
// gathered row) with the L2 misses behind it sets their time.  Here each
// CTA (one per SM, 1024 threads) sweeps the transposed operand [n_op][BW]
// through shared memory in column panels of PW = 64 KB / (4 BW) lines,
// three panels resident at a time:
//
//  * warp 31 is the producer: its lane 0 copies panel p into stage p % 3
//    with cp.async.bulk (completion on that stage's "full" mbarrier) once
//    all 31 consumer warps have released the panel that stage held (its
//    "empty" mbarrier).  Every wait is bounded; a wait that gives up sets
//    the layer's device error flag and the CTA winds down.
//  * each consumer warp owns a contiguous range of the line-ordered entry
//    stream (the CTA's lines are a row-aligned, entry-balanced share of the
//    table; its 31 warps split that share evenly), covering at most RW
//    lines.  Entries of a line are sorted by the operand index, so the part
//    of a line that falls in panel p is the next run of its entries: the
//    warp keeps a cursor per line and, for each resident panel, walks each
//    line's run in steps of one quad (4 entries) per group of G lanes,
//    gathering the operand rows from shared memory.
//  * forward / dX: the lines' sums stay in registers across all panels.  At
//    the end each warp reduces them over its groups; lines wholly inside a
//    warp's range are written directly, a line cut by warp boundaries is
//    summed by the warp where it starts, adding the other warps' parts in
//    warp order through shared memory (deterministic, no atomics).
//  * dW: the line's dY slice stays in registers; each entry's dot product
//    is finished by a shuffle reduction over its group and stored.
//
// The index and value streams of the warp's range are asked into L2 at the
// start (cp.async.bulk.prefetch.L2, before the wait on the producing
// transpose): the sweep reads each line's runs panel by panel, not in one
// pass, and L2 hits keep those short runs cheap.
#include <algorithm>
#include <cstdlib>
#include <map>
#include <mutex>
#include <utility>

#include "spmm_dispatch.cuh"

namespace snack {

namespace {

constexpr int kPanelThreads = 1024;
constexpr int kConsumers = 31;          // warps 0-30 consume, warp 31 produces
constexpr int kStages = 3;
constexpr int kStageBytes = 64 * 1024;  // one panel
constexpr int kChunkBytes = 32 * 1024;  // bulk copies per panel are cut at this size
constexpr uint32_t kWaitPolls = 1u << 22;

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ bool bar_wait(uint64_t *bar, uint32_t parity) {
  for (uint32_t it = 0; it <= kWaitPolls; ++it) {
    uint32_t done;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(done)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    if (done) return true;
  }
  return false;
}

__device__ __forceinline__ void bar_arrive(uint64_t *bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

// Panel p of the operand (lines [p PW, p PW + rows)) into `dst`, completing
// on `bar` (lane 0 of the producer).
__device__ __forceinline__ void load_panel(const float *src, int64_t first_line, int rows, int bw,
                                           float *dst, uint64_t *bar) {
  const uint32_t bytes = (uint32_t)rows * (uint32_t)bw * 4u;
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
               "r"(bytes)
               : "memory");
  const char *g = reinterpret_cast<const char *>(src + first_line * bw);
  char *sdst = reinterpret_cast<char *>(dst);
  for (uint32_t off = 0; off < bytes; off += kChunkBytes) {
    const uint32_t n = bytes - off < (uint32_t)kChunkBytes ? bytes - off : (uint32_t)kChunkBytes;
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_addr(sdst + off)),
        "l"(g + off), "r"(n), "r"(smem_addr(bar))
        : "memory");
  }
}

// Consumer-warp barrier (named barrier 1, the 31 consumer warps only).
__device__ __forceinline__ void consumers_sync() {
  asm volatile("bar.sync 1, %0;" ::"r"(kConsumers * 32) : "memory");
}

template <int BW>
__host__ __device__ constexpr int panel_lines() {
  return kStageBytes / (4 * BW);
}

// One quad (entries kb..kb+3) of the index / value streams.
template <int MODE>
__device__ __forceinline__ void panel_quad(const PanelArgs &a, int kb, int (&c)[4], float (&w)[4]) {
  const int4 c4 = ld_stream_i4(a.idx + kb);
  c[0] = c4.x;
  c[1] = c4.y;
  c[2] = c4.z;
  c[3] = c4.w;
  if constexpr (MODE == kPanelSpmm) {
    const float4 v4 = ld_stream_f4(a.val + kb);
    w[0] = v4.x;
    w[1] = v4.y;
    w[2] = v4.z;
    w[3] = v4.w;
  } else if constexpr (MODE == kPanelSpmmPerm) {
    const int4 p4 = ld_stream_i4(a.perm + kb);
    w[0] = __ldg(a.val + p4.x);
    w[1] = __ldg(a.val + p4.y);
    w[2] = __ldg(a.val + p4.z);
    w[3] = __ldg(a.val + p4.w);
  }
}

// Forward / dX epilogue of a consumer warp: reduce the lines' sums over the
// groups, then write them out.  A line that starts in this warp's range is
// this warp's to write; its parts in later warps (a line cut by warp
// boundaries) arrive through `slot`, added in warp order.  Lines without
// entries get zeros.
template <int BW, int RW>
__device__ __forceinline__ void panel_spmm_out(const PanelArgs &a,
                                               float (&acc)[RW][SliceShape<BW>::NV]
                                                           [SliceShape<BW>::VEC],
                                               const int4 *part, float *slot, int warp, int lane,
                                               int nl, int first, int W0, int W1) {
  using S = SliceShape<BW>;
  constexpr int VEC = S::VEC, NV = S::NV, G = S::G;
  const int grp = lane / G, sub = lane % G;
#pragma unroll
  for (int j = 0; j < RW; ++j)
#pragma unroll
    for (int off = G; off < 32; off <<= 1)
#pragma unroll
      for (int v = 0; v < NV; ++v)
#pragma unroll
        for (int i = 0; i < VEC; ++i) acc[j][v][i] += __shfl_xor_sync(0xffffffffu, acc[j][v][i], off);
  const bool head_cut = nl > 0 && a.ptr[first] < W0;  // first line started in an earlier warp
  if (head_cut && grp == 0) {
#pragma unroll
    for (int v = 0; v < NV; ++v)
#pragma unroll
      for (int i = 0; i < VEC; ++i) slot[warp * BW + v * G * VEC + sub * VEC + i] = acc[0][v][i];
  }
  consumers_sync();
  const int4 cta = part[kConsumers];  // {first line, end line} of this CTA
#pragma unroll
  for (int j = 0; j < RW; ++j) {
    if (j >= nl || (j == 0 && head_cut)) continue;
    const int r = first + j;
    const int rend = a.ptr[r + 1];
    if (rend > W1) {  // cut: add the later warps' parts in order
      for (int w2 = warp + 1; w2 < kConsumers && part[w2].x < rend; ++w2) {
        if (part[w2].y <= part[w2].x) continue;
#pragma unroll
        for (int v = 0; v < NV; ++v)
#pragma unroll
          for (int i = 0; i < VEC; ++i) acc[j][v][i] += slot[w2 * BW + v * G * VEC + sub * VEC + i];
      }
    }
    if (grp == 0) {
#pragma unroll
      for (int v = 0; v < NV; ++v)
#pragma unroll
        for (int i = 0; i < VEC; ++i) {
          const int b = v * G * VEC + sub * VEC + i;
          if (b < a.nb) a.dst[(int64_t)b * a.ld + r] = acc[j][v][i];
        }
    }
  }
  for (int r = cta.x + warp * 32 + lane; r < cta.y; r += kConsumers * 32) {
    if (a.ptr[r] == a.ptr[r + 1])
      for (int b = 0; b < a.nb; ++b) a.dst[(int64_t)b * a.ld + r] = 0.f;
  }
}

template <int BW, int RW, int MODE>
__global__ void __launch_bounds__(kPanelThreads, 1) panel_kernel(const PanelArgs a) {
  using S = SliceShape<BW>;
  constexpr int VEC = S::VEC, NV = S::NV, G = S::G;
  constexpr int PW = panel_lines<BW>();
  static_assert(PW * BW * 4 == kStageBytes, "panel size");

  extern __shared__ __align__(128) float smem_f[];
  float *stage = smem_f;                                  // [kStages][PW][BW]
  float *slot = smem_f + kStages * PW * BW;               // [kConsumers][BW]
  __shared__ __align__(8) uint64_t full[kStages], empty[kStages];
  __shared__ int4 part[32];

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid < 32) part[tid] = a.part[(int64_t)blockIdx.x * 32 + tid];
  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(&full[s])), "r"(1)
                   : "memory");
      asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(&empty[s])),
                   "r"(kConsumers)
                   : "memory");
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  // The warp's index / value streams are immutable here: ask L2 for them
  // while the producing transpose may still run.
  if (warp < kConsumers && lane == 0) {
    const int4 me = part[warp];
    const int k0 = me.x & ~3, k1 = (me.y + 3) & ~3;
    if (k1 > k0) {
      l2_prefetch(a.idx + k0, (uint32_t)(k1 - k0) * 4);
      if (MODE == kPanelSpmmPerm) l2_prefetch(a.perm + k0, (uint32_t)(k1 - k0) * 4);
      else if (MODE == kPanelSpmm) l2_prefetch(a.val + k0, (uint32_t)(k1 - k0) * 4);
    }
  }
  griddep_wait();
  const int npanels = (int)((a.n_op + PW - 1) / PW);

  if (warp == kConsumers) {
    // ---------------------------------------------------------- producer
    if (lane == 0) {
      int issued = 0;
      for (int p = 0; p < npanels; ++p) {
        const int s = p % kStages;
        if (p >= kStages) {
          if (!bar_wait(&empty[s], (uint32_t)((p / kStages - 1) & 1))) {
            atomicOr(a.err, 1);
            break;
          }
          asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        }
        const int64_t l0 = (int64_t)p * PW;
        const int rows = (int)(a.n_op - l0 < PW ? a.n_op - l0 : PW);
        load_panel(a.src, l0, rows, BW, stage + (size_t)s * PW * BW, &full[s]);
        issued = p + 1;
      }
      // No copy may be in flight when the CTA exits: wait (bounded) for the
      // last panel issued into each stage.
      for (int s = 0; s < kStages && s < issued; ++s) {
        const int last = s + ((issued - 1 - s) / kStages) * kStages;
        if (!bar_wait(&full[s], (uint32_t)((last / kStages) & 1))) atomicOr(a.err, 1);
      }
    }
    return;
  }

  // ------------------------------------------------------------ consumers
  const int grp = lane / G, sub = lane % G;
  const int4 me = part[warp];
  const int W0 = me.x, W1 = me.y, first = me.z, nl = me.w;
  // Per line: cursor (first entry not yet taken), end of the warp's part,
  // and the operand index at the cursor once known (a line whose next entry
  // lies in a later panel is skipped without touching its streams).
  int kcur[RW], kend[RW], cnext[RW];
  float acc[RW][NV][VEC];  // forward / dX: line sums; dW: the line's dY slice
#pragma unroll
  for (int j = 0; j < RW; ++j) {
    kcur[j] = 0;
    kend[j] = 0;
    cnext[j] = 0;
    if (j < nl) {
      const int r = first + j;
      kcur[j] = max(a.ptr[r], W0);
      kend[j] = min(a.ptr[r + 1], W1);
    }
#pragma unroll
    for (int v = 0; v < NV; ++v)
#pragma unroll
      for (int i = 0; i < VEC; ++i) acc[j][v][i] = 0.f;
    if constexpr (MODE == kPanelSddmm) {
      if (j < nl) {
        const float *p = a.dyt + (int64_t)(first + j) * BW + sub * VEC;
#pragma unroll
        for (int v = 0; v < NV; ++v) load_vec<VEC>(p + v * G * VEC, acc[j][v]);
      }
    }
  }

  bool ok = true;
  for (int p = 0; p < npanels && ok; ++p) {
    const int s = p % kStages;
    ok = bar_wait(&full[s], (uint32_t)((p / kStages) & 1));
    if (!ok) {
      if (lane == 0) atomicOr(a.err, 1);
      break;
    }
    const float *st = stage + (size_t)s * PW * BW + sub * VEC;
    const int pend = (p + 1) * PW;  // entries of this panel have index < pend
#pragma unroll
    for (int j = 0; j < RW; ++j) {
      if (j >= nl || cnext[j] >= pend) continue;
      int k = kcur[j];
      const int k1 = kend[j];
      while (k < k1) {  // warp-uniform
        const int kb = (k & ~3) + 4 * grp;
        int c[4] = {0, 0, 0, 0};
        float w[4] = {0.f, 0.f, 0.f, 0.f};
        if (kb < k1) panel_quad<MODE>(a, kb, c, w);
        bool take[4];
        int cnt = 0, first_beyond = 0x7fffffff;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const bool in = kb + e >= k && kb + e < k1;
          take[e] = in && c[e] < pend;
          if (in && c[e] >= pend) first_beyond = min(first_beyond, c[e]);
          cnt += take[e] ? 1 : 0;
        }
        float x[4][NV][VEC];
#pragma unroll
        for (int e = 0; e < 4; ++e)
#pragma unroll
          for (int v = 0; v < NV; ++v) {
            if (take[e]) {
              load_op<VEC, true>(st + (c[e] & (PW - 1)) * BW + v * G * VEC, x[e][v]);
            } else {
#pragma unroll
              for (int i = 0; i < VEC; ++i) x[e][v][i] = 0.f;
            }
          }
        if constexpr (MODE == kPanelSddmm) {
          float res[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            float d = 0.f;
#pragma unroll
            for (int v = 0; v < NV; ++v)
#pragma unroll
              for (int i = 0; i < VEC; ++i) d = fmaf(acc[j][v][i], x[e][v][i], d);
#pragma unroll
            for (int off = 1; off < G; off <<= 1) d += __shfl_xor_sync(0xffffffffu, d, off);
            res[e] = d;
          }
          if (sub == 0) {
            float *dwp = a.dw + kb;
            if (take[0] && take[1] && take[2] && take[3]) {
              float4 o = make_float4(res[0], res[1], res[2], res[3]);
              if (a.accumulate) {
                const float4 old = *reinterpret_cast<const float4 *>(dwp);
                o.x += old.x;
                o.y += old.y;
                o.z += old.z;
                o.w += old.w;
              }
              *reinterpret_cast<float4 *>(dwp) = o;
            } else {
#pragma unroll
              for (int e = 0; e < 4; ++e)
                if (take[e]) dwp[e] = a.accumulate ? dwp[e] + res[e] : res[e];
            }
          }
        } else {
#pragma unroll
          for (int e = 0; e < 4; ++e)
#pragma unroll
            for (int v = 0; v < NV; ++v)
#pragma unroll
              for (int i = 0; i < VEC; ++i)
                acc[j][v][i] = fmaf(take[e] ? w[e] : 0.f, x[e][v][i], acc[j][v][i]);
        }
        // The taken entries are a prefix of [k, k1): advance past them; stop
        // at the first entry of a later panel.
        const int total = __reduce_add_sync(0xffffffffu, (unsigned)cnt) / G;
        k += total;
        // entries of a line are sorted: the smallest index past the panel is
        // the one at the new cursor
        const int nxt = (int)__reduce_min_sync(0xffffffffu, (unsigned)first_beyond);
        if (nxt != 0x7fffffff) {
          cnext[j] = nxt;
          break;
        }
      }
      kcur[j] = k;
      if (k >= k1) cnext[j] = 0x7fffffff;  // the warp's part of this line is done
    }
    __syncwarp();
    if (lane == 0) bar_arrive(&empty[s]);
  }
  if constexpr (MODE != kPanelSddmm)
    panel_spmm_out<BW, RW>(a, acc, part, slot, warp, lane, nl, first, W0, W1);
}

template <typename K>
cudaError_t launch_panel_kernel(K kern, const PanelArgs &a, int64_t ctas, size_t smem, bool pdl,
                                cudaStream_t s) {
  static std::mutex mu;
  static std::map<std::pair<int, const void *>, bool> raised;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  {
    std::lock_guard<std::mutex> lock(mu);
    const std::pair<int, const void *> key(dev, reinterpret_cast<const void *>(kern));
    if (!raised[key]) {
      e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      if (e != cudaSuccess) return e;
      raised[key] = true;
    }
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)ctas);
  cfg.blockDim = dim3(kPanelThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, a);
}

}  // namespace

int64_t panel_min_nnz() {
  const char *e = std::getenv("SNACK_PANEL_MIN_NNZ");
  if (e && *e) {
    char *end = nullptr;
    const long long v = std::strtoll(e, &end, 10);
    if (end != e && v >= 0) return (int64_t)v;
  }
  return int64_t(1) << 21;
}

bool panel_fits(const PanelTable &t, int bw) {
  return t.d_part != nullptr && t.lines_max <= kPanelLinesPerWarp &&
         (bw == 8 || bw == 16 || bw == 32 || bw == 64);
}

cudaError_t launch_panel(int mode, int bw, const PanelTable &t, const PanelArgs &args, bool pdl,
                         cudaStream_t s) {
  PanelArgs a = args;
  a.part = t.d_part;
  const size_t smem = (size_t)kStages * kStageBytes + (size_t)kConsumers * bw * 4;
#define SNACK_PANEL(W)                                                                         \
  case W:                                                                                      \
    if (mode == kPanelSpmm)                                                                    \
      return launch_panel_kernel(panel_kernel<W, kPanelLinesPerWarp, kPanelSpmm>, a, t.ctas,   \
                                 smem, pdl, s);                                                \
    if (mode == kPanelSpmmPerm)                                                                \
      return launch_panel_kernel(panel_kernel<W, kPanelLinesPerWarp, kPanelSpmmPerm>, a,       \
                                 t.ctas, smem, pdl, s);                                        \
    return launch_panel_kernel(panel_kernel<W, kPanelLinesPerWarp, kPanelSddmm>, a, t.ctas,    \
                               smem, pdl, s);
  switch (bw) {
    SNACK_PANEL(8)
    SNACK_PANEL(16)
    SNACK_PANEL(32)
    SNACK_PANEL(64)
    default:
      return cudaErrorInvalidValue;
  }
#undef SNACK_PANEL
}

// Entry-balanced partition of a line table for the panel kernels: `ctas`
// CTAs take row-aligned shares of about nnz / ctas entries; each CTA's 31
// consumer warps split its share evenly.  Per CTA 32 int4: warps 0-30
// {first entry, end entry, first line, lines}, then {first line, end line}.
void build_panel_partition(const std::vector<int32_t> &ptr, int64_t nlines, int64_t nnz,
                           int ctas, std::vector<int4> &part, int *lines_max) {
  part.assign((size_t)ctas * 32, make_int4(0, 0, 0, 0));
  *lines_max = 0;
  int64_t r0 = 0;
  for (int c = 0; c < ctas; ++c) {
    // end line: the line boundary nearest to the CTA's share of entries (a
    // line much longer than a share then gets a CTA to itself, instead of
    // stretching one CTA's warp ranges over many short lines)
    int64_t r1 = nlines;
    if (c + 1 < ctas) {
      const int64_t target = (nnz * (c + 1)) / ctas;
      const int64_t up =
          std::lower_bound(ptr.begin() + r0, ptr.begin() + nlines, (int32_t)target) - ptr.begin();
      r1 = up;
      if (up > r0 && target - ptr[up - 1] < ptr[up] - target) r1 = up - 1;
      if (r1 < r0) r1 = r0;
    }
    const int64_t e0 = ptr[r0], e1 = ptr[r1];
    for (int w = 0; w < kConsumers; ++w) {
      const int64_t w0 = e0 + (e1 - e0) * w / kConsumers;
      const int64_t w1 = e0 + (e1 - e0) * (w + 1) / kConsumers;
      int first = (int)r0, n = 0;
      if (w1 > w0) {
        // line holding entry w0 (the last line starting at or before it
        // whose range is not empty) and line holding entry w1 - 1
        const int64_t fa =
            std::upper_bound(ptr.begin() + r0, ptr.begin() + r1 + 1, (int32_t)w0) - ptr.begin() - 1;
        const int64_t la = std::upper_bound(ptr.begin() + r0, ptr.begin() + r1 + 1,
                                            (int32_t)(w1 - 1)) -
                           ptr.begin() - 1;
        first = (int)fa;
        n = (int)(la - fa + 1);
      }
      part[(size_t)c * 32 + w] = make_int4((int)w0, (int)w1, first, n);
      *lines_max = std::max(*lines_max, n);
    }
    part[(size_t)c * 32 + kConsumers] = make_int4((int)r0, (int)r1, 0, 0);
    r0 = r1;
  }
}

}  // namespace snack
