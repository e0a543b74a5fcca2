// Column-panel SDDMM: the backward-weight product dW[k] = sum_b dY[b][row_k]
// X[b][col_k] with X^T staged in shared memory panel by panel, for batch
// slices of 8-64 floats on layers whose rows are long.
//
// The segment kernels gather every entry's X^T row (32-256 bytes) through
// L1.  Here each CTA (one per SM, 768 threads) sweeps X^T [in][BW] through
// shared memory in column panels of PW = 64 KB / (4 BW) lines, three panels
// resident at a time:
//
//  * warp 23 is the producer: its lane 0 copies panel p into stage p % 3
//    with cp.async.bulk (completion on that stage's "full" mbarrier) once
//    all 23 consumer warps have released the panel that stage held (its
//    "empty" mbarrier).  Every wait is bounded; a wait that gives up sets
//    the layer's device error flag and the CTA winds down.
//  * each consumer warp owns a contiguous range of the row-ordered entry
//    stream (the CTA's rows are a row-aligned, entry-balanced share of the
//    table; its 23 warps split that share evenly, at most four rows each).
//    Entries of a row are sorted by column, so the part of a row that falls
//    in panel p is one run of consecutive entries; a table built with the
//    topology holds every row's run offsets for every panel.  For each
//    resident panel the warp walks its rows' runs in steps of two quads (4
//    entries each) per group of G lanes, gathering X^T rows from shared
//    memory; the rows' dY slices stay in registers, and each entry's dot
//    product is finished by a butterfly over its group and stored.  Every
//    step's address is known in advance (the next quads of the run, or the
//    first of the next non-empty run, in this panel or the next), so the
//    next step's index loads are always in flight.
//
// It pays when a row's run per panel is long (a step covers 64 / 32 / 16 /
// 16 entries at slices of 8 / 16 / 32 / 64): measured on GB300 against the
// segment SDDMM, 10000 x 10000 at 90 % (1000 entries per row) batch 8 / 16 /
// 32: 41.5 / 63.9 / 118.3 us vs 48.3 / 71.2 / 123.5; at 95 % batch 8: 27.9
// vs 31.3, batch 16: 43.0 vs 41.5.  The launcher takes it when the mean run
// per panel is at least 64 entries.  (The same sweep for the forward and dX
// products measured slower than the segment kernels at every width.)
//
// The index stream of the warp's range is asked into L2 at the start
// (cp.async.bulk.prefetch.L2, before the wait on the producing transpose):
// the sweep reads each row's runs panel by panel, not in one pass, and L2
// hits keep those short runs cheap.
#include <algorithm>
#include <cstdlib>
#include <map>
#include <mutex>
#include <utility>

#include "spmm_dispatch.cuh"

namespace snack {

namespace {

constexpr int kPanelThreads = 768;
constexpr int kConsumers = 23;          // warps 0-22 consume, warp 23 produces
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

template <int BW>
__host__ __device__ constexpr int panel_lines() {
  return kStageBytes / (4 * BW);
}

// Batch-slice shape of the panel kernels: G lanes per entry, each holding
// NV 16-byte vectors of the row, QPS quads (4 entries each) per group per
// step.  A warp's shared-memory gathers cost the most bank conflicts when a
// lane reads part of a short row, so rows of up to 128 bytes are read whole
// by one instruction of their group (G = BW / 4), and the per-step work of
// a lane (stream loads, masks, addresses) is spread over two quads instead;
// 64-float rows are read as two 128-byte halves (one vector per lane each,
// conflict-free), one quad per step.
template <int BW>
struct PanelShape {
  static constexpr int VEC = 4, NV = BW == 64 ? 2 : 1, G = BW == 64 ? 8 : BW / 4;
  static constexpr int QPS = BW == 64 ? 1 : 2;
};

// Operand indices of one quad (entries kb..kb+3).
__device__ __forceinline__ void panel_quad(const PanelArgs &a, int kb, int (&c)[4]) {
  const int4 c4 = ld_stream_i4(a.idx + kb);
  c[0] = c4.x;
  c[1] = c4.y;
  c[2] = c4.z;
  c[3] = c4.w;
}

// dW of one quad: d[e] holds each lane's part of entry e's dot product
// (its 4 floats of the batch).  A butterfly over the G lanes of the group
// sums and spreads at once: the first level leaves each lane two of the four
// entries, the second one, and the remaining levels finish the sum; with
// G = 2 / 4 / 8 / 16 the group spends 2 / 3 / 4 / 5 shuffles on its four
// entries, and lane sub ends with entry (sub / (G / 4)) when G >= 4 (of
// those, the lanes with sub % (G / 4) == 0 store it), or, for G = 2, with
// entries 2 sub and 2 sub + 1.  With G = 1 the lane has the sums already.
template <int G>
__device__ __forceinline__ void panel_dw_store(const PanelArgs &a, int kb, int sub,
                                               const bool (&t)[4], float (&d)[4]) {
  const unsigned m = 0xffffffffu;
  if constexpr (G == 1) {  // the lane holds whole dot products
    float *dst = a.dw + kb;
    if (t[0] && t[1] && t[2] && t[3]) {
      float4 o = make_float4(d[0], d[1], d[2], d[3]);
      if (a.accumulate) {
        const float4 old = *reinterpret_cast<const float4 *>(dst);
        o.x += old.x;
        o.y += old.y;
        o.z += old.z;
        o.w += old.w;
      }
      *reinterpret_cast<float4 *>(dst) = o;
    } else {
#pragma unroll
      for (int e = 0; e < 4; ++e)
        if (t[e]) dst[e] = a.accumulate ? dst[e] + d[e] : d[e];
    }
    return;
  } else {
  const bool up = (sub & (G / 2)) != 0;  // level 1: keep entries 2-3 (up) or 0-1
  const float s0 = __shfl_xor_sync(m, up ? d[0] : d[2], G / 2);
  const float s1 = __shfl_xor_sync(m, up ? d[1] : d[3], G / 2);
  d[0] = (up ? d[2] : d[0]) + s0;
  d[1] = (up ? d[3] : d[1]) + s1;
  const int base = up ? 2 : 0;
  if constexpr (G == 2) {
#pragma unroll
    for (int e = 0; e < 2; ++e)
      if (t[base + e]) {
        float *dst = a.dw + kb + base + e;
        *dst = a.accumulate ? *dst + d[e] : d[e];
      }
  } else {
    const bool up2 = (sub & (G / 4)) != 0;  // level 2: keep one entry
    d[0] = (up2 ? d[1] : d[0]) + __shfl_xor_sync(m, up2 ? d[0] : d[1], G / 4);
#pragma unroll
    for (int off = G / 8; off >= 1; off >>= 1) d[0] += __shfl_xor_sync(m, d[0], off);
    const int e = base + (up2 ? 1 : 0);
    if ((sub & (G / 4 - 1)) == 0 && t[e]) {
      float *dst = a.dw + kb + e;
      *dst = a.accumulate ? *dst + d[0] : d[0];
    }
  }
  }
}

template <int BW, int RW>
__global__ void __launch_bounds__(kPanelThreads, 1) panel_sddmm(const PanelArgs a) {
  using S = PanelShape<BW>;
  constexpr int VEC = S::VEC, NV = S::NV, G = S::G, QPS = S::QPS;
  constexpr int PW = panel_lines<BW>();
  static_assert(PW * BW * 4 == kStageBytes, "panel size");

  extern __shared__ __align__(128) float smem_f[];
  float *stage = smem_f;  // [kStages][PW][BW]
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
  // The warp's index stream is immutable here: ask L2 for it while the
  // producing transpose may still run.
  if (warp < kConsumers && lane == 0) {
    const int4 me = part[warp];
    const int k0 = me.x & ~3, k1 = (me.y + 3) & ~3;
    if (k1 > k0) l2_prefetch(a.idx + k0, (uint32_t)(k1 - k0) * 4);
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
  constexpr int NPT = 32 / G;            // groups per warp
  constexpr int STEP = 4 * NPT * QPS;    // entries per warp step
  const int4 me = part[warp];
  const int W0 = me.x, W1 = me.y, first = me.z, nl = me.w;
  // Run offsets of row j (lane j < nl holds them): lo = its first entry in
  // panel p, hi = first entry in panel p + 1, hh = in panel p + 2.
  const bool holder = lane < nl;
  const int32_t *offl = a.off + first + lane;
  int lo = 0, hi = 0, hh = 0;
  if (holder) {
    lo = offl[0];
    hi = npanels >= 1 ? offl[(int64_t)a.lines] : lo;
  }
  float dy[RW][NV][VEC];  // each row's dY slice (the lane's part of the batch)
#pragma unroll
  for (int j = 0; j < RW; ++j) {
#pragma unroll
    for (int v = 0; v < NV; ++v)
#pragma unroll
      for (int i = 0; i < VEC; ++i) dy[j][v][i] = 0.f;
    if (j < nl) {
      const float *p = a.dyt + (int64_t)(first + j) * BW + sub * VEC;
#pragma unroll
      for (int v = 0; v < NV; ++v) load_vec<VEC>(p + v * G * VEC, dy[j][v]);
    }
  }

  // The quads of the step based at pre (a multiple of 4), loaded ahead: this
  // group's quad q starts at pre + 4 grp + 4 NPT q.
  int pre = -1;
  int c[QPS][4] = {};
  bool ok = true;
  for (int p = 0; p < npanels && ok; ++p) {
    const int s = p % kStages;
    // the offsets closing panel p + 1: used by the look-ahead at the end of
    // this panel, loaded now
    if (holder && p + 2 <= npanels) hh = offl[(int64_t)(p + 2) * a.lines];
    ok = bar_wait(&full[s], (uint32_t)((p / kStages) & 1));
    if (!ok) {
      if (lane == 0) atomicOr(a.err, 1);
      break;
    }
    const float *st = stage + (size_t)s * PW * BW + sub * VEC - (int64_t)p * PW * BW;
#pragma unroll
    for (int j = 0; j < RW; ++j) {
      if (j >= nl) continue;  // warp-uniform
      const int ra = max(__shfl_sync(0xffffffffu, lo, j), W0);
      const int rb = min(__shfl_sync(0xffffffffu, hi, j), W1);
      for (int kb0 = ra & ~3; kb0 < rb; kb0 += STEP) {  // warp-uniform
        const int kb = kb0 + 4 * grp;
        if (pre != kb0) {
#pragma unroll
          for (int q = 0; q < QPS; ++q)
            if (kb + 4 * NPT * q < rb) panel_quad(a, kb + 4 * NPT * q, c[q]);
        }
        // the next step: further along this run, or the first step of the
        // next non-empty run (later rows of this panel, then the next panel)
        int nk = -1, nb = 0;
        if (kb0 + STEP < rb) {
          nk = kb0 + STEP;
          nb = rb;
        } else {
          for (int jj = j + 1; jj < nl; ++jj) {
            const int xa = max(__shfl_sync(0xffffffffu, lo, jj), W0);
            const int xb = min(__shfl_sync(0xffffffffu, hi, jj), W1);
            if (xb > xa) {
              nk = xa & ~3;
              nb = xb;
              break;
            }
          }
          if (nk < 0 && p + 1 < npanels) {
            for (int jj = 0; jj < nl; ++jj) {
              const int xa = max(__shfl_sync(0xffffffffu, hi, jj), W0);
              const int xb = min(__shfl_sync(0xffffffffu, hh, jj), W1);
              if (xb > xa) {
                nk = xa & ~3;
                nb = xb;
                break;
              }
            }
          }
        }
        int cn[QPS][4] = {};
        if (nk >= 0) {
#pragma unroll
          for (int q = 0; q < QPS; ++q) {
            const int kq = nk + 4 * grp + 4 * NPT * q;
            if (kq < nb) panel_quad(a, kq, cn[q]);
          }
        }

#pragma unroll
        for (int q = 0; q < QPS; ++q) {
          const int kq = kb + 4 * NPT * q;
          bool t[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) t[e] = kq + e >= ra && kq + e < rb;
          float d[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            float x[NV][VEC];
            float dot = 0.f;
            if (t[e]) {
#pragma unroll
              for (int v = 0; v < NV; ++v) load_op<VEC, true>(st + c[q][e] * BW + v * G * VEC, x[v]);
#pragma unroll
              for (int v = 0; v < NV; ++v)
#pragma unroll
                for (int i = 0; i < VEC; ++i) dot = fmaf(dy[j][v][i], x[v][i], dot);
            }
            d[e] = dot;
          }
          panel_dw_store<G>(a, kq, sub, t, d);
        }
        pre = nk;
#pragma unroll
        for (int q = 0; q < QPS; ++q)
#pragma unroll
          for (int e = 0; e < 4; ++e) c[q][e] = cn[q][e];
      }
    }
    __syncwarp();
    if (lane == 0) bar_arrive(&empty[s]);
    lo = hi;
    hi = hh;
  }
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

namespace {
int width_index(int bw) { return bw == 8 ? 0 : bw == 16 ? 1 : bw == 32 ? 2 : 3; }
int width_of(int i) { return 8 << i; }
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

bool panel_fits(const PanelTable &t, int bw, double mean_len, int64_t n_op) {
  if (t.d_part == nullptr || t.lines_max > kPanelLinesPerWarp ||
      !(bw == 8 || bw == 16 || bw == 32 || bw == 64) || t.d_off[width_index(bw)] == nullptr)
    return false;
  // mean entries of a row per panel: the sweep pays only on long runs
  const double pw = (double)(kStageBytes / (4 * bw));
  return mean_len * pw / (double)n_op >= 64.0;
}

namespace {
// off[p][l] = first entry of line l (entries ptr[l] .. ptr[l+1], sorted by
// operand index) whose operand index is at least p * pw.
__global__ void panel_offsets(const int32_t *__restrict__ ptr, const int32_t *__restrict__ idx,
                              int64_t lines, int npan, int pw, int32_t *__restrict__ off) {
  const int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (t >= lines * (int64_t)(npan + 1)) return;
  const int p = (int)(t / lines);
  const int64_t l = t - (int64_t)p * lines;
  int lo = ptr[l], hi = ptr[l + 1];
  if (p == 0) {
    off[t] = lo;
    return;
  }
  if (p == npan) {
    off[t] = hi;
    return;
  }
  const int key = p * pw;
  while (lo < hi) {
    const int mid = lo + (hi - lo) / 2;
    if (idx[mid] < key) lo = mid + 1;
    else hi = mid;
  }
  off[t] = lo;
}
}  // namespace

cudaError_t build_panel_offsets(PanelTable &t, const int32_t *ptr, const int32_t *idx,
                                int64_t lines, int64_t n_op, size_t *acct, cudaStream_t s) {
  for (int i = 0; i < kPanelWidths; ++i) {
    const int pw = kStageBytes / (4 * width_of(i));
    const int64_t npan = (n_op + pw - 1) / pw;
    const int64_t n = lines * (npan + 1);
    cudaError_t e = dev_alloc(&t.d_off[i], (size_t)n, acct);
    t.bytes += (size_t)n * 4;
    if (e != cudaSuccess) return e;
    panel_offsets<<<(unsigned)((n + 255) / 256), 256, 0, s>>>(ptr, idx, lines, (int)npan, pw,
                                                              t.d_off[i]);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  return cudaSuccess;
}

void free_panel_table(PanelTable &t) {
  if (t.d_part) cudaFree(t.d_part);
  for (int32_t *&p : t.d_off)
    if (p) cudaFree(p);
  t = PanelTable();
}

cudaError_t launch_panel_sddmm(int bw, const PanelTable &t, const PanelArgs &args, bool pdl,
                               cudaStream_t s) {
  PanelArgs a = args;
  a.part = t.d_part;
  a.off = t.d_off[width_index(bw)];
  a.lines = t.lines;
  const size_t smem = (size_t)kStages * kStageBytes;
#define SNACK_PANEL(W) \
  case W:              \
    return launch_panel_kernel(panel_sddmm<W, kPanelLinesPerWarp>, a, t.ctas, smem, pdl, s);
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
// CTAs take row-aligned shares of about nnz / ctas entries; each CTA's
// consumer warps split its share evenly, except that a warp's range is cut
// at the start of its (kPanelLinesPerWarp + 1)-th line (the next warps take
// the rest).  Per CTA 32 int4: one per consumer warp {first entry, end
// entry, first line, lines}, then {first line, end line} of the CTA.
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
    int64_t w0 = e0;
    for (int w = 0; w < kConsumers; ++w) {
      // ideal end of the warp's share; cut earlier if the range would cover
      // more lines than a warp holds (the following warps take the rest)
      int64_t w1 = w + 1 == kConsumers ? e1 : e0 + (e1 - e0) * (w + 1) / kConsumers;
      if (w1 < w0) w1 = w0;
      int first = (int)r0, n = 0;
      if (w1 > w0) {
        // line holding entry w0 (the last line starting at or before it
        // whose range is not empty)
        const int64_t fa =
            std::upper_bound(ptr.begin() + r0, ptr.begin() + r1 + 1, (int32_t)w0) - ptr.begin() - 1;
        if (fa + kPanelLinesPerWarp < r1 && ptr[fa + kPanelLinesPerWarp] < w1 &&
            w + 1 < kConsumers)
          w1 = ptr[fa + kPanelLinesPerWarp];
        const int64_t la = std::upper_bound(ptr.begin() + r0, ptr.begin() + r1 + 1,
                                            (int32_t)(w1 - 1)) -
                           ptr.begin() - 1;
        first = (int)fa;
        n = (int)(la - fa + 1);
      }
      part[(size_t)c * 32 + w] = make_int4((int)w0, (int)w1, first, n);
      *lines_max = std::max(*lines_max, n);
      w0 = w1;
    }
    part[(size_t)c * 32 + kConsumers] = make_int4((int)r0, (int)r1, 0, 0);
    r0 = r1;
  }
}

}  // namespace snack
