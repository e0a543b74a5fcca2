// Topology work of the SNACK layer, all on the device: canonical order, the
// CSR / CSC segmentations (Appendix B, Table 7), the work decomposition into
// segments, the uniform connection initializer (§3.3 Algorithm 2) and the
// magnitude-prune / uniform-regrow step (Appendix G).
//
// Building blocks written here: a stable LSD radix sort of (u64 key, u32
// payload) pairs (8-bit digits; per tile a digit histogram, one exclusive
// scan over the digit-major histogram table, then a stable scatter that
// ranks equal digits with warp match masks) and a multi-level exclusive scan.
// These run once per topology change, never per training step; they may
// allocate temporaries and synchronise the stream.
#include <algorithm>
#include <utility>
#include <climits>
#include <cmath>
#include <cstring>
#include <vector>

#include "snack_internal.cuh"

namespace snack {
namespace {

#define TRY_CUDA(expr)                                                 \
  do {                                                                 \
    cudaError_t e_ = (expr);                                           \
    if (e_ != cudaSuccess) {                                           \
      err = std::string(#expr) + ": " + cudaGetErrorString(e_);        \
      return e_ == cudaErrorMemoryAllocation ? SNACK_ERR_ALLOC : SNACK_ERR_CUDA; \
    }                                                                  \
  } while (0)

// RAII bag of temporary device buffers.
struct Temps {
  std::vector<void *> ptrs;
  ~Temps() {
    for (void *p : ptrs) cudaFree(p);
  }
  template <typename T>
  cudaError_t get(T **p, size_t count) {
    size_t bytes = std::max<size_t>(count * sizeof(T), 16);
    cudaError_t e = device_malloc(reinterpret_cast<void **>(p), bytes);
    if (e == cudaSuccess) ptrs.push_back(*p);
    return e;
  }
};

inline unsigned grid_for(int64_t n, int threads) {
  return (unsigned)std::max<int64_t>(1, (n + threads - 1) / threads);
}

// ---------------------------------------------------------------- scan ----

constexpr int kScanThreads = 1024;
constexpr int kScanItems = 4;
constexpr int kScanTile = kScanThreads * kScanItems;

__device__ __forceinline__ int block_exclusive_sum(int x, int *total) {
  __shared__ int warp_tot[32];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int incl = x;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) warp_tot[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    const int nw = blockDim.x >> 5;
    int w = lane < nw ? warp_tot[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    warp_tot[lane] = w;  // inclusive over warps
  }
  __syncthreads();
  const int before = warp == 0 ? 0 : warp_tot[warp - 1];
  *total = warp_tot[(blockDim.x >> 5) - 1];
  __syncthreads();
  return before + incl - x;
}

__global__ void __launch_bounds__(kScanThreads) scan_tile_sums(const int *in, int64_t n, int *sums) {
  const int64_t base = (int64_t)blockIdx.x * kScanTile + (int64_t)threadIdx.x * kScanItems;
  int s = 0;
#pragma unroll
  for (int i = 0; i < kScanItems; ++i)
    if (base + i < n) s += in[base + i];
  int total;
  block_exclusive_sum(s, &total);
  if (threadIdx.x == 0) sums[blockIdx.x] = total;
}

__global__ void __launch_bounds__(kScanThreads) scan_tiles(const int *in, int *out, int64_t n,
                                                           const int *tile_off) {
  const int64_t base = (int64_t)blockIdx.x * kScanTile + (int64_t)threadIdx.x * kScanItems;
  int v[kScanItems];
  int s = 0;
#pragma unroll
  for (int i = 0; i < kScanItems; ++i) {
    v[i] = base + i < n ? in[base + i] : 0;
    s += v[i];
  }
  int total;
  int run = block_exclusive_sum(s, &total) + (tile_off ? tile_off[blockIdx.x] : 0);
#pragma unroll
  for (int i = 0; i < kScanItems; ++i) {
    if (base + i < n) out[base + i] = run;
    run += v[i];
  }
}

snack_status exclusive_scan(const int *in, int *out, int64_t n, cudaStream_t s, std::string &err) {
  if (n <= 0) return SNACK_OK;
  const int64_t tiles = (n + kScanTile - 1) / kScanTile;
  if (tiles == 1) {
    scan_tiles<<<1, kScanThreads, 0, s>>>(in, out, n, nullptr);
    TRY_CUDA(cudaGetLastError());
    return SNACK_OK;
  }
  Temps t;
  int *sums = nullptr, *offs = nullptr;
  TRY_CUDA(t.get(&sums, tiles));
  TRY_CUDA(t.get(&offs, tiles));
  scan_tile_sums<<<(unsigned)tiles, kScanThreads, 0, s>>>(in, n, sums);
  TRY_CUDA(cudaGetLastError());
  snack_status st = exclusive_scan(sums, offs, tiles, s, err);
  if (st != SNACK_OK) return st;
  scan_tiles<<<(unsigned)tiles, kScanThreads, 0, s>>>(in, out, n, offs);
  TRY_CUDA(cudaGetLastError());
  TRY_CUDA(cudaStreamSynchronize(s));  // temporaries are freed on return
  return SNACK_OK;
}

// ---------------------------------------------------------- radix sort ----

constexpr int kSortThreads = 256;
constexpr int kSortRounds = 16;
constexpr int kSortTile = kSortThreads * kSortRounds;

__global__ void __launch_bounds__(kSortThreads)
radix_hist(const uint64_t *keys, int64_t n, int shift, int *hist, int64_t nblocks) {
  __shared__ int h[256];
  h[threadIdx.x] = 0;
  __syncthreads();
  const int64_t base = (int64_t)blockIdx.x * kSortTile;
#pragma unroll 4
  for (int r = 0; r < kSortRounds; ++r) {
    const int64_t i = base + r * kSortThreads + threadIdx.x;
    if (i < n) atomicAdd(&h[(keys[i] >> shift) & 255u], 1);
  }
  __syncthreads();
  hist[(int64_t)threadIdx.x * nblocks + blockIdx.x] = h[threadIdx.x];
}

__global__ void __launch_bounds__(kSortThreads)
radix_scatter(const uint64_t *kin, const uint32_t *vin, uint64_t *kout, uint32_t *vout, int64_t n,
              int shift, const int *offs, int64_t nblocks) {
  __shared__ int base[256];
  __shared__ int wcount[kSortThreads / 32][256];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  base[threadIdx.x] = offs[(int64_t)threadIdx.x * nblocks + blockIdx.x];
  const unsigned lt = (1u << lane) - 1u;
  const int64_t tile = (int64_t)blockIdx.x * kSortTile;
  for (int r = 0; r < kSortRounds; ++r) {
    const int64_t i = tile + r * kSortThreads + threadIdx.x;
    const bool valid = i < n;
    uint64_t key = 0;
    uint32_t val = 0;
    int d = 256;  // invalid lanes share a sentinel digit
    if (valid) {
      key = kin[i];
      val = vin[i];
      d = (int)((key >> shift) & 255u);
    }
#pragma unroll
    for (int w = 0; w < kSortThreads / 32; ++w) wcount[w][threadIdx.x] = 0;
    __syncthreads();
    const unsigned peers = __match_any_sync(0xffffffffu, d);
    const int rank = __popc(peers & lt);
    if (valid && rank == 0) wcount[warp][d] = __popc(peers);
    __syncthreads();
    {
      int run = base[threadIdx.x];
#pragma unroll
      for (int w = 0; w < kSortThreads / 32; ++w) {
        const int c = wcount[w][threadIdx.x];
        wcount[w][threadIdx.x] = run;
        run += c;
      }
      base[threadIdx.x] = run;
    }
    __syncthreads();
    if (valid) {
      const int pos = wcount[warp][d] + rank;
      kout[pos] = key;
      vout[pos] = val;
    }
    __syncthreads();
  }
}

int bits_for(uint64_t max_key) {
  int b = 0;
  while (b < 64 && (max_key >> b) != 0) ++b;
  return b;
}

// Stable sort of (key, val) by the low `nbits` bits of key.  The result ends
// in (*k, *v); the other pair of buffers is scratch.
snack_status radix_sort(uint64_t **k, uint32_t **v, uint64_t **k_alt, uint32_t **v_alt, int64_t n,
                        int nbits, cudaStream_t s, std::string &err) {
  if (n <= 1 || nbits <= 0) return SNACK_OK;
  const int64_t nblocks = (n + kSortTile - 1) / kSortTile;
  if (nblocks * 256 > INT_MAX) {
    err = "radix sort: too many entries";
    return SNACK_ERR_UNSUPPORTED;
  }
  Temps t;
  int *hist = nullptr, *offs = nullptr;
  TRY_CUDA(t.get(&hist, nblocks * 256));
  TRY_CUDA(t.get(&offs, nblocks * 256));
  for (int shift = 0; shift < nbits; shift += 8) {
    radix_hist<<<(unsigned)nblocks, kSortThreads, 0, s>>>(*k, n, shift, hist, nblocks);
    TRY_CUDA(cudaGetLastError());
    snack_status st = exclusive_scan(hist, offs, nblocks * 256, s, err);
    if (st != SNACK_OK) return st;
    radix_scatter<<<(unsigned)nblocks, kSortThreads, 0, s>>>(*k, *v, *k_alt, *v_alt, n, shift, offs,
                                                            nblocks);
    TRY_CUDA(cudaGetLastError());
    std::swap(*k, *k_alt);
    std::swap(*v, *v_alt);
  }
  TRY_CUDA(cudaStreamSynchronize(s));
  return SNACK_OK;
}

// ------------------------------------------------ canonical order, CSR/CSC --

__global__ void make_cell_keys(const int32_t *row, const int32_t *col, int64_t n, int64_t out,
                               int64_t in, uint64_t *key, uint32_t *idx,
                               unsigned long long *bad) {
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n) return;
  const int64_t r = row[i], c = col[i];
  if (r < 0 || r >= out || c < 0 || c >= in) {
    atomicMin(bad, (unsigned long long)i);
    key[i] = 0;
  } else {
    key[i] = (uint64_t)r * (uint64_t)in + (uint64_t)c;
  }
  idx[i] = (uint32_t)i;
}

__global__ void finish_canonical(const uint64_t *key, const uint32_t *src, int64_t n, int64_t in,
                                 const float *val_src, int32_t *row, int32_t *col, float *val,
                                 unsigned long long *dup) {
  const int64_t k = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (k >= n) return;
  const uint64_t c = key[k];
  if (k > 0 && key[k - 1] == c) atomicMin(dup, (unsigned long long)src[k]);
  row[k] = (int32_t)(c / (uint64_t)in);
  col[k] = (int32_t)(c % (uint64_t)in);
  val[k] = val_src ? val_src[src[k]] : 0.f;
}

// ptr[l] = first position whose key >= l * stride (keys sorted), l in [0, nlines].
__global__ void line_offsets(const uint64_t *key, int64_t n, int64_t nlines, uint64_t stride,
                             int32_t *ptr) {
  const int64_t l = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (l > nlines) return;
  const uint64_t target = (uint64_t)l * stride;
  int64_t lo = 0, hi = n;
  while (lo < hi) {
    const int64_t mid = (lo + hi) >> 1;
    if (key[mid] < target)
      lo = mid + 1;
    else
      hi = mid;
  }
  ptr[l] = (int32_t)lo;
}

__global__ void make_csc_keys(const int32_t *row, const int32_t *col, int64_t n, int64_t out,
                              uint64_t *key, uint32_t *idx) {
  const int64_t k = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (k >= n) return;
  key[k] = (uint64_t)col[k] * (uint64_t)out + (uint64_t)row[k];
  idx[k] = (uint32_t)k;
}

__global__ void gather_by_perm(const int32_t *perm, const float *val, int64_t n, float *out) {
  const int64_t s = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (s < n) out[s] = val[perm[s]];
}

__global__ void finish_csc(const uint64_t *key, const uint32_t *src, int64_t n, int64_t out,
                           int32_t *csc_row, int32_t *csc_perm) {
  const int64_t s = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (s >= n) return;
  csc_row[s] = (int32_t)(key[s] % (uint64_t)out);
  csc_perm[s] = (int32_t)src[s];
}

// Host: cut lines into segments of at most `cap` entries (balanced parts).
// Lines up to max(256, 2 x mean) entries stay whole.  On a heavy-tailed
// table (longest line over 8 x the mean) the cap is instead about the
// entries one resident team gets on average (nnz / (32 x SMs), kept in
// [64, 256]): the longest parts otherwise outlast the other teams (8192 x
// 8192 Zipf rows, batch 16: 23.0 us with 256-entry parts, 21.8 us with 138;
// parts of 64 / 96 / 112 / 192 entries measured 29.8 / 27.0 / 24.0 / 22.1
// us, the combines and a second wave of teams of the shorter parts costing
// more than the balance gained.  Emitting the segments longest line first
// and dealing them to the teams in snake order across rounds measured
// 22.6-25.0 us at those part sizes and was not kept).
void build_segments(const std::vector<int32_t> &ptr, int64_t nlines, int64_t nnz,
                    std::vector<int4> &seg, std::vector<int4> &split, SegTable &t) {
  seg.clear();
  split.clear();
  t.mean_len = nlines > 0 ? (double)nnz / (double)nlines : 0.0;
  t.max_len = 0;
  t.max_parts = 0;
  for (int64_t l = 0; l < nlines; ++l) t.max_len = std::max<int64_t>(t.max_len, ptr[l + 1] - ptr[l]);
  int64_t cap = std::max<int64_t>(256, 2 * (int64_t)std::ceil(t.mean_len));
  if ((double)t.max_len > 8.0 * t.mean_len)
    cap = std::min<int64_t>(256, std::max<int64_t>(64, nnz / (32 * (int64_t)device_sms())));
  int64_t slots = 0;
  for (int64_t l = 0; l < nlines; ++l) {
    const int64_t b = ptr[l], e = ptr[l + 1], len = e - b;
    const int64_t parts = len > cap ? (len + cap - 1) / cap : 1;
    if (parts == 1) {
      seg.push_back(make_int4((int)l, (int)b, (int)e, -1));
      continue;
    }
    const int sid = (int)split.size();
    split.push_back(make_int4((int)seg.size(), (int)parts, (int)slots, 0));
    slots += parts;
    t.max_parts = std::max<int>(t.max_parts, (int)parts);
    for (int64_t p = 0; p < parts; ++p)
      seg.push_back(make_int4((int)l, (int)(b + p * len / parts), (int)(b + (p + 1) * len / parts),
                              sid));
  }
  t.nseg = (int64_t)seg.size();
  t.nsplit = (int64_t)split.size();
  t.nslots = slots;
}

// Host: every line of `parts` or more entries cut into that many balanced
// parts (a split line each), the others kept whole.
void build_cut(const std::vector<int32_t> &ptr, int64_t nlines, int64_t nnz, int parts,
               std::vector<int4> &seg, std::vector<int4> &split, SegTable &t) {
  seg.clear();
  split.clear();
  t.mean_len = nlines > 0 ? (double)nnz / (double)nlines : 0.0;
  t.max_len = 0;
  t.max_parts = 0;
  int64_t slots = 0;
  for (int64_t l = 0; l < nlines; ++l) {
    const int64_t b = ptr[l], e = ptr[l + 1], len = e - b;
    t.max_len = std::max<int64_t>(t.max_len, len);
    if (len < parts) {
      seg.push_back(make_int4((int)l, (int)b, (int)e, -1));
      continue;
    }
    const int sid = (int)split.size();
    split.push_back(make_int4((int)seg.size(), parts, (int)slots, 0));
    slots += parts;
    t.max_parts = std::max(t.max_parts, parts);
    for (int q = 0; q < parts; ++q)
      seg.push_back(make_int4((int)l, (int)(b + q * len / parts), (int)(b + (q + 1) * len / parts),
                              sid));
  }
  t.nseg = (int64_t)seg.size();
  t.nsplit = (int64_t)split.size();
  t.nslots = slots;
}

// Whether table t gets its cut copies (halves and quarters): a large layer
// (2^21+ entries) of long, evenly filled lines.  Measured on 10000 x 10000
// at 90 % (1000 entries per line), 64-wide slices, forward 182 us with whole
// lines, 159 / 148 / 144 / 146 with 2 / 3 / 4 / 5 parts; dW 187 -> 166 /
// 157 / 151 / 149 (the fifth part lost on the forward and on the 95 %
// layer).  Which slices walk which copy is decided per product at launch
// (the SpMMs' combines cost more than they save on narrow slices: batch 8
// forward 44 -> 63 us with halves).
bool halves_pay(const SegTable &t, int64_t nnz) {
  return nnz >= (int64_t(1) << 21) && t.mean_len >= 400.0 && (double)t.max_len <= 8.0 * t.mean_len;
}

void free_segments(SegTable &t) {
  if (t.d_seg) cudaFree(t.d_seg);
  if (t.d_split) cudaFree(t.d_split);
  free_panel_table(t.panel);
  t = SegTable();
}

snack_status upload_segments(const std::vector<int4> &seg, const std::vector<int4> &split,
                             SegTable &t, size_t *acct, cudaStream_t s, std::string &err) {
  if (t.d_seg) cudaFree(t.d_seg);
  if (t.d_split) cudaFree(t.d_split);
  t.d_seg = nullptr;
  t.d_split = nullptr;
  TRY_CUDA(dev_alloc(&t.d_seg, seg.size(), acct));
  TRY_CUDA(dev_alloc(&t.d_split, split.size(), acct));
  // Stream-ordered copies, then wait: the host vectors die on return and the
  // caller's stream may not be ordered with the legacy default stream.
  if (!seg.empty())
    TRY_CUDA(cudaMemcpyAsync(t.d_seg, seg.data(), seg.size() * sizeof(int4),
                             cudaMemcpyHostToDevice, s));
  if (!split.empty())
    TRY_CUDA(cudaMemcpyAsync(t.d_split, split.data(), split.size() * sizeof(int4),
                             cudaMemcpyHostToDevice, s));
  TRY_CUDA(cudaStreamSynchronize(s));
  return SNACK_OK;
}

// Given canonical d_row/d_col (and sorted cell keys), build row_ptr, the CSC
// arrays, both segment tables and the split workspace.
snack_status finish_layout(Layer &L, const uint64_t *d_cell_key, cudaStream_t s, std::string &err) {
  const int64_t n = L.nnz;
  line_offsets<<<grid_for(L.out + 1, 256), 256, 0, s>>>(d_cell_key, n, L.out, (uint64_t)L.in,
                                                        L.d_row_ptr);
  TRY_CUDA(cudaGetLastError());
  {
    Temps t;
    uint64_t *ka, *kb;
    uint32_t *va, *vb;
    TRY_CUDA(t.get(&ka, n));
    TRY_CUDA(t.get(&kb, n));
    TRY_CUDA(t.get(&va, n));
    TRY_CUDA(t.get(&vb, n));
    if (n > 0) {
      make_csc_keys<<<grid_for(n, 256), 256, 0, s>>>(L.d_row, L.d_col, n, L.out, ka, va);
      TRY_CUDA(cudaGetLastError());
    }
    const uint64_t cells = (uint64_t)L.out * (uint64_t)L.in;
    snack_status st = radix_sort(&ka, &va, &kb, &vb, n, bits_for(cells - 1), s, err);
    if (st != SNACK_OK) return st;
    if (n > 0) {
      finish_csc<<<grid_for(n, 256), 256, 0, s>>>(ka, va, n, L.out, L.d_csc_row, L.d_csc_perm);
      TRY_CUDA(cudaGetLastError());
    }
    line_offsets<<<grid_for(L.in + 1, 256), 256, 0, s>>>(ka, n, L.in, (uint64_t)L.out, L.d_col_ptr);
    TRY_CUDA(cudaGetLastError());
    TRY_CUDA(cudaStreamSynchronize(s));
  }
  {
    snack_status st = refresh_csc_values(L, s, err);
    if (st != SNACK_OK) return st;
  }
  std::vector<int32_t> rp(L.out + 1), cp(L.in + 1);
  TRY_CUDA(cudaMemcpyAsync(rp.data(), L.d_row_ptr, rp.size() * 4, cudaMemcpyDeviceToHost, s));
  TRY_CUDA(cudaMemcpyAsync(cp.data(), L.d_col_ptr, cp.size() * 4, cudaMemcpyDeviceToHost, s));
  TRY_CUDA(cudaStreamSynchronize(s));
  std::vector<int4> seg, split;
  build_segments(rp, L.out, n, seg, split, L.csr);
  snack_status st = upload_segments(seg, split, L.csr, &L.device_bytes, s, err);
  if (st != SNACK_OK) return st;
  build_segments(cp, L.in, n, seg, split, L.csc);
  st = upload_segments(seg, split, L.csc, &L.device_bytes, s, err);
  if (st != SNACK_OK) return st;
  for (SegTable *t : {&L.csr_half, &L.csc_half, &L.csr_wide, &L.csc_wide}) free_segments(*t);
  for (int parts : {2, kWideCutParts}) {
    if (halves_pay(L.csr, n)) {
      SegTable &t = parts == 2 ? L.csr_half : L.csr_wide;
      build_cut(rp, L.out, n, parts, seg, split, t);
      st = upload_segments(seg, split, t, &L.device_bytes, s, err);
      if (st != SNACK_OK) return st;
    }
    if (halves_pay(L.csc, n)) {
      SegTable &t = parts == 2 ? L.csc_half : L.csc_wide;
      build_cut(cp, L.in, n, parts, seg, split, t);
      st = upload_segments(seg, split, t, &L.device_bytes, s, err);
      if (st != SNACK_OK) return st;
    }
  }
  // Column-panel partition of the row table (large layers only; the panel
  // SDDMM runs over rows).
  {
    PanelTable &pt = L.csr.panel;
    free_panel_table(pt);
    std::vector<int4> part;
    int lines_max = 0;
    const int ctas = device_sms();
    if (n >= panel_min_nnz() && n > 0)
      build_panel_partition(rp, L.out, n, ctas, part, &lines_max);
    if (!part.empty() && lines_max <= kPanelLinesPerWarp) {
      TRY_CUDA(dev_alloc(&pt.d_part, part.size(), &L.device_bytes));
      TRY_CUDA(cudaMemcpyAsync(pt.d_part, part.data(), part.size() * sizeof(int4),
                               cudaMemcpyHostToDevice, s));
      TRY_CUDA(build_panel_offsets(pt, L.d_row_ptr, L.d_col, L.out, L.in, &L.device_bytes, s));
      TRY_CUDA(cudaStreamSynchronize(s));
      pt.ctas = ctas;
      pt.lines = L.out;
      pt.lines_max = lines_max;
      pt.bytes += part.size() * sizeof(int4);
    }
  }
  // Split workspace: partial slots and re-armed tickets (zero between calls).
  if (L.d_partial) cudaFree(L.d_partial);
  if (L.d_counter) cudaFree(L.d_counter);
  L.d_partial = nullptr;
  L.d_counter = nullptr;
  TRY_CUDA(dev_alloc(&L.d_partial, partial_floats(L), &L.device_bytes));
  const int64_t tickets = std::max({L.csr.nsplit, L.csc.nsplit, L.csr_half.nsplit,
                                    L.csc_half.nsplit, L.csr_wide.nsplit, L.csc_wide.nsplit});
  TRY_CUDA(dev_alloc(&L.d_counter, (size_t)tickets, &L.device_bytes));
  TRY_CUDA(cudaMemsetAsync(L.d_counter, 0, std::max<size_t>(tickets, 1) * sizeof(int), s));
  TRY_CUDA(cudaStreamSynchronize(s));
  return SNACK_OK;
}

// ------------------------------------------------------ getrand(): draws --

// SplitMix64 (Steele, Lea and Flood, OOPSLA 2014): draw t of the stream whose
// state starts at `seed` is the finaliser applied to seed + (t+1) * gamma.
__device__ __forceinline__ uint64_t splitmix_draw(uint64_t seed, uint64_t t) {
  uint64_t z = seed + (t + 1ull) * 0x9E3779B97F4A7C15ull;
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

// Cell of draw x among n cells: floor(x * n / 2^64) (Lemire's reduction).
__device__ __forceinline__ uint64_t draw_cell(uint64_t x, uint64_t n) { return __umul64hi(x, n); }

__global__ void gen_candidates(uint64_t seed, uint64_t t0, int64_t m, uint64_t ncells,
                               uint64_t *key, uint32_t *idx) {
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= m) return;
  key[i] = draw_cell(splitmix_draw(seed, t0 + (uint64_t)i), ncells);
  idx[i] = (uint32_t)i;
}

__device__ __forceinline__ bool sorted_contains(const uint64_t *a, int64_t n, uint64_t x) {
  int64_t lo = 0, hi = n;
  while (lo < hi) {
    const int64_t mid = (lo + hi) >> 1;
    if (a[mid] < x)
      lo = mid + 1;
    else
      hi = mid;
  }
  return lo < n && a[lo] == x;
}

// Is cell x held by a surviving entry of the canonical layer?
__device__ __forceinline__ bool held_by_survivor(const int32_t *row, const int32_t *col,
                                                 const unsigned char *gone, int64_t n, int64_t in,
                                                 uint64_t x) {
  int64_t lo = 0, hi = n;
  while (lo < hi) {
    const int64_t mid = (lo + hi) >> 1;
    const uint64_t c = (uint64_t)row[mid] * (uint64_t)in + (uint64_t)col[mid];
    if (c < x)
      lo = mid + 1;
    else
      hi = mid;
  }
  if (lo >= n) return false;
  const uint64_t c = (uint64_t)row[lo] * (uint64_t)in + (uint64_t)col[lo];
  return c == x && !gone[lo];
}

// flag[t] = 1 iff candidate t is the first draw of its cell in this batch and
// the cell is neither held by a survivor nor taken in an earlier batch.
__global__ void flag_fresh(const uint64_t *skey, const uint32_t *sidx, int64_t m,
                           const int32_t *row, const int32_t *col, const unsigned char *gone,
                           int64_t n, int64_t in, const uint64_t *taken, int64_t ntaken,
                           int *flag) {
  const int64_t j = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (j >= m) return;
  const uint64_t x = skey[j];
  bool ok = (j == 0) || skey[j - 1] != x;
  if (ok && n > 0) ok = !held_by_survivor(row, col, gone, n, in, x);
  if (ok && ntaken > 0) ok = !sorted_contains(taken, ntaken, x);
  flag[sidx[j]] = ok ? 1 : 0;
}

// Append the first `want` fresh candidates (in draw order) to acc[base...].
__global__ void take_fresh(const int *flag, const int *rank, int64_t m, int64_t want, uint64_t seed,
                           uint64_t t0, uint64_t ncells, uint64_t *acc, int64_t base,
                           unsigned long long *last_t) {
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= m || !flag[i]) return;
  const int64_t r = rank[i];
  if (r >= want) return;
  acc[base + r] = draw_cell(splitmix_draw(seed, t0 + (uint64_t)i), ncells);
  if (r == want - 1) *last_t = t0 + (unsigned long long)i;
}

// Draw `want` fresh cells with Algorithm 2's rejection rule against the
// survivors of a canonical layer (n entries, `gone` marks pruned ones; n = 0
// for an empty layer).  acc[0..want) receives them in draw order.
snack_status draw_fresh(uint64_t seed, uint64_t ncells, int64_t want, const int32_t *row,
                        const int32_t *col, const unsigned char *gone, int64_t n, int64_t in,
                        int64_t survivors, uint64_t *acc, int64_t *trials, cudaStream_t s,
                        std::string &err) {
  *trials = 0;
  if (want <= 0) return SNACK_OK;
  const int nbits = bits_for(ncells - 1);
  Temps t;
  uint64_t *taken = nullptr, *taken_alt = nullptr;
  uint32_t *taken_v = nullptr, *taken_v_alt = nullptr;
  unsigned long long *d_last = nullptr;
  TRY_CUDA(t.get(&taken, want));
  TRY_CUDA(t.get(&taken_alt, want));
  TRY_CUDA(t.get(&taken_v, want));
  TRY_CUDA(t.get(&taken_v_alt, want));
  TRY_CUDA(t.get(&d_last, 1));
  int64_t have = 0;
  uint64_t t0 = 0;
  const uint64_t limit = 1ull << 40;
  while (have < want) {
    const double free_cells = (double)ncells - (double)survivors - (double)have;
    const double need = (double)(want - have);
    double mm = need * ((double)ncells / std::max(1.0, free_cells)) * 1.25 + 1024.0;
    mm = std::min(mm, (double)(1ll << 26));
    const int64_t m = (int64_t)mm;
    Temps bt;
    uint64_t *ka, *kb;
    uint32_t *va, *vb;
    int *flag, *rank;
    TRY_CUDA(bt.get(&ka, m));
    TRY_CUDA(bt.get(&kb, m));
    TRY_CUDA(bt.get(&va, m));
    TRY_CUDA(bt.get(&vb, m));
    TRY_CUDA(bt.get(&flag, m));
    TRY_CUDA(bt.get(&rank, m));
    gen_candidates<<<grid_for(m, 256), 256, 0, s>>>(seed, t0, m, ncells, ka, va);
    TRY_CUDA(cudaGetLastError());
    snack_status st = radix_sort(&ka, &va, &kb, &vb, m, nbits, s, err);
    if (st != SNACK_OK) return st;
    // `taken` (cells accepted in earlier batches) is kept sorted for lookup.
    flag_fresh<<<grid_for(m, 256), 256, 0, s>>>(ka, va, m, row, col, gone, n, in, taken_alt, have,
                                                flag);
    TRY_CUDA(cudaGetLastError());
    st = exclusive_scan(flag, rank, m, s, err);
    if (st != SNACK_OK) return st;
    int last_flag = 0, last_rank = 0;
    TRY_CUDA(cudaMemcpyAsync(&last_flag, flag + m - 1, 4, cudaMemcpyDeviceToHost, s));
    TRY_CUDA(cudaMemcpyAsync(&last_rank, rank + m - 1, 4, cudaMemcpyDeviceToHost, s));
    TRY_CUDA(cudaStreamSynchronize(s));
    const int64_t fresh = (int64_t)last_flag + last_rank;
    const int64_t use = std::min(fresh, want - have);
    take_fresh<<<grid_for(m, 256), 256, 0, s>>>(flag, rank, m, use, seed, t0, ncells, acc, have,
                                                d_last);
    TRY_CUDA(cudaGetLastError());
    if (fresh >= want - have) {
      unsigned long long last = 0;
      TRY_CUDA(cudaMemcpyAsync(&last, d_last, 8, cudaMemcpyDeviceToHost, s));
      TRY_CUDA(cudaStreamSynchronize(s));
      *trials = (int64_t)last + 1;
      return SNACK_OK;
    }
    have += use;
    t0 += (uint64_t)m;
    if (t0 > limit) {
      err = "regrow: no fresh cells after 2^40 draws";
      return SNACK_ERR_TIMEOUT;
    }
    // Re-sort the accepted cells into taken_alt for the next batch's lookups.
    TRY_CUDA(cudaMemcpyAsync(taken, acc, have * sizeof(uint64_t), cudaMemcpyDeviceToDevice, s));
    TRY_CUDA(cudaMemsetAsync(taken_v, 0, have * sizeof(uint32_t), s));
    uint64_t *k1 = taken, *k2 = taken_alt;
    uint32_t *v1 = taken_v, *v2 = taken_v_alt;
    st = radix_sort(&k1, &v1, &k2, &v2, have, nbits, s, err);
    if (st != SNACK_OK) return st;
    if (k1 != taken_alt)
      TRY_CUDA(cudaMemcpyAsync(taken_alt, k1, have * sizeof(uint64_t), cudaMemcpyDeviceToDevice, s));
    TRY_CUDA(cudaStreamSynchronize(s));
  }
  return SNACK_OK;
}

__global__ void split_cells(const uint64_t *cell, int64_t n, int64_t in, int32_t *row,
                            int32_t *col) {
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n) return;
  row[i] = (int32_t)(cell[i] / (uint64_t)in);
  col[i] = (int32_t)(cell[i] % (uint64_t)in);
}

// ---------------------------------------------------------- prune step ----

__global__ void magnitude_keys(const float *val, int64_t n, uint64_t *key, uint32_t *idx) {
  const int64_t k = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (k >= n) return;
  key[k] = (uint64_t)(__float_as_uint(val[k]) & 0x7FFFFFFFu);
  idx[k] = (uint32_t)k;
}

__global__ void mark_pruned(const uint32_t *order, int64_t p, unsigned char *gone) {
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i < p) gone[order[i]] = 1;
}

constexpr uint32_t kRegrown = 0xFFFFFFFFu;

// Survivors keep (cell, k); the i-th pruned slot (magnitude order) takes the
// i-th regrown cell.  `order` is a permutation, so every k is written once.
__global__ void merged_keys(const int32_t *row, const int32_t *col, int64_t n, int64_t in,
                            const uint32_t *order, int64_t p, const uint64_t *fresh, uint64_t *key,
                            uint32_t *src) {
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n) return;
  const uint32_t k = order[i];
  if (i < p) {
    key[k] = fresh[i];
    src[k] = kRegrown;
  } else {
    key[k] = (uint64_t)row[k] * (uint64_t)in + (uint64_t)col[k];
    src[k] = k;
  }
}

__global__ void regrown_values(const uint64_t *key, const uint32_t *src, int64_t n, int64_t in,
                               const float *old_val, int32_t *row, int32_t *col, float *val) {
  const int64_t k = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (k >= n) return;
  row[k] = (int32_t)(key[k] / (uint64_t)in);
  col[k] = (int32_t)(key[k] % (uint64_t)in);
  val[k] = src[k] == kRegrown ? 0.f : old_val[src[k]];
}

// Per-entry optimizer state follows its entry through the new order; regrown
// entries start from zero state.
__global__ void carry_state(const uint32_t *src, int64_t n, const float *old, float *state) {
  const int64_t k = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (k >= n) return;
  state[k] = src[k] == kRegrown ? 0.f : old[src[k]];
}

}  // namespace

// ------------------------------------------------------------- public -----

snack_status build_topology(Layer &L, int64_t nnz, const int32_t *d_row_user,
                            const int32_t *d_col_user, const float *d_val_user, cudaStream_t s,
                            std::string &err, bool workspace) {
  L.nnz = nnz;
  L.nnz_pad = pad4(nnz);
  size_t *acct = &L.device_bytes;
  TRY_CUDA(dev_alloc(&L.d_col, L.nnz_pad, acct));
  TRY_CUDA(dev_alloc(&L.d_row, L.nnz_pad, acct));
  TRY_CUDA(dev_alloc(&L.d_val, L.nnz_pad, acct));
  TRY_CUDA(dev_alloc(&L.d_csc_row, L.nnz_pad, acct));
  TRY_CUDA(dev_alloc(&L.d_csc_perm, L.nnz_pad, acct));
  TRY_CUDA(dev_alloc(&L.d_val_csc, L.nnz_pad, acct));
  TRY_CUDA(dev_alloc(&L.d_row_ptr, L.out + 1, acct));
  TRY_CUDA(dev_alloc(&L.d_col_ptr, L.in + 1, acct));
  if (workspace) {
    TRY_CUDA(dev_alloc(&L.d_xt, (size_t)L.in * kMaxSlice, acct));
    TRY_CUDA(dev_alloc(&L.d_dyt, (size_t)L.out * kMaxSlice, acct));
    TRY_CUDA(dev_alloc(&L.d_err, 1, acct));
    TRY_CUDA(cudaMemsetAsync(L.d_err, 0, sizeof(int), s));
  }
  TRY_CUDA(cudaMemsetAsync(L.d_col, 0, L.nnz_pad * 4, s));
  TRY_CUDA(cudaMemsetAsync(L.d_row, 0, L.nnz_pad * 4, s));
  TRY_CUDA(cudaMemsetAsync(L.d_val, 0, L.nnz_pad * 4, s));
  TRY_CUDA(cudaMemsetAsync(L.d_csc_row, 0, L.nnz_pad * 4, s));
  TRY_CUDA(cudaMemsetAsync(L.d_csc_perm, 0, L.nnz_pad * 4, s));
  TRY_CUDA(cudaMemsetAsync(L.d_val_csc, 0, L.nnz_pad * 4, s));

  Temps t;
  uint64_t *ka, *kb;
  uint32_t *va, *vb;
  unsigned long long *flags;  // [0] = first out-of-range index, [1] = duplicate
  TRY_CUDA(t.get(&ka, nnz));
  TRY_CUDA(t.get(&kb, nnz));
  TRY_CUDA(t.get(&va, nnz));
  TRY_CUDA(t.get(&vb, nnz));
  TRY_CUDA(t.get(&flags, 2));
  TRY_CUDA(cudaMemsetAsync(flags, 0xFF, 2 * sizeof(unsigned long long), s));
  if (nnz > 0) {
    make_cell_keys<<<grid_for(nnz, 256), 256, 0, s>>>(d_row_user, d_col_user, nnz, L.out, L.in, ka,
                                                      va, flags);
    TRY_CUDA(cudaGetLastError());
  }
  unsigned long long h_flags[2];
  TRY_CUDA(cudaMemcpyAsync(h_flags, flags, sizeof(h_flags), cudaMemcpyDeviceToHost, s));
  TRY_CUDA(cudaStreamSynchronize(s));
  if (h_flags[0] != ~0ull) {
    err = "entry " + std::to_string(h_flags[0]) + " has a row or column outside the layer";
    return SNACK_ERR_OUT_OF_RANGE;
  }
  const uint64_t cells = (uint64_t)L.out * (uint64_t)L.in;
  snack_status st = radix_sort(&ka, &va, &kb, &vb, nnz, bits_for(cells - 1), s, err);
  if (st != SNACK_OK) return st;
  if (nnz > 0) {
    finish_canonical<<<grid_for(nnz, 256), 256, 0, s>>>(ka, va, nnz, L.in, d_val_user, L.d_row,
                                                        L.d_col, L.d_val, flags + 1);
    TRY_CUDA(cudaGetLastError());
  }
  TRY_CUDA(cudaMemcpyAsync(h_flags, flags, sizeof(h_flags), cudaMemcpyDeviceToHost, s));
  TRY_CUDA(cudaStreamSynchronize(s));
  if (h_flags[1] != ~0ull) {
    err = "entry " + std::to_string(h_flags[1]) + " repeats a (row, col) already stored";
    return SNACK_ERR_DUPLICATE;
  }
  return finish_layout(L, ka, s, err);
}

snack_status draw_random_cells(int64_t out, int64_t in, int64_t count, uint64_t seed,
                               int32_t *d_row, int32_t *d_col, int64_t *trials, cudaStream_t s,
                               std::string &err) {
  Temps t;
  uint64_t *acc;
  TRY_CUDA(t.get(&acc, count));
  const uint64_t cells = (uint64_t)out * (uint64_t)in;
  snack_status st = draw_fresh(seed, cells, count, nullptr, nullptr, nullptr, 0, in, 0, acc, trials,
                               s, err);
  if (st != SNACK_OK) return st;
  if (count > 0) {
    split_cells<<<grid_for(count, 256), 256, 0, s>>>(acc, count, in, d_row, d_col);
    TRY_CUDA(cudaGetLastError());
  }
  TRY_CUDA(cudaStreamSynchronize(s));
  return SNACK_OK;
}

// Magnitude prune + uniform regrow.  The new entry set (survivors and
// regrown cells, its values and optimizer state) is built beside the layer,
// as a second layer of the same shape; only once all of it exists is it
// committed: values and state are copied into the layer's own buffers
// (their pointers stay valid) and the topology arrays are swapped.  A
// failure before that, an allocation included, leaves the layer as it was.
snack_status prune_regrow(Layer &L, float frac, uint64_t seed, int64_t *pruned, int64_t *trials,
                          cudaStream_t s, std::string &err) {
  const int64_t n = L.nnz;
  int64_t P = 0;
  if (frac > 0.0f) P = frac >= 1.0f ? n : (int64_t)std::floor((double)frac * (double)n);
  *pruned = P;
  *trials = 0;
  if (P == 0) return SNACK_OK;
  Temps t;
  uint64_t *ka, *kb, *fresh;
  uint32_t *va, *vb;
  unsigned char *gone;
  int32_t *new_row, *new_col;
  float *new_val, *new_state[2] = {nullptr, nullptr};
  TRY_CUDA(t.get(&ka, n));
  TRY_CUDA(t.get(&kb, n));
  TRY_CUDA(t.get(&va, n));
  TRY_CUDA(t.get(&vb, n));
  TRY_CUDA(t.get(&fresh, P));
  TRY_CUDA(t.get(&gone, n));
  TRY_CUDA(t.get(&new_row, n));
  TRY_CUDA(t.get(&new_col, n));
  TRY_CUDA(t.get(&new_val, n));
  for (int i = 0; i < 2; ++i)
    if (L.d_opt[i]) TRY_CUDA(t.get(&new_state[i], n));
  TRY_CUDA(cudaMemsetAsync(gone, 0, n, s));
  magnitude_keys<<<grid_for(n, 256), 256, 0, s>>>(L.d_val, n, ka, va);
  TRY_CUDA(cudaGetLastError());
  snack_status st = radix_sort(&ka, &va, &kb, &vb, n, 31, s, err);
  if (st != SNACK_OK) return st;
  mark_pruned<<<grid_for(P, 256), 256, 0, s>>>(va, P, gone);
  TRY_CUDA(cudaGetLastError());
  const uint64_t cells = (uint64_t)L.out * (uint64_t)L.in;
  st = draw_fresh(seed, cells, P, L.d_row, L.d_col, gone, n, L.in, n - P, fresh, trials, s, err);
  if (st != SNACK_OK) return st;
  // New entry set: survivors and regrown cells, back into canonical order.
  // va still holds the magnitude order (a permutation of 0..n-1).
  merged_keys<<<grid_for(n, 256), 256, 0, s>>>(L.d_row, L.d_col, n, L.in, va, P, fresh, kb, vb);
  TRY_CUDA(cudaGetLastError());
  uint64_t *k1 = kb, *k2 = ka;
  uint32_t *v1 = vb, *v2 = va;
  st = radix_sort(&k1, &v1, &k2, &v2, n, bits_for(cells - 1), s, err);
  if (st != SNACK_OK) return st;
  regrown_values<<<grid_for(n, 256), 256, 0, s>>>(k1, v1, n, L.in, L.d_val, new_row, new_col,
                                                  new_val);
  TRY_CUDA(cudaGetLastError());
  for (int i = 0; i < 2; ++i) {
    if (!L.d_opt[i]) continue;
    carry_state<<<grid_for(n, 256), 256, 0, s>>>(v1, n, L.d_opt[i], new_state[i]);
    TRY_CUDA(cudaGetLastError());
  }
  // The new layout beside the layer (canonical input: its sort keeps the order).
  Layer N;
  N.out = L.out;
  N.in = L.in;
  N.device = L.device;
  st = build_topology(N, n, new_row, new_col, new_val, s, err, false);
  if (st != SNACK_OK) {
    free_layer(N);
    return st;
  }
  // Commit: nothing below allocates.
  cudaError_t e = cudaMemcpyAsync(L.d_val, N.d_val, n * sizeof(float), cudaMemcpyDeviceToDevice, s);
  for (int i = 0; i < 2 && e == cudaSuccess; ++i)
    if (L.d_opt[i])
      e = cudaMemcpyAsync(L.d_opt[i], new_state[i], n * sizeof(float), cudaMemcpyDeviceToDevice, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) {
    free_layer(N);
    err = std::string("prune/regrow commit: ") + cudaGetErrorString(e);
    return SNACK_ERR_CUDA;
  }
  std::swap(L.d_row, N.d_row);
  std::swap(L.d_col, N.d_col);
  std::swap(L.d_row_ptr, N.d_row_ptr);
  std::swap(L.d_col_ptr, N.d_col_ptr);
  std::swap(L.d_csc_row, N.d_csc_row);
  std::swap(L.d_csc_perm, N.d_csc_perm);
  std::swap(L.d_val_csc, N.d_val_csc);
  std::swap(L.csr, N.csr);
  std::swap(L.csc, N.csc);
  std::swap(L.csr_half, N.csr_half);
  std::swap(L.csc_half, N.csc_half);
  std::swap(L.csr_wide, N.csr_wide);
  std::swap(L.csc_wide, N.csc_wide);
  std::swap(L.d_partial, N.d_partial);
  std::swap(L.d_counter, N.d_counter);
  L.csc_vals = !L.values_shared;  // the copy was derived from these values
  free_layer(N);  // the old topology and the shadow's own values
  return SNACK_OK;
}

snack_status refresh_csc_values(Layer &L, cudaStream_t s, std::string &err) {
  if (L.nnz > 0) {
    gather_by_perm<<<grid_for(L.nnz, 256), 256, 0, s>>>(L.d_csc_perm, L.d_val, L.nnz,
                                                        L.d_val_csc);
    TRY_CUDA(cudaGetLastError());
  }
  L.csc_vals = !L.values_shared;
  return SNACK_OK;
}

size_t partial_floats(const Layer &L) {
  return (size_t)std::max({L.csr.nslots * kMaxSlice, L.csc.nslots * kMaxSlice,
                           L.csr_half.nslots * kHalfLineWidth,
                           L.csc_half.nslots * kHalfLineWidth,
                           L.csr_wide.nslots * kHalfLineWidth,
                           L.csc_wide.nslots * kHalfLineWidth});
}

void free_layer(Layer &L) {
  void *ptrs[] = {L.d_col,     L.d_row,     L.d_val,         L.d_row_ptr,     L.d_csc_row,
                  L.d_csc_perm, L.d_col_ptr, L.csr.d_seg,     L.csr.d_split,   L.csc.d_seg,
                  L.csc.d_split, L.d_xt,     L.d_dyt,         L.d_partial,     L.d_counter,
                  L.d_err,     L.d_opt[0],  L.d_opt[1],
                  L.d_gacc,    L.d_val_csc};
  for (void *p : ptrs)
    if (p) cudaFree(p);
  free_panel_table(L.csr.panel);
  free_panel_table(L.csc.panel);
  for (SegTable *t : {&L.csr_half, &L.csc_half, &L.csr_wide, &L.csc_wide}) free_segments(*t);
  L = Layer();
}

}  // namespace snack
