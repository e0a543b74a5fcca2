// Internal declarations of the SNACK sparse-layer library (sm_103a).
//
// Device data layout of one layer (all owned by the handle):
//   col      [nnz_pad] int32   column of entry k, canonical (row, col) order
//   row      [nnz_pad] int32   row of entry k (canonical order)
//   val      [nnz_pad] fp32    value of entry k (canonical order)
//   row_ptr  [out+1]   int32   CSR index pointer
//   csc_row  [nnz_pad] int32   row of the s-th entry in (col, row) order
//   csc_perm [nnz_pad] int32   canonical k of the s-th entry in (col, row) order
//   val_csc  [nnz_pad] fp32    val[csc_perm[s]]: the values in (col, row) order,
//                              trusted while the values have not changed since
//                              it was derived (see Layer::csc_vals)
//   col_ptr  [in+1]    int32   CSC index pointer
//   seg_csr / seg_csc  int4    work decomposition of rows / columns into
//                              segments {line, begin, end, split_id}
//   split_csr / split_csc int4 {first_segment, parts, first_slot, 0} for
//                              lines cut into several segments
//   workspace                  transposed dense operand slices, split partial
//                              sums, split counters
// nnz_pad rounds nnz up to a multiple of 4 (plus 4) so that 16-byte vector
// loads of the index and value streams never leave the allocation; padding
// entries hold index 0 and value 0 and are masked out by the kernels.
#pragma once

#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>
#include <string>
#include <vector>

#include "../../include/snack.h"

namespace snack {

constexpr int kMaxSlice = 256;  // widest batch slice one kernel launch handles
constexpr int kOptNone = 0, kOptSgd = 1, kOptAdam = 2;  // optimizer kinds

// Entry-balanced partition of the row table for the column-panel SDDMM
// (panel.cu): per CTA 32 int4, one per consumer warp {first entry, end
// entry, first line, lines}, then {first line, end line} of the CTA.  Built
// at topology time for layers of at least panel_min_nnz() entries.
constexpr int kPanelLinesPerWarp = 4;  // lines one consumer warp can hold

constexpr int kPanelWidths = 4;  // slices of 8, 16, 32, 64 floats

// Widest slice that walks the cut-line tables (Layer::csr_half, csr_wide):
// at 64 floats per entry a team's walk of a long line is latency-bound, and
// the last round of teams runs mostly empty.
constexpr int kHalfLineWidth = 64;
// Parts per line of the cut copy that slices of kHalfLineWidth walk.
constexpr int kWideCutParts = 4;

struct PanelTable {
  int4 *d_part = nullptr;  // [ctas][32]
  int64_t ctas = 0;
  int64_t lines = 0;       // lines of the table
  int lines_max = 0;       // most lines any consumer warp covers
  // Per slice width (8, 16, 32, 64): run offsets [P + 1][lines], where
  // off[p][l] is the first entry of line l whose operand index is at least
  // p * PW (PW = operand lines per panel), off[0] = line start, off[P] = end.
  int32_t *d_off[kPanelWidths] = {nullptr, nullptr, nullptr, nullptr};
  size_t bytes = 0;        // device bytes of the partition and the offsets
};

struct SegTable {
  int64_t nseg = 0;
  int64_t nsplit = 0;
  int64_t nslots = 0;      // partial-sum slots (sum of parts over split lines)
  double mean_len = 0.0;   // mean entries per line
  int64_t max_len = 0;     // longest line
  int max_parts = 0;       // most parts of one split line
  int4 *d_seg = nullptr;   // [nseg]
  int4 *d_split = nullptr; // [nsplit]
  PanelTable panel;        // column-panel partition (d_part null when not built)
};

struct Layer {
  int64_t out = 0, in = 0, nnz = 0, nnz_pad = 0;
  int device = 0;
  int *d_err = nullptr;        // device error flag (a bounded wait gave up)
  int32_t *d_col = nullptr;
  int32_t *d_row = nullptr;
  float *d_val = nullptr;
  int32_t *d_row_ptr = nullptr;
  int32_t *d_csc_row = nullptr;
  int32_t *d_csc_perm = nullptr;
  float *d_val_csc = nullptr;      // [nnz_pad] values in (col, row) order
  bool csc_vals = false;           // d_val_csc equals val through csc_perm
  bool values_shared = false;      // a writable values pointer is out (snack_values)
  int32_t *d_col_ptr = nullptr;
  SegTable csr, csc;
  // The same lines cut into 2 (half) and kWideCutParts (wide) balanced parts
  // each, for wide slices on layers of 2^21+ entries whose lines average
  // 400+ entries (nseg 0 when not built).
  SegTable csr_half, csc_half, csr_wide, csc_wide;
  // workspace
  float *d_xt = nullptr;       // [in][kMaxSlice]   transposed X slice
  float *d_dyt = nullptr;      // [out][kMaxSlice]  transposed dY slice
  float *d_partial = nullptr;  // [max(csr.nslots, csc.nslots)][kMaxSlice]
  int *d_counter = nullptr;    // [max(csr.nsplit, csc.nsplit)], zero between calls
  // optimizer (allocated by the first step that needs them)
  int opt_kind = kOptNone;     // kind the state below belongs to
  float *d_opt[2] = {nullptr, nullptr};  // [nnz_pad] momentum / first moment, second moment
  float *d_gacc = nullptr;     // [nnz_pad] whole-batch gradient of the unfused steps (batch > 4)
  size_t device_bytes = 0;
  std::string last_error;
};

// Everything a segmented SpMM / SDDMM launch needs.
struct SpmmArgs {
  const int4 *seg;
  int64_t nseg;
  const int4 *split;
  const int32_t *idx;   // column (rows) or row (columns) index stream
  const float *val;     // canonical values
  const int32_t *perm;  // column-order -> canonical position (or null)
  const float *src;     // transposed dense operand [lines_src][bw]
  float *dst;           // dense output, element (b, line) at dst[b * ld + line]
  int64_t ld;
  int nb;               // valid batch rows in this slice
  float *partial;
  int *counter;
  int lps;              // lanes per segment team (set by the launcher)
  int64_t nval;         // floats in the padded value array (L2 prefetch bound)
  int prefetch;         // pull the segments' streams into L2 while waiting on a transpose
  int stride;           // floats between operand rows (the transposed slice's width)
  int nsub;             // batch sub-slices of BW columns, one team per (sub-slice, segment);
                        // > 1 only for tables without split lines
  int stage;            // table without split lines (segment s is line s): slices of 128+
                        // with one team per warp write their outputs through shared memory
};

// Optimizer step fused into the SDDMM epilogue (kind != kOptNone): the
// gradient of each stored entry updates its value and state in place and
// dW is not written.  Coefficients are prepared on the host.
struct OptArgs {
  int kind = kOptNone;
  float lr = 0.f, mom = 0.f, wd = 0.f;            // SGD: lr, momentum; both: weight decay
  float b1 = 0.f, c1 = 0.f, b2 = 0.f, c2 = 0.f;   // Adam: beta1, 1 - beta1, beta2, 1 - beta2
  float eps = 0.f, step = 0.f, sbc2 = 1.f;        // Adam: eps, lr / (1 - b1^t), sqrt(1 - b2^t)
  float *val = nullptr;                           // [nnz] values, canonical order
  float *s0 = nullptr;                            // momentum buffer / first moment (or null)
  float *s1 = nullptr;                            // second moment (Adam)
};

struct SddmmArgs {
  const int4 *seg;
  int64_t nseg;
  const int32_t *col;
  const float *xt;   // [in][bw]
  const float *dyt;  // [out][bw]
  float *dw;         // [nnz]
  int accumulate;    // add to dw instead of overwriting (batch slices > 0)
  int lps;           // lanes per segment team (set by the launcher)
  int prefetch;      // pull the segments' column streams into L2 while waiting on a transpose
  int nsub;          // entry sub-ranges per segment, one team each
  OptArgs opt;       // optimizer step fused in instead of writing dw (slices of 1-4)
};

// Everything a column-panel SDDMM launch needs (panel.cu).
struct PanelArgs {
  const int4 *part;      // the row table's partition (set by the launcher)
  const int32_t *idx;    // column of each entry, canonical order
  const float *src;      // transposed X slice [n_op][bw]
  int64_t n_op;          // X^T lines (in_features)
  const float *dyt;      // transposed dY slice [rows][bw]
  float *dw;             // dW output (canonical order)
  int accumulate;        // add to dw (batch slices after the first)
  int *err;              // the layer's device error flag
  const int32_t *off;    // the table's run offsets for this width (set by the launcher)
  int64_t lines;         // rows of the table (row stride of off)
};

// Kernel selection: batch slice width, lanes per entry group, lanes per segment.
struct Plan {
  int bw = 1;
  int lanes = 32;
  double mean_len = 0.0;  // mean entries per segment of the table planned for
};
int slice_width(int64_t nb);
Plan choose_plan(const SegTable &t, int64_t nb);
Plan plan_for_width(const SegTable &t, int bw);
int plan_team_lanes(const Plan &p);  // lanes per team the launchers use
int device_sms();                    // SM count of the current device
int entry_lanes(int bw);

// Launchers (spmm_*.cu).  Return the launch's cudaError_t.
// pdl: launch as a programmatic dependent of the previous kernel on the
// stream (the kernels wait for it before touching any memory it may use).
cudaError_t launch_spmm_rows(const Plan &p, const SpmmArgs &a, bool pdl, cudaStream_t s);
cudaError_t launch_spmm_cols(const Plan &p, const SpmmArgs &a, bool pdl, cudaStream_t s);
// Second pass summing the split lines' partials of an SpMM launched with
// a.counter null (bw = that launch's slice width).
cudaError_t launch_split_sums(int bw, const SpmmArgs &a, int64_t nsplit, int max_parts,
                              bool pdl, cudaStream_t s);
cudaError_t launch_sddmm(const Plan &p, const SddmmArgs &a, bool pdl, cudaStream_t s);
// The same with the optimizer step of a.opt applied instead of writing dW.
cudaError_t launch_sddmm_step(const Plan &p, const SddmmArgs &a, bool pdl, cudaStream_t s);
cudaError_t launch_opt_apply(const OptArgs &o, const float *g, int64_t nnz, bool pdl,
                             cudaStream_t s);
cudaError_t launch_backward_fused(const Plan &pc, const SpmmArgs &cols, const Plan &pr,
                                  const SddmmArgs &rows, bool pdl, cudaStream_t s);
// Variants with the whole operand resident in shared memory (slices of 1-4
// floats; resident_operand.cu).  n_op = operand lines (in for the forward
// and dW, out for dX); err = the layer's device error flag.
bool resident_fits(int bw, int64_t n_op, int64_t nseg, int64_t nnz);
cudaError_t launch_resident_spmm(bool perm, const Plan &p, const SpmmArgs &a, int64_t n_op,
                                 int *err, bool pdl, cudaStream_t s);
// Column-panel SDDMM (slices of 8-64 floats) on the row table, when it has a
// partition and its rows' runs per panel are long (mean_len entries per row,
// n_op = in_features).
bool panel_fits(const PanelTable &t, int bw, double mean_len, int64_t n_op);
cudaError_t launch_panel_sddmm(int bw, const PanelTable &t, const PanelArgs &a, bool pdl,
                               cudaStream_t s);
void build_panel_partition(const std::vector<int32_t> &ptr, int64_t nlines, int64_t nnz, int ctas,
                           std::vector<int4> &part, int *lines_max);
// Run offsets of every width for a table of `lines` lines over an operand of
// n_op lines (ptr / idx: the table's line pointer and index stream on the
// device).  Allocates t.d_off[*] (bytes added to *acct); asynchronous on s.
cudaError_t build_panel_offsets(PanelTable &t, const int32_t *ptr, const int32_t *idx,
                                int64_t lines, int64_t n_op, size_t *acct, cudaStream_t s);
void free_panel_table(PanelTable &t);
// Smallest layer (stored entries) that gets panel partitions: 2^21, or the
// SNACK_PANEL_MIN_NNZ environment variable when set.
int64_t panel_min_nnz();
// One block that waits, with a short bound, on an mbarrier nothing completes
// and sets *err when it gives up (the failure path of the bounded waits).
cudaError_t launch_wait_selftest(int *err, cudaStream_t s);
cudaError_t launch_resident_sddmm(const Plan &p, const SddmmArgs &a, int64_t n_op, int *err,
                                  bool pdl, cudaStream_t s);
// at[c * bw + b] = a[b * a_ld + c] and bt likewise, in one launch.
cudaError_t launch_transpose_pair(const float *a, int64_t a_ld, int64_t a_cols, float *at,
                                  const float *b, int64_t b_ld, int64_t b_cols, float *bt, int nb,
                                  int bw, cudaStream_t s, bool pdl = false);
// dst[c * bw + b] = b < nb ? src[b * ld + c] : 0, for c < ncols, b < bw.
cudaError_t launch_transpose(const float *src, int64_t ld, int nb, int64_t ncols, float *dst,
                             int bw, cudaStream_t s, bool pdl = false);

// Topology (topology.cu).  workspace = false leaves out the per-slice
// workspace (transposed operands, error flag): a layer built only to take
// another's topology.
snack_status build_topology(Layer &L, int64_t nnz, const int32_t *d_row_user,
                            const int32_t *d_col_user, const float *d_val_user,
                            cudaStream_t s, std::string &err, bool workspace = true);
snack_status draw_random_cells(int64_t out, int64_t in, int64_t count, uint64_t seed,
                               int32_t *d_row, int32_t *d_col, int64_t *trials,
                               cudaStream_t s, std::string &err);
snack_status prune_regrow(Layer &L, float frac, uint64_t seed, int64_t *pruned,
                          int64_t *trials, cudaStream_t s, std::string &err);
void free_layer(Layer &L);
// Floats of the split-line partial workspace: kMaxSlice per slot of the
// row and column tables, kHalfLineWidth per slot of their cut copies.
size_t partial_floats(const Layer &L);
// val_csc[s] = val[csc_perm[s]]; the copy is current unless a writable
// values pointer is out.
snack_status refresh_csc_values(Layer &L, cudaStream_t s, std::string &err);

// Every device allocation of the library: cudaMalloc, unless the
// out-of-memory test hook (snack_debug_fail_alloc) makes this one fail.
cudaError_t device_malloc(void **p, size_t bytes);

// Device memory helper: device_malloc with byte accounting.
template <typename T>
cudaError_t dev_alloc(T **p, size_t count, size_t *acct) {
  size_t bytes = count * sizeof(T);
  if (bytes == 0) bytes = sizeof(T);
  cudaError_t e = device_malloc(reinterpret_cast<void **>(p), bytes);
  if (e == cudaSuccess && acct) *acct += bytes;
  return e;
}

inline int64_t pad4(int64_t n) { return ((n + 3) / 4) * 4 + 4; }

}  // namespace snack
