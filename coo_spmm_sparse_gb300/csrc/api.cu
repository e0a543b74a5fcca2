// C ABI of the SNACK sparse layer (declarations and contracts in snack.h).
// Host-side orchestration only: argument checks, batch slicing, kernel
// selection and launches.  All arithmetic runs in the kernels.
#include <algorithm>
#include <cmath>
#include <atomic>
#include <cstdio>
#include <cstring>
#include <new>
#include <string>
#include <vector>

#include "snack_internal.cuh"

struct snack_layer {
  snack::Layer L;
};

namespace {

thread_local std::string g_create_error;
std::atomic<uint64_t> g_launches{0};
std::atomic<int64_t> g_fail_alloc{-1};  // allocations left before the test hook fires

snack_status fail(snack_handle h, snack_status st, const std::string &msg) {
  if (h)
    h->L.last_error = msg;
  else
    g_create_error = msg;
  return st;
}

snack_status cuda_fail(snack_handle h, cudaError_t e, const char *what) {
  return fail(h, e == cudaErrorMemoryAllocation ? SNACK_ERR_ALLOC : SNACK_ERR_CUDA,
              std::string(what) + ": " + cudaGetErrorString(e));
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// The handle's device must be current: the kernels address its memory.
snack_status check_device(snack_handle h) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(h, e, "cudaGetDevice");
  if (dev != h->L.device)
    return fail(h, SNACK_ERR_INVALID_ARG,
                "device " + std::to_string(dev) + " is current but the layer lives on device " +
                    std::to_string(h->L.device));
  return SNACK_OK;
}

snack_status check_dense(snack_handle h, const void *p, const char *name) {
  if (!p) return fail(h, SNACK_ERR_INVALID_ARG, std::string(name) + " is NULL");
  if (!aligned16(p)) return fail(h, SNACK_ERR_INVALID_ARG, std::string(name) + " is not 16-byte aligned");
  return SNACK_OK;
}

snack_status check_shape(int64_t out, int64_t in, int64_t nnz) {
  if (out < 1 || in < 1 || out > 0x7fffffffLL || in > 0x7fffffffLL)
    return fail(nullptr, SNACK_ERR_INVALID_ARG, "out_features and in_features must be in [1, 2^31)");
  if (nnz < 0) return fail(nullptr, SNACK_ERR_INVALID_ARG, "nnz must be >= 0");
  if (nnz > 0x7fffff00LL)
    return fail(nullptr, SNACK_ERR_UNSUPPORTED, "nnz must stay below 2^31 - 256");
  if ((uint64_t)nnz > (uint64_t)out * (uint64_t)in)
    return fail(nullptr, SNACK_ERR_INVALID_ARG, "nnz exceeds out_features * in_features");
  return SNACK_OK;
}

void account(snack::Layer &L) {
  size_t b = 0;
  b += (size_t)L.nnz_pad * 4 * 5;  // col, row, val, csc_row, csc_perm
  b += (size_t)(L.out + 1 + L.in + 1) * 4;
  for (const snack::SegTable *t :
       {&L.csr, &L.csc, &L.csr_half, &L.csc_half, &L.csr_wide, &L.csc_wide})
    b += (size_t)(t->nseg + t->nsplit) * sizeof(int4);
  b += L.csr.panel.bytes + L.csc.panel.bytes;
  b += (size_t)(L.in + L.out) * snack::kMaxSlice * 4;
  b += snack::partial_floats(L) * 4;
  b += (size_t)std::max({L.csr.nsplit, L.csc.nsplit, L.csr_half.nsplit, L.csc_half.nsplit,
                         L.csr_wide.nsplit, L.csc_wide.nsplit}) *
       4;
  b += 4;  // error flag
  // column-ordered values; optimizer state, gradient buffer
  const void *extra[] = {L.d_val_csc, L.d_opt[0], L.d_opt[1], L.d_gacc};
  for (const void *p : extra)
    if (p) b += (size_t)L.nnz_pad * 4;
  L.device_bytes = b;
}

snack_status finish_create(snack_layer *h, snack_status st, const std::string &err,
                           snack_handle *out) {
  if (st != SNACK_OK) {
    snack::free_layer(h->L);
    delete h;
    return fail(nullptr, st, err);
  }
  account(h->L);
  *out = h;
  return SNACK_OK;
}

// The row (rows) or column table one product (SpMM or SDDMM) walks for a
// slice of nb batch rows, where the cut copies are built: slices of
// kHalfLineWidth walk the lines in kWideCutParts parts (10000 x 10000 at
// 90 %, batch 64: forward / dX / dW 157 / 156 / 169 us in halves, 144 / 144
// / 151 in quarters; at 95 % dW 88 -> 84), and so do the SDDMM's wider
// slices (its entries need no partial sums; batch 128 / 256 dW at 90 % 356
// / 669 -> 277 / 573 us, at 95 % 181 / 348 -> 151 / 302; the SpMMs' partial
// sums are sized for 64-float slices), 32-wide slices of the SDDMM in
// halves (its entries need no combining: batch 32 dW at 90 % 123.9 -> 106.1
// us, at 95 % 66.3 -> 59.9; thirds 106.6 / 61.7, and the SpMMs lost there,
// 101.8 -> 106.7 and 58.5 -> 59.3 with halves).
const snack::SegTable &line_table(const snack::Layer &L, bool rows, int64_t nb, bool sddmm) {
  const snack::SegTable &half = rows ? L.csr_half : L.csc_half;
  const snack::SegTable &wide = rows ? L.csr_wide : L.csc_wide;
  const int w = snack::slice_width(std::min<int64_t>(nb, snack::kMaxSlice));
  if (wide.nseg > 0 && (w == snack::kHalfLineWidth || (sddmm && w > snack::kHalfLineWidth)))
    return wide;
  if (sddmm && w == 32 && half.nseg > 0) return half;
  return rows ? L.csr : L.csc;
}

snack::SpmmArgs spmm_args(snack::Layer &L, const snack::SegTable &tab, bool rows, const float *op,
                          float *dst, int nb) {
  snack::SpmmArgs a;
  a.seg = tab.d_seg;
  a.nseg = tab.nseg;
  a.split = tab.d_split;
  a.idx = rows ? L.d_col : L.d_csc_row;
  a.val = L.d_val;
  a.perm = rows ? nullptr : L.d_csc_perm;
  if (!rows && L.csc_vals) {  // values already in column order: no permutation
    a.val = L.d_val_csc;
    a.perm = nullptr;
  }
  a.src = op;
  a.dst = dst;
  a.ld = rows ? L.out : L.in;
  a.nb = nb;
  a.partial = L.d_partial;
  a.counter = L.d_counter;
  a.lps = 32;
  a.nval = L.nnz_pad;
  a.prefetch = 0;
  a.stride = 0;  // set with the plan
  a.nsub = 1;
  a.stage = tab.nsplit == 0;
  return a;
}

// Batch sub-slices for a table too small to fill the GPU: while its teams
// would fill fewer blocks than there are SMs, the slice (width p.bw, the
// transposed operand's row stride) is cut into sub-slices of half the
// width, each covered by its own teams in the same launch (no combining:
// they write different rows of the output).  Tables with split lines keep
// whole slices, their partial sums being per slice.
snack::Plan sub_slices(const snack::SegTable &t, const snack::Plan &p, int nb, int *nsub) {
  *nsub = 1;
  snack::Plan q = p;
  if (t.nsplit != 0 || t.nseg == 0) return q;
  const int64_t sms = snack::device_sms();
  while (q.bw >= 16) {
    const int64_t blocks = (t.nseg * *nsub * snack::plan_team_lanes(q) + 255) / 256;
    if (blocks >= sms) break;
    const snack::Plan h = snack::plan_for_width(t, q.bw / 2);
    *nsub = (nb + h.bw - 1) / h.bw;
    q = h;
  }
  return q;
}

// Entry sub-ranges for the SDDMM of a table too small to fill the GPU:
// while its teams would fill fewer blocks than there are SMs, each segment
// is cut into twice as many parts (of 16 or more entries on average), each
// taken by its own team; the entries are independent, nothing is combined.
int sddmm_subranges(const snack::SegTable &t, const snack::Plan &p) {
  const int64_t sms = snack::device_sms();
  const int64_t lanes = snack::plan_team_lanes(p);
  int nsub = 1;
  while (nsub < 8 && (t.nseg * nsub * lanes + 255) / 256 < sms && t.mean_len >= 32.0 * nsub)
    nsub *= 2;
  return nsub;
}

// Whether the split lines of an SpMM over table t with plan q are summed by
// a second pass (split_sums) instead of by the last part's team: for slices
// of 8+ floats (16+ inside the fused backward), where the tickets' fences and
// the serial sum of the parts sit on the kernel's critical path (10000 x
// 10000 at 95 %, halved lines, batch 64 forward 91.1 -> 84.7 us; 8192 x 8192
// Zipf rows forward, batch 16 20.8 -> 20.1, batch 8 18.5 -> 16.9).  At
// narrower slices the extra launch costs what it saves (Zipf rows, batch 1:
// forward 12.3 -> 12.8 us, fused backward 12.8 -> 14.4; batch 2 and 4 even),
// and so does it in the fused backward at 8 (20.5 -> 21.0).
bool two_pass(const snack::SegTable &t, const snack::Plan &q, bool fused = false) {
  return t.nsplit > 0 && q.bw >= (fused ? 16 : 8);
}

// dX over the column segments: through the permutation, or (values in
// column order) with the canonical-order kernels.
cudaError_t launch_cols(const snack::SegTable &t, const snack::Plan &p, snack::SpmmArgs a, int nb,
                        cudaStream_t s) {
  const snack::Plan q = sub_slices(t, p, nb, &a.nsub);
  const bool two = two_pass(t, q);
  if (two) a.counter = nullptr;
  cudaError_t e =
      a.perm ? snack::launch_spmm_cols(q, a, true, s) : snack::launch_spmm_rows(q, a, true, s);
  if (e != cudaSuccess || !two) return e;
  g_launches.fetch_add(1, std::memory_order_relaxed);  // the first; the caller counts the second
  return snack::launch_split_sums(q.bw, a, t.nsplit, t.max_parts, true, s);
}

// Rows of the next batch slice when `left` rows remain: at most kMaxSlice.
// On a large layer a batch just above a power of two w (left - w <= w / 4,
// w >= 32) is cut into w and the remainder: a slice is padded to the next
// power of two, and gathering 2w floats per entry costs more there than a
// second pass over the index / value stream (10000 x 10000 @ 95 %: batch 33
// as one 64-wide slice 94 us, as 32 + 1 60 + 17 us).
int next_slice(const snack::Layer &L, int64_t left) {
  if (left >= snack::kMaxSlice) return snack::kMaxSlice;
  const int n = (int)left;
  if (L.nnz >= (int64_t(1) << 21)) {
    int w = 1;
    while (w * 2 <= n) w *= 2;  // largest power of two <= n
    if (w >= 32 && w < n && n - w <= w / 4) return w;
  }
  return n;
}

// Forward Y = X W^T over batch slices of at most 256: the slice of X is
// transposed into the workspace (not needed for a single row), then the
// row-segment kernel runs.  Every launch is a programmatic dependent of the
// kernel before it on the stream (the caller's or this call's own): its
// launch and start-up overlap that kernel's end, and it waits for it before
// touching memory.
snack_status run_forward(snack_handle h, const float *X, float *Y, int64_t batch, cudaStream_t s) {
  snack::Layer &L = h->L;
  for (int64_t b0 = 0, nb = 0; b0 < batch; b0 += nb) {
    nb = next_slice(L, batch - b0);
    const snack::SegTable &t = line_table(L, true, nb, false);
    const snack::Plan p = snack::choose_plan(t, nb);
    const float *op = X + b0 * L.in;
    const bool transposed = p.bw > 1;
    if (transposed) {
      cudaError_t e = snack::launch_transpose(op, L.in, nb, L.in, L.d_xt, p.bw, s, true);
      if (e != cudaSuccess) return cuda_fail(h, e, "transpose launch");
      g_launches.fetch_add(1, std::memory_order_relaxed);
      op = L.d_xt;
    }
    cudaError_t e;
    snack::SpmmArgs a = spmm_args(L, t, true, op, Y + b0 * L.out, nb);
    a.prefetch = transposed;
    a.stride = p.bw;
    if (snack::resident_fits(p.bw, L.in, L.csr.nseg, L.nnz)) {
      e = snack::launch_resident_spmm(false, p, a, L.in, L.d_err, true, s);
    } else {
      const snack::Plan q = sub_slices(t, p, nb, &a.nsub);
      const bool two = two_pass(t, q);
      if (two) a.counter = nullptr;
      e = snack::launch_spmm_rows(q, a, true, s);
      if (e == cudaSuccess && two) {
        g_launches.fetch_add(1, std::memory_order_relaxed);
        e = snack::launch_split_sums(q.bw, a, t.nsplit, t.max_parts, true, s);
      }
    }
    if (e != cudaSuccess) return cuda_fail(h, e, "forward launch");
    g_launches.fetch_add(1, std::memory_order_relaxed);
  }
  return SNACK_OK;
}

// One batch slice of the backward: dX (if dX) and / or the weight product
// (into dW, or, with an optimizer step in `opt`, into the values).  One
// launch transposes the slices of dY (and X for the weight product); one
// launch then computes what is asked, both products sharing the transposed
// dY.
snack_status run_backward_slice(snack_handle h, const float *X, const float *dY, float *dX,
                                float *dW, int64_t b0, int nb, cudaStream_t s,
                                const snack::OptArgs *opt = nullptr) {
  snack::Layer &L = h->L;
  const bool fused_opt = opt && opt->kind != snack::kOptNone;
  // Both products in the shared-grid kernel (its grid split by segment
  // counts) walk halved lines on both sides or on neither: from 32-wide
  // slices on, dX's halves summed by the second pass.  10000 x 10000, batch
  // 64: 90 % 307.6 -> 285.7 us, 95 % 157.8 -> 154.1; batch 32: 90 % 194.6 ->
  // 181.9, 95 % 102.5 -> 102.9; batch 16 lost (90 % 116.8 -> 126.7), and so
  // did halving only the rows at batch 32 (194.6 -> 227.8); thirds measured
  // the same at batch 64 and slower at 32 (95 %: 101.4 -> 107.0), and
  // quarters at batch 64 split the layers (90 % 285.8 -> 284.4, 95 % 152.1 ->
  // 156.2).
  const bool both = dX && dW;
  const int w = snack::slice_width(std::min<int64_t>(nb, snack::kMaxSlice));
  const bool fused_halves = both && w >= 32 && w <= snack::kHalfLineWidth &&
                            L.csr_half.nseg > 0 && L.csc_half.nseg > 0 &&
                            !snack::panel_fits(L.csr.panel, w, L.csr.mean_len, L.in);
  const snack::SegTable &tc = fused_halves ? L.csc_half : line_table(L, false, nb, false);
  const snack::SegTable &tr = fused_halves ? L.csr_half : line_table(L, true, nb, !both);
  const snack::Plan pc = snack::choose_plan(tc, nb);
  const snack::Plan pr = snack::choose_plan(tr, nb);
  if (fused_opt && dX) return fail(h, SNACK_ERR_INVALID_ARG, "an optimizer step reads no dX");
  const bool want_w = dW || fused_opt;  // the fused step writes values, not dW
  const float *xt = want_w ? X + b0 * L.in : nullptr;
  const float *dyt = dY + b0 * L.out;
  const bool transposed = pc.bw > 1;
  if (transposed) {
    cudaError_t e =
        want_w ? snack::launch_transpose_pair(dyt, L.out, L.out, L.d_dyt, xt, L.in, L.in, L.d_xt,
                                              nb, pc.bw, s, true)
               : snack::launch_transpose(dyt, L.out, nb, L.out, L.d_dyt, pc.bw, s, true);
    if (e != cudaSuccess) return cuda_fail(h, e, "transpose launch");
    g_launches.fetch_add(1, std::memory_order_relaxed);
    dyt = L.d_dyt;
    if (want_w) xt = L.d_xt;
  }
  snack::SpmmArgs cols;
  if (dX) {
    cols = spmm_args(L, tc, false, dyt, dX + b0 * L.in, nb);
    cols.prefetch = transposed;
    cols.stride = pc.bw;
  }
  snack::SddmmArgs rows;
  if (want_w) {
    rows.seg = tr.d_seg;
    rows.nseg = tr.nseg;
    rows.col = L.d_col;
    rows.xt = xt;
    rows.dyt = dyt;
    rows.dw = dW;
    rows.accumulate = b0 > 0;
    rows.lps = 32;
    rows.prefetch = transposed;
    rows.nsub = 1;
    if (opt) rows.opt = *opt;
  }
  cudaError_t e;
  const bool pan_r =
      want_w && !fused_opt && snack::panel_fits(L.csr.panel, pr.bw, L.csr.mean_len, L.in);
  if (pan_r) {
    // The weight product as a column-panel sweep (long rows): dX, when asked
    // for, in its own launch first, then the sweep as its dependent.
    if (dX) {
      e = snack::resident_fits(pc.bw, L.out, L.csc.nseg, L.nnz)
              ? snack::launch_resident_spmm(cols.perm != nullptr, pc, cols, L.out, L.d_err, true, s)
              : launch_cols(tc, pc, cols, nb, s);
      if (e != cudaSuccess) return cuda_fail(h, e, "backward-input launch");
      g_launches.fetch_add(1, std::memory_order_relaxed);
    }
    snack::PanelArgs pa = {};
    pa.idx = L.d_col;
    pa.src = xt;
    pa.n_op = L.in;
    pa.dyt = dyt;
    pa.dw = dW;
    pa.accumulate = b0 > 0;
    pa.err = L.d_err;
    e = snack::launch_panel_sddmm(pr.bw, L.csr.panel, pa, true, s);
    if (e != cudaSuccess) return cuda_fail(h, e, "backward-weight launch");
    g_launches.fetch_add(1, std::memory_order_relaxed);
    return SNACK_OK;
  }
  const bool res_c = dX && snack::resident_fits(pc.bw, L.out, L.csc.nseg, L.nnz);
  const bool res_r = want_w && !fused_opt && snack::resident_fits(pr.bw, L.in, L.csr.nseg, L.nnz);
  if (want_w && !res_r) rows.nsub = sddmm_subranges(tr, pr);
  if (fused_opt) {  // the optimizer step has its own kernel
    e = snack::launch_sddmm_step(pr, rows, true, s);
    if (e != cudaSuccess) return cuda_fail(h, e, "optimizer step launch");
    g_launches.fetch_add(1, std::memory_order_relaxed);
    return SNACK_OK;
  }
  if ((res_c || res_r) && (!(dX && want_w) || L.nnz >= (int64_t(1) << 19))) {
    // Operand resident in shared memory for at least one product (and, when
    // both are wanted, a layer large enough that a second launch is cheap):
    // one launch per product, the second waiting for the first.
    if (dX) {
      e = res_c ? snack::launch_resident_spmm(cols.perm != nullptr, pc, cols, L.out, L.d_err,
                                              true, s)
                : launch_cols(tc, pc, cols, nb, s);
      if (e != cudaSuccess) return cuda_fail(h, e, "backward-input launch");
      g_launches.fetch_add(1, std::memory_order_relaxed);
    }
    if (want_w) {
      e = res_r ? snack::launch_resident_sddmm(pr, rows, L.in, L.d_err, true, s)
                : snack::launch_sddmm(pr, rows, true, s);
      if (e != cudaSuccess) return cuda_fail(h, e, "backward-weight launch");
      g_launches.fetch_add(1, std::memory_order_relaxed);
    }
    return SNACK_OK;
  }
  if (dX && want_w) {
    const bool two = two_pass(tc, pc, true);
    if (two) cols.counter = nullptr;
    e = snack::launch_backward_fused(pc, cols, pr, rows, true, s);
    if (e == cudaSuccess && two) {
      g_launches.fetch_add(1, std::memory_order_relaxed);
      e = snack::launch_split_sums(pc.bw, cols, tc.nsplit, tc.max_parts, true, s);
    }
  } else if (dX)
    e = launch_cols(tc, pc, cols, nb, s);
  else
    e = snack::launch_sddmm(pr, rows, true, s);
  if (e != cudaSuccess) return cuda_fail(h, e, "backward launch");
  g_launches.fetch_add(1, std::memory_order_relaxed);
  return SNACK_OK;
}

// Batches of 1-4 (slices of 1-4 floats) take the SDDMM with the optimizer
// step fused in; wider ones go through the gradient buffer (see run_opt_step).
constexpr int kFusedStepMaxWidth = 4;

bool step_is_fused(const snack::Layer &L, int64_t batch) {
  return snack::choose_plan(L.csr, std::min<int64_t>(batch, snack::kMaxSlice)).bw <=
         kFusedStepMaxWidth;
}

// Device buffers of an optimizer step, allocated on first use: the gradient
// buffer (unfused batches) and `arrays` state arrays of `kind` (zeroed; all
// state is zeroed again when the kind changes).  If an allocation fails,
// what this call allocated is freed again, so the handle stays as it was.
snack_status ensure_step_buffers(snack_handle h, int kind, int arrays, int64_t batch,
                                 cudaStream_t s) {
  snack::Layer &L = h->L;
  float **made[3];
  int nmade = 0;
  auto undo = [&](cudaError_t e, const char *what) {
    for (int i = 0; i < nmade; ++i) {
      cudaFree(*made[i]);
      *made[i] = nullptr;
    }
    return cuda_fail(h, e, what);
  };
  cudaError_t e;
  size_t acct = 0;
  if (L.nnz > 0 && !step_is_fused(L, batch) && !L.d_gacc) {
    if ((e = snack::dev_alloc(&L.d_gacc, (size_t)L.nnz_pad, &acct)) != cudaSuccess)
      return undo(e, "gradient buffer allocation");
    made[nmade++] = &L.d_gacc;
  }
  for (int i = 0; i < arrays; ++i) {
    if (L.d_opt[i]) continue;
    if ((e = snack::dev_alloc(&L.d_opt[i], (size_t)L.nnz_pad, &acct)) != cudaSuccess)
      return undo(e, "optimizer state allocation");
    made[nmade++] = &L.d_opt[i];
    if ((e = cudaMemsetAsync(L.d_opt[i], 0, (size_t)L.nnz_pad * 4, s)) != cudaSuccess)
      return undo(e, "optimizer state zeroing");
  }
  if (arrays > 0 && L.opt_kind != kind) {
    for (float *p : L.d_opt)
      if (p && (e = cudaMemsetAsync(p, 0, (size_t)L.nnz_pad * 4, s)) != cudaSuccess)
        return undo(e, "optimizer state zeroing");
    L.opt_kind = kind;
  }
  account(L);
  return SNACK_OK;
}

// One optimizer step.  Batches of 1-4 (slices of 1-4 floats): one launch of
// the SDDMM with the step fused in, each entry's gradient updating its value
// and state in place.  Wider: the plain SDDMM (two quads per step, slices of
// up to 256, later slices accumulating) writes the whole batch's gradient
// into the handle's gradient buffer, then a streaming kernel applies the
// step; the fused kernel's one quad per step halves its gathers in flight,
// which at 8+ floats per gathered row costs more than the gradient's round
// trip through memory (10000x10000 @95% Adam at batch 16: 97 -> 58 us).
// The buffers are allocated beforehand (ensure_step_buffers).

snack_status run_opt_step(snack_handle h, const float *X, const float *dY, int64_t batch,
                          snack::OptArgs o, cudaStream_t s) {
  snack::Layer &L = h->L;
  if (L.nnz == 0) return SNACK_OK;
  o.val = L.d_val;
  o.s0 = L.d_opt[0];
  o.s1 = o.kind == snack::kOptAdam ? L.d_opt[1] : nullptr;
  if (o.kind == snack::kOptSgd && o.mom == 0.f) o.s0 = nullptr;
  snack_status st;
  if (step_is_fused(L, batch)) {
    st = run_backward_slice(h, X, dY, nullptr, nullptr, 0, (int)batch, s, &o);
  } else {
    for (int64_t b0 = 0, nb = 0; b0 < batch; b0 += nb) {
      nb = next_slice(L, batch - b0);
      if ((st = run_backward_slice(h, X, dY, nullptr, L.d_gacc, b0, nb, s)) != SNACK_OK) return st;
    }
    cudaError_t e = snack::launch_opt_apply(o, L.d_gacc, L.nnz, true, s);
    if (e != cudaSuccess) return cuda_fail(h, e, "optimizer step launch");
    g_launches.fetch_add(1, std::memory_order_relaxed);
    st = SNACK_OK;
  }
  if (st != SNACK_OK) return st;
  // The values changed: the column-ordered copy is stale (dX reads through
  // the permutation) until snack_values_changed() re-derives it.  Keeping it
  // current inside the step (a scattered 4-byte store per entry) measured
  // slower than the permutation path it saves.
  L.csc_vals = false;
  return SNACK_OK;
}

bool finite(float x) { return x == x && x - x == 0.f; }

}  // namespace

namespace snack {
cudaError_t device_malloc(void **p, size_t bytes) {
  int64_t left = g_fail_alloc.load(std::memory_order_relaxed);
  while (left >= 0 && !g_fail_alloc.compare_exchange_weak(left, left - 1)) {
  }
  if (left == 0) {
    *p = nullptr;
    return cudaErrorMemoryAllocation;
  }
  return cudaMalloc(p, bytes);
}

// Failures of entry points that have no handle report through
// snack_last_error(NULL), like snack_create.
void record_thread_error(const std::string &msg) { g_create_error = msg; }
}  // namespace snack

extern "C" {

snack_status snack_create(int64_t out_features, int64_t in_features, int64_t nnz,
                          const int32_t *row, const int32_t *col, const float *val,
                          int ptrs_on_device, void *stream, snack_handle *out) {
  if (!out) return fail(nullptr, SNACK_ERR_INVALID_ARG, "out handle pointer is NULL");
  snack_status st = check_shape(out_features, in_features, nnz);
  if (st != SNACK_OK) return st;
  if (nnz > 0 && (!row || !col))
    return fail(nullptr, SNACK_ERR_INVALID_ARG, "row and col must not be NULL when nnz > 0");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  snack_layer *h = new (std::nothrow) snack_layer();
  if (!h) return fail(nullptr, SNACK_ERR_ALLOC, "host allocation failed");
  cudaError_t e = cudaGetDevice(&h->L.device);
  if (e != cudaSuccess) {
    delete h;
    return fail(nullptr, SNACK_ERR_CUDA, std::string("cudaGetDevice: ") + cudaGetErrorString(e));
  }
  h->L.out = out_features;
  h->L.in = in_features;
  std::string err;
  int32_t *d_row = nullptr, *d_col = nullptr;
  float *d_val = nullptr;
  const int32_t *urow = row, *ucol = col;
  const float *uval = val;
  if (!ptrs_on_device && nnz > 0) {
    // Stage host arrays on the device.
    if ((e = snack::dev_alloc(&d_row, (size_t)nnz, nullptr)) != cudaSuccess ||
        (e = snack::dev_alloc(&d_col, (size_t)nnz, nullptr)) != cudaSuccess ||
        (val && (e = snack::dev_alloc(&d_val, (size_t)nnz, nullptr)) != cudaSuccess) ||
        (e = cudaMemcpyAsync(d_row, row, nnz * 4, cudaMemcpyHostToDevice, s)) != cudaSuccess ||
        (e = cudaMemcpyAsync(d_col, col, nnz * 4, cudaMemcpyHostToDevice, s)) != cudaSuccess ||
        (val && (e = cudaMemcpyAsync(d_val, val, nnz * 4, cudaMemcpyHostToDevice, s)) != cudaSuccess)) {
      cudaFree(d_row);
      cudaFree(d_col);
      cudaFree(d_val);
      delete h;
      return fail(nullptr, e == cudaErrorMemoryAllocation ? SNACK_ERR_ALLOC : SNACK_ERR_CUDA,
                  std::string("staging input: ") + cudaGetErrorString(e));
    }
    urow = d_row;
    ucol = d_col;
    uval = d_val;
  }
  st = snack::build_topology(h->L, nnz, urow, ucol, uval, s, err);
  cudaFree(d_row);
  cudaFree(d_col);
  cudaFree(d_val);
  return finish_create(h, st, err, out);
}

snack_status snack_create_random(int64_t out_features, int64_t in_features, int64_t nnz,
                                 uint64_t seed, void *stream, snack_handle *out,
                                 int64_t *n_trials) {
  if (!out) return fail(nullptr, SNACK_ERR_INVALID_ARG, "out handle pointer is NULL");
  snack_status st = check_shape(out_features, in_features, nnz);
  if (st != SNACK_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  snack_layer *h = new (std::nothrow) snack_layer();
  if (!h) return fail(nullptr, SNACK_ERR_ALLOC, "host allocation failed");
  cudaError_t e = cudaGetDevice(&h->L.device);
  if (e != cudaSuccess) {
    delete h;
    return fail(nullptr, SNACK_ERR_CUDA, std::string("cudaGetDevice: ") + cudaGetErrorString(e));
  }
  h->L.out = out_features;
  h->L.in = in_features;
  std::string err;
  int32_t *d_row = nullptr, *d_col = nullptr;
  if ((e = snack::dev_alloc(&d_row, (size_t)std::max<int64_t>(nnz, 1), nullptr)) != cudaSuccess ||
      (e = snack::dev_alloc(&d_col, (size_t)std::max<int64_t>(nnz, 1), nullptr)) != cudaSuccess) {
    cudaFree(d_row);
    delete h;
    return fail(nullptr, SNACK_ERR_ALLOC, std::string("cudaMalloc: ") + cudaGetErrorString(e));
  }
  int64_t trials = 0;
  st = snack::draw_random_cells(out_features, in_features, nnz, seed, d_row, d_col, &trials, s, err);
  if (st == SNACK_OK) st = snack::build_topology(h->L, nnz, d_row, d_col, nullptr, s, err);
  cudaFree(d_row);
  cudaFree(d_col);
  if (st == SNACK_OK && n_trials) *n_trials = trials;
  return finish_create(h, st, err, out);
}

snack_status snack_forward(snack_handle h, const float *X, float *Y, int64_t batch, void *stream) {
  if (!h) return fail(nullptr, SNACK_ERR_INVALID_ARG, "handle is NULL");
  if (batch < 1) return fail(h, SNACK_ERR_INVALID_ARG, "batch must be >= 1");
  snack_status st;
  if ((st = check_dense(h, X, "X")) != SNACK_OK || (st = check_dense(h, Y, "Y")) != SNACK_OK ||
      (st = check_device(h)) != SNACK_OK)
    return st;
  return run_forward(h, X, Y, batch, static_cast<cudaStream_t>(stream));
}

snack_status snack_backward_input(snack_handle h, const float *dY, float *dX, int64_t batch,
                                  void *stream) {
  if (!h) return fail(nullptr, SNACK_ERR_INVALID_ARG, "handle is NULL");
  if (batch < 1) return fail(h, SNACK_ERR_INVALID_ARG, "batch must be >= 1");
  snack_status st;
  if ((st = check_dense(h, dY, "dY")) != SNACK_OK || (st = check_dense(h, dX, "dX")) != SNACK_OK ||
      (st = check_device(h)) != SNACK_OK)
    return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  for (int64_t b0 = 0, nb = 0; b0 < batch; b0 += nb) {
    nb = next_slice(h->L, batch - b0);
    if ((st = run_backward_slice(h, nullptr, dY, dX, nullptr, b0, nb, s)) != SNACK_OK) return st;
  }
  return SNACK_OK;
}

snack_status snack_backward_weight(snack_handle h, const float *X, const float *dY, float *dW,
                                   int64_t batch, void *stream) {
  if (!h) return fail(nullptr, SNACK_ERR_INVALID_ARG, "handle is NULL");
  if (batch < 1) return fail(h, SNACK_ERR_INVALID_ARG, "batch must be >= 1");
  snack_status st;
  if ((st = check_dense(h, X, "X")) != SNACK_OK || (st = check_dense(h, dY, "dY")) != SNACK_OK ||
      (st = check_dense(h, dW, "dW")) != SNACK_OK || (st = check_device(h)) != SNACK_OK)
    return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  for (int64_t b0 = 0, nb = 0; b0 < batch; b0 += nb) {
    nb = next_slice(h->L, batch - b0);
    if ((st = run_backward_slice(h, X, dY, nullptr, dW, b0, nb, s)) != SNACK_OK) return st;
  }
  return SNACK_OK;
}

snack_status snack_backward(snack_handle h, const float *X, const float *dY, float *dX, float *dW,
                            int64_t batch, void *stream) {
  if (!h) return fail(nullptr, SNACK_ERR_INVALID_ARG, "handle is NULL");
  if (batch < 1) return fail(h, SNACK_ERR_INVALID_ARG, "batch must be >= 1");
  if (!dX && !dW) return SNACK_OK;
  snack_status st;
  if ((st = check_dense(h, dY, "dY")) != SNACK_OK || (st = check_device(h)) != SNACK_OK) return st;
  if (dX && (st = check_dense(h, dX, "dX")) != SNACK_OK) return st;
  if (dW && ((st = check_dense(h, dW, "dW")) != SNACK_OK || (st = check_dense(h, X, "X")) != SNACK_OK))
    return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  snack::Layer &L = h->L;
  for (int64_t b0 = 0, nb = 0; b0 < batch; b0 += nb) {
    nb = next_slice(L, batch - b0);
    if ((st = run_backward_slice(h, X, dY, dX, dW, b0, nb, s)) != SNACK_OK) return st;
  }
  return SNACK_OK;
}

snack_status snack_prune_regrow(snack_handle h, float prune_frac, uint64_t seed, void *stream,
                                int64_t *n_pruned, int64_t *n_trials) {
  if (!h) return fail(nullptr, SNACK_ERR_INVALID_ARG, "handle is NULL");
  if (!(prune_frac >= 0.0f) || prune_frac > 1.0f)
    return fail(h, SNACK_ERR_INVALID_ARG, "prune_frac must be in [0, 1]");
  snack_status st = check_device(h);
  if (st != SNACK_OK) return st;
  std::string err;
  int64_t p = 0, t = 0;
  st = snack::prune_regrow(h->L, prune_frac, seed, &p, &t, static_cast<cudaStream_t>(stream), err);
  if (st != SNACK_OK) return fail(h, st, err);
  account(h->L);
  if (n_pruned) *n_pruned = p;
  if (n_trials) *n_trials = t;
  return SNACK_OK;
}

snack_status snack_sgd_step(snack_handle h, const float *X, const float *dY, int64_t batch,
                            float lr, float momentum, float weight_decay, void *stream) {
  if (!h) return fail(nullptr, SNACK_ERR_INVALID_ARG, "handle is NULL");
  if (batch < 1) return fail(h, SNACK_ERR_INVALID_ARG, "batch must be >= 1");
  if (!finite(lr) || !finite(momentum) || momentum < 0.f || !finite(weight_decay))
    return fail(h, SNACK_ERR_INVALID_ARG, "lr and weight_decay must be finite, momentum >= 0");
  snack_status st;
  if ((st = check_dense(h, X, "X")) != SNACK_OK || (st = check_dense(h, dY, "dY")) != SNACK_OK ||
      (st = check_device(h)) != SNACK_OK)
    return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  snack::OptArgs o;
  o.kind = snack::kOptSgd;
  o.lr = lr;
  o.mom = momentum;
  o.wd = weight_decay;
  if ((st = ensure_step_buffers(h, snack::kOptSgd, momentum != 0.f ? 1 : 0, batch, s)) != SNACK_OK)
    return st;
  return run_opt_step(h, X, dY, batch, o, s);
}

snack_status snack_adam_step(snack_handle h, const float *X, const float *dY, int64_t batch,
                             float lr, float beta1, float beta2, float eps, float weight_decay,
                             int64_t step, void *stream) {
  if (!h) return fail(nullptr, SNACK_ERR_INVALID_ARG, "handle is NULL");
  if (batch < 1) return fail(h, SNACK_ERR_INVALID_ARG, "batch must be >= 1");
  if (step < 1) return fail(h, SNACK_ERR_INVALID_ARG, "step must be >= 1");
  if (!finite(lr) || !finite(weight_decay) || !(beta1 >= 0.f && beta1 < 1.f) ||
      !(beta2 >= 0.f && beta2 < 1.f) || !(eps > 0.f) || !finite(eps))
    return fail(h, SNACK_ERR_INVALID_ARG,
                "need finite lr, weight_decay; betas in [0, 1); finite eps > 0");
  snack_status st;
  if ((st = check_dense(h, X, "X")) != SNACK_OK || (st = check_dense(h, dY, "dY")) != SNACK_OK ||
      (st = check_device(h)) != SNACK_OK)
    return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if ((st = ensure_step_buffers(h, snack::kOptAdam, 2, batch, s)) != SNACK_OK) return st;
  const double bc1 = 1.0 - std::pow((double)beta1, (double)step);
  const double bc2 = 1.0 - std::pow((double)beta2, (double)step);
  snack::OptArgs o;
  o.kind = snack::kOptAdam;
  o.wd = weight_decay;
  o.b1 = beta1;
  o.c1 = (float)(1.0 - (double)beta1);
  o.b2 = beta2;
  o.c2 = (float)(1.0 - (double)beta2);
  o.eps = eps;
  o.step = (float)((double)lr / bc1);
  o.sbc2 = (float)std::sqrt(bc2);
  return run_opt_step(h, X, dY, batch, o, s);
}

snack_status snack_optimizer_state(snack_handle h, int which, float **dev_state) {
  if (!h || !dev_state) return fail(h, SNACK_ERR_INVALID_ARG, "NULL argument");
  if (which < 0 || which > 1) return fail(h, SNACK_ERR_INVALID_ARG, "which must be 0 or 1");
  if (!h->L.d_opt[which])
    return fail(h, SNACK_ERR_INVALID_ARG, "no optimizer state of that index yet");
  *dev_state = h->L.d_opt[which];
  return SNACK_OK;
}

snack_status snack_values(snack_handle h, float **dev_val) {
  if (!h || !dev_val) return fail(h, SNACK_ERR_INVALID_ARG, "NULL argument");
  *dev_val = h->L.d_val;
  // The caller may write the values from now on: the column-ordered copy
  // can no longer be trusted.
  h->L.values_shared = true;
  h->L.csc_vals = false;
  return SNACK_OK;
}

snack_status snack_values_changed(snack_handle h, void *stream) {
  if (!h) return fail(nullptr, SNACK_ERR_INVALID_ARG, "handle is NULL");
  snack_status st = check_device(h);
  if (st != SNACK_OK) return st;
  h->L.values_shared = false;
  std::string err;
  if ((st = snack::refresh_csc_values(h->L, static_cast<cudaStream_t>(stream), err)) != SNACK_OK)
    return fail(h, st, err);
  return SNACK_OK;
}

snack_status snack_export(snack_handle h, int32_t *row, int32_t *col, float *val, int ptrs_on_device,
                          void *stream) {
  if (!h) return fail(nullptr, SNACK_ERR_INVALID_ARG, "handle is NULL");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const cudaMemcpyKind kind = ptrs_on_device ? cudaMemcpyDeviceToDevice : cudaMemcpyDeviceToHost;
  const size_t bytes = (size_t)h->L.nnz * 4;
  cudaError_t e = cudaSuccess;
  if (bytes && row && (e = cudaMemcpyAsync(row, h->L.d_row, bytes, kind, s)) != cudaSuccess)
    return cuda_fail(h, e, "export row");
  if (bytes && col && (e = cudaMemcpyAsync(col, h->L.d_col, bytes, kind, s)) != cudaSuccess)
    return cuda_fail(h, e, "export col");
  if (bytes && val && (e = cudaMemcpyAsync(val, h->L.d_val, bytes, kind, s)) != cudaSuccess)
    return cuda_fail(h, e, "export val");
  if ((e = cudaStreamSynchronize(s)) != cudaSuccess) return cuda_fail(h, e, "export sync");
  return SNACK_OK;
}

snack_status snack_export_segments(snack_handle h, int32_t *row_ptr, int32_t *col_ptr,
                                   int32_t *csc_row, int32_t *csc_perm, void *stream) {
  if (!h) return fail(nullptr, SNACK_ERR_INVALID_ARG, "handle is NULL");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const snack::Layer &L = h->L;
  cudaError_t e = cudaSuccess;
  const auto d2h = cudaMemcpyDeviceToHost;
  if (row_ptr && (e = cudaMemcpyAsync(row_ptr, L.d_row_ptr, (L.out + 1) * 4, d2h, s)) != cudaSuccess)
    return cuda_fail(h, e, "export row_ptr");
  if (col_ptr && (e = cudaMemcpyAsync(col_ptr, L.d_col_ptr, (L.in + 1) * 4, d2h, s)) != cudaSuccess)
    return cuda_fail(h, e, "export col_ptr");
  if (L.nnz && csc_row && (e = cudaMemcpyAsync(csc_row, L.d_csc_row, L.nnz * 4, d2h, s)) != cudaSuccess)
    return cuda_fail(h, e, "export csc_row");
  if (L.nnz && csc_perm && (e = cudaMemcpyAsync(csc_perm, L.d_csc_perm, L.nnz * 4, d2h, s)) != cudaSuccess)
    return cuda_fail(h, e, "export csc_perm");
  if ((e = cudaStreamSynchronize(s)) != cudaSuccess) return cuda_fail(h, e, "export sync");
  return SNACK_OK;
}

snack_status snack_plan(snack_handle h, int op, int64_t batch, int32_t *slice_width,
                        int32_t *lanes_per_segment, int64_t *segments, int32_t *resident) {
  if (!h) return fail(nullptr, SNACK_ERR_INVALID_ARG, "handle is NULL");
  if (op < 0 || op > 2 || batch < 1) return fail(h, SNACK_ERR_INVALID_ARG, "bad op or batch");
  const snack::Layer &L = h->L;
  const int nb = next_slice(L, batch);  // the first slice
  const snack::SegTable &t = line_table(L, op != 1, nb, op == 2);
  const snack::SegTable &base = op == 1 ? L.csc : L.csr;
  const snack::Plan p = snack::choose_plan(t, nb);
  if (slice_width) *slice_width = p.bw;
  if (lanes_per_segment) *lanes_per_segment = p.lanes;
  if (segments) *segments = t.nseg;
  // as the launches decide: the panel partition and the resident operand
  // belong to the row and column tables themselves
  if (resident)
    *resident = op == 2 && snack::panel_fits(L.csr.panel, p.bw, L.csr.mean_len, L.in)
                    ? 2
                    : (snack::resident_fits(p.bw, op == 1 ? L.out : L.in, base.nseg, L.nnz) ? 1
                                                                                            : 0);
  return SNACK_OK;
}

uint64_t snack_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

void snack_debug_fail_alloc(int64_t after) {
  g_fail_alloc.store(after < 0 ? -1 : after, std::memory_order_relaxed);
}

snack_status snack_selftest_wait(void *stream, int *timed_out) {
  if (!timed_out) return fail(nullptr, SNACK_ERR_INVALID_ARG, "timed_out is NULL");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int *d = nullptr;
  cudaError_t e = snack::dev_alloc(&d, 1, nullptr);
  if (e != cudaSuccess) return cuda_fail(nullptr, e, "self-test flag allocation");
  int v = 0;
  if ((e = cudaMemsetAsync(d, 0, sizeof(int), s)) != cudaSuccess ||
      (e = snack::launch_wait_selftest(d, s)) != cudaSuccess ||
      (e = cudaMemcpyAsync(&v, d, sizeof(int), cudaMemcpyDeviceToHost, s)) != cudaSuccess ||
      (e = cudaStreamSynchronize(s)) != cudaSuccess) {
    cudaFree(d);
    return cuda_fail(nullptr, e, "self-test");
  }
  cudaFree(d);
  *timed_out = v;
  return SNACK_OK;
}

snack_status snack_device_error(snack_handle h, int *flag, void *stream) {
  if (!h || !flag) return fail(h, SNACK_ERR_INVALID_ARG, "NULL argument");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int v = 0;
  cudaError_t e;
  if ((e = cudaMemcpyAsync(&v, h->L.d_err, sizeof(int), cudaMemcpyDeviceToHost, s)) != cudaSuccess ||
      (e = cudaMemsetAsync(h->L.d_err, 0, sizeof(int), s)) != cudaSuccess ||
      (e = cudaStreamSynchronize(s)) != cudaSuccess)
    return cuda_fail(h, e, "reading the device error flag");
  *flag = v;
  return SNACK_OK;
}

int64_t snack_nnz(snack_handle h) { return h ? h->L.nnz : -1; }
int64_t snack_out_features(snack_handle h) { return h ? h->L.out : -1; }
int64_t snack_in_features(snack_handle h) { return h ? h->L.in : -1; }
size_t snack_device_bytes(snack_handle h) { return h ? h->L.device_bytes : 0; }

const char *snack_last_error(snack_handle h) {
  return h ? h->L.last_error.c_str() : g_create_error.c_str();
}

const char *snack_status_string(snack_status s) {
  switch (s) {
    case SNACK_OK: return "ok";
    case SNACK_ERR_INVALID_ARG: return "invalid argument";
    case SNACK_ERR_OUT_OF_RANGE: return "index out of range";
    case SNACK_ERR_DUPLICATE: return "duplicate (row, col)";
    case SNACK_ERR_ALLOC: return "allocation failed";
    case SNACK_ERR_CUDA: return "CUDA error";
    case SNACK_ERR_UNSUPPORTED: return "unsupported size";
    case SNACK_ERR_TIMEOUT: return "bounded search gave up";
  }
  return "unknown status";
}

void snack_destroy(snack_handle h) {
  if (!h) return;
  int prev = -1;
  const bool switched = cudaGetDevice(&prev) == cudaSuccess && prev != h->L.device &&
                        cudaSetDevice(h->L.device) == cudaSuccess;
  cudaDeviceSynchronize();
  snack::free_layer(h->L);
  if (switched) cudaSetDevice(prev);
  delete h;
}

}  // extern "C"
