/*
 * snack.h - C ABI of the SNACK truly-sparse linear layer for NVIDIA GB300
 * (sm_103a).
 *
 * The layer keeps its weight W (out_features x in_features) only as its
 * stored nonzeros (row, col, val) and never forms a dense out x in matrix
 * ("Beyond Masked Sparsity: SNACK Enables Truly Sparse Neural Networks on
 * GPU", §3 and Appendix F "End-to-end sparsity").  The operations are
 *
 *   forward           Y  = X W^T                  (§3.1 Algorithm 1)
 *   backward_input    dX = dY W                   (§3.4; Appendix F, W^T by
 *                                                  swapping the index arrays)
 *   backward_weight   dW[k] = sum_b dY[b,row_k] X[b,col_k], only at the
 *                     stored entries              (§3.4; Appendix F)
 *   prune_regrow      magnitude prune + uniform regrow (Appendix G, with the
 *                     regrow draw of §3.3 Algorithm 2)
 *
 * Conventions used by every call:
 *   - Indices are 0-based int32.  Stored entries are kept in CANONICAL ORDER:
 *     rows ascending, columns ascending within a row.  snack_values(),
 *     snack_export() and the dW output of the backward calls use that order.
 *   - X is [batch][in_features], Y and dY are [batch][out_features], dX is
 *     [batch][in_features]: dense, row-major, contiguous fp32 (the PyTorch
 *     nn.Linear layout).  Outputs are overwritten, never accumulated into.
 *   - `stream` is a cudaStream_t passed as void* (NULL = the legacy default
 *     stream).  Compute calls are asynchronous on that stream; the caller
 *     owns every X / Y / dY / dX / dW buffer, which must be device memory,
 *     16-byte aligned.
 *   - The handle owns the topology, the values and a workspace on the
 *     device that was current at creation.  Calls must run with that device
 *     current.  Use one handle from one stream at a time: calls on the same
 *     handle that overlap on the GPU share its workspace and race.
 *   - No call aborts, traps or prints.  Every call returns a snack_status;
 *     snack_last_error() gives a one-line reason.  A call that fails leaves
 *     the handle as it was.
 *   - Limits: 1 <= out_features, in_features < 2^31; 0 <= nnz < 2^31 and
 *     nnz <= out_features * in_features; batch >= 1 (any size: batches above
 *     256 run as consecutive slices of 256, each padded to a power of two).
 */
#ifndef SNACK_H
#define SNACK_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct snack_layer *snack_handle;

typedef enum {
  SNACK_OK = 0,
  SNACK_ERR_INVALID_ARG = 1,  /* null / misaligned pointer, bad size        */
  SNACK_ERR_OUT_OF_RANGE = 2, /* an index outside [0,out) x [0,in)          */
  SNACK_ERR_DUPLICATE = 3,    /* the same (row, col) stored twice           */
  SNACK_ERR_ALLOC = 4,        /* device or host allocation failed           */
  SNACK_ERR_CUDA = 5,         /* a CUDA runtime call failed                 */
  SNACK_ERR_UNSUPPORTED = 6,  /* size beyond a documented limit             */
  SNACK_ERR_TIMEOUT = 7       /* a bounded search gave up (prune/regrow)    */
} snack_status;

/*
 * Build a layer from a COO triple given in any order (Appendix B, Table 7:
 * the COO, CSR and CSC forms of one matrix).  The library validates the
 * indices, sorts the entries into canonical order and builds, on the
 * device, the row segmentation (CSR index pointer, out_features+1 entries)
 * and the column segmentation (CSC index pointer, in_features+1 entries,
 * plus the row index and canonical position of every entry in column
 * order).  These are rebuilt only when the topology changes.
 *
 *   row, col  [nnz] int32 indices; val [nnz] fp32 values or NULL (zeros).
 *   ptrs_on_device  1 if row/col/val are device pointers, 0 if host.
 *   out       receives the new handle (unchanged on failure).
 * Errors: SNACK_ERR_OUT_OF_RANGE or SNACK_ERR_DUPLICATE (no entry is summed
 * or dropped), SNACK_ERR_INVALID_ARG, SNACK_ERR_ALLOC, SNACK_ERR_CUDA.
 * Synchronises `stream`.
 */
snack_status snack_create(int64_t out_features, int64_t in_features, int64_t nnz,
                          const int32_t *row, const int32_t *col, const float *val,
                          int ptrs_on_device, void *stream, snack_handle *out);

/*
 * Build a layer whose nnz stored cells are drawn on the device by the
 * uniform connection initializer (§3.3 Algorithm 2): candidate t is cell
 * floor(x_t * out*in / 2^64) of the row-major cell numbering, where x_t is
 * draw t of the counter-based SplitMix64 stream started at `seed` (the
 * finaliser applied to seed + (t+1) * 0x9E3779B97F4A7C15); a candidate
 * already drawn is rejected.  Values start at 0 (write them through
 * snack_values(), then call snack_values_changed()).  n_trials (may be
 * NULL) receives the number of
 * candidates drawn.  Synchronises `stream`.
 */
snack_status snack_create_random(int64_t out_features, int64_t in_features, int64_t nnz,
                                 uint64_t seed, void *stream, snack_handle *out,
                                 int64_t *n_trials);

/*
 * Y = X W^T (§3.1 Algorithm 1; Y^T = C, X^T = B in the paper's notation).
 *   X [batch][in_features] in, Y [batch][out_features] out (overwritten).
 * Asynchronous on `stream`.
 */
snack_status snack_forward(snack_handle h, const float *X, float *Y, int64_t batch,
                           void *stream);

/*
 * dX = dY W, the input gradient W^T (dL/dA) of §3.4, evaluated over the
 * column segmentation (W^T has W's support with the index arrays swapped,
 * Appendix F).  dY [batch][out_features] in, dX [batch][in_features] out.
 */
snack_status snack_backward_input(snack_handle h, const float *dY, float *dX,
                                  int64_t batch, void *stream);

/*
 * Sparse outer-product weight gradient (§3.4; Appendix F, the mini-batch sum
 * of rank-1 terms restricted to supp(W)):
 *   dW[k] = sum_{b<batch} dY[b][row_k] * X[b][col_k]   for each stored k,
 * written in canonical order (nnz floats; aligned with snack_values()).
 */
snack_status snack_backward_weight(snack_handle h, const float *X, const float *dY,
                                   float *dW, int64_t batch, void *stream);

/*
 * Both backward products of §3.4 in one call: dX as snack_backward_input and
 * dW as snack_backward_weight, sharing one transposed copy of dY.  Either
 * output may be NULL to skip it.
 */
snack_status snack_backward(snack_handle h, const float *X, const float *dY, float *dX,
                            float *dW, int64_t batch, void *stream);

/*
 * One optimizer step on the stored entries from the weight gradient.
 * §3.4: the gradient exists only at supp(W), so only the nnz stored values
 * are trained (frozen cells see no gradient); §4.1 trains with SGD and
 * Appendix G with Adam.  For every stored entry k, with
 *   g_k = sum_{b<batch} dY[b][row_k] * X[b][col_k] + weight_decay * val_k
 * (X, dY as for snack_backward_weight; dW is never written):
 *   snack_sgd_step:  momentum > 0:  buf_k = momentum * buf_k + g_k,
 *                                   val_k -= lr * buf_k
 *                    momentum == 0: val_k -= lr * g_k   (no state)
 *   snack_adam_step (Kingma and Ba, ICLR 2015; step = t >= 1):
 *                    m_k = beta1 m_k + (1 - beta1) g_k
 *                    v_k = beta2 v_k + (1 - beta2) g_k^2
 *                    val_k -= lr / (1 - beta1^t) * m_k
 *                             / (sqrt(v_k) / sqrt(1 - beta2^t) + eps)
 * (the conventions of torch.optim.SGD without dampening and torch.optim.Adam).
 * Values change in place: compute dX (snack_backward_input, which reads
 * them) before the step.  The column-ordered value copy becomes stale (see
 * snack_values).
 *
 * State: nnz-long fp32 arrays owned by the handle, in canonical order
 * (snack_optimizer_state).  The first step that needs them allocates and
 * zeroes them (that call allocates device memory, so make it outside graph
 * capture); a step of the other optimizer kind zeroes them first.  Batches
 * of 1-4 compute the gradient and the step in one kernel; larger batches
 * write the gradient into an nnz-long buffer of the handle (allocated on
 * first use, same capture rule) and apply the step in a second kernel.
 * snack_prune_regrow keeps each surviving entry's state and starts regrown
 * entries from zero.  Errors: SNACK_ERR_INVALID_ARG for non-finite lr /
 * weight_decay, momentum < 0, betas outside [0, 1), eps <= 0, step < 1,
 * batch < 1 or misaligned X / dY.  Asynchronous on `stream`.
 */
snack_status snack_sgd_step(snack_handle h, const float *X, const float *dY, int64_t batch,
                            float lr, float momentum, float weight_decay, void *stream);
snack_status snack_adam_step(snack_handle h, const float *X, const float *dY, int64_t batch,
                             float lr, float beta1, float beta2, float eps, float weight_decay,
                             int64_t step, void *stream);

/*
 * Device pointer to optimizer state array `which` (nnz floats, canonical
 * order, owned by the handle): 0 = SGD momentum buffer or Adam first moment,
 * 1 = Adam second moment.  SNACK_ERR_INVALID_ARG when that array does not
 * exist yet.  The caller may read or overwrite it (e.g. to checkpoint and
 * restore); the pointer stays valid until snack_destroy.
 */
snack_status snack_optimizer_state(snack_handle h, int which, float **dev_state);

/*
 * One topology update (Appendix G "Sparsity schedule and DST"):
 *  1. prune P = floor((double)prune_frac * nnz) stored entries with the
 *     smallest |val|: ordered by the bit pattern of |val| as an unsigned
 *     integer (-0 equals +0, NaN sorts above +inf), ties by canonical
 *     position;
 *  2. regrow P cells with Algorithm 2's rejection draw (the SplitMix64
 *     stream of snack_create_random, started at `seed`), rejecting cells
 *     held by a surviving entry or already regrown; just-pruned cells may be
 *     drawn again;
 *  3. survivors keep their values, regrown entries get 0; the result is put
 *     back into canonical order and the segmentations are rebuilt.
 * nnz is unchanged.  n_pruned / n_trials (either may be NULL) receive P and
 * the number of candidates drawn.  Pointers previously returned by
 * snack_values() stay valid.  Synchronises `stream`.  SNACK_ERR_TIMEOUT if
 * 2^40 candidates do not yield P fresh cells.
 */
snack_status snack_prune_regrow(snack_handle h, float prune_frac, uint64_t seed,
                                void *stream, int64_t *n_pruned, int64_t *n_trials);

/*
 * Device pointer to the nnz stored values in canonical order.  The caller
 * may read and write them in place (e.g. an optimizer step); they stay
 * valid until snack_destroy().
 *
 * The handle also keeps the values in column order, so that dX streams them
 * instead of reading each through the column permutation (creation and
 * snack_prune_regrow derive it).  It is trusted only while the values stay
 * as they were when it was derived: handing out this writable pointer, or an
 * optimizer step (snack_sgd_step / snack_adam_step), makes it stale, and dX then reads the values through
 * the permutation (same results, slower) until snack_values_changed().
 * Layers whose values stay fixed across many backward calls (a frozen layer,
 * repeated evaluation) gain from calling it once.
 */
snack_status snack_values(snack_handle h, float **dev_val);

/*
 * Tell the handle that the values will not change for a while (the caller
 * has finished writing them through the snack_values() pointer, or a run of
 * optimizer steps is over): re-derives the column-ordered copy
 * (asynchronous on `stream`, one gather of the values) and lets dX stream
 * it.  The library then assumes the values change only through its own
 * calls until snack_values() is called again; an optimizer step makes the
 * copy stale again.  The paper has no counterpart to this call; it
 * exists only for the column-ordered copy.
 */
snack_status snack_values_changed(snack_handle h, void *stream);

/*
 * Copy the stored entries out in canonical order: row, col [nnz] int32 and
 * val [nnz] fp32 (any may be NULL).  ptrs_on_device says whether the
 * destinations are device (1) or host (0) memory.  Synchronises `stream`.
 */
snack_status snack_export(snack_handle h, int32_t *row, int32_t *col, float *val,
                          int ptrs_on_device, void *stream);

/*
 * Copy the segmentations to host memory (any pointer may be NULL):
 * row_ptr [out_features+1], col_ptr [in_features+1], csc_row [nnz],
 * csc_perm [nnz] (canonical position of the s-th entry in column order).
 * Synchronises `stream`.
 */
snack_status snack_export_segments(snack_handle h, int32_t *row_ptr, int32_t *col_ptr,
                                   int32_t *csc_row, int32_t *csc_perm, void *stream);

/*
 * Which kernel variant a call would run: for op 0 = forward, 1 =
 * backward_input, 2 = backward_weight and the given batch, returns the
 * width of its first batch slice (1, 2, 4, 8, 16, 32, 64, 128 or 256; on
 * layers of 2^21+ entries a batch just above a power of two w >= 32 runs as
 * a slice of w and one of the remainder), the lanes that
 * share one row (or column) segment (the launch may halve them when that
 * keeps every segment in one wave of resident teams), the number of
 * segments (on layers of 2^21+ entries whose lines average 400+ entries,
 * 64-wide slices and the wider ones of op 2 walk every line in four parts
 * and 32-wide slices of op 2 in two, so four or two times the lines), and
 * where the dense operand is
 * gathered from: 0 = global memory
 * (through L1), 1 = a copy of the whole operand in every block's shared
 * memory, 2 = shared memory one column panel at a time (the column-panel
 * kernels of slices of 8-64 floats on layers with a panel partition).  Any
 * output may be NULL.  Pure host query.
 */
snack_status snack_plan(snack_handle h, int op, int64_t batch, int32_t *slice_width,
                        int32_t *lanes_per_segment, int64_t *segments, int32_t *resident);

/*
 * Forward pass Y = X W^T for callers that cannot allocate device memory.
 * The paper has no counterpart to this entry point; it exists for callers
 * that hold no allocation rights when they run the layer: serving loops
 * whose device memory is already reserved by another allocator (a pool that
 * has taken all free memory at start-up), latency-critical paths where an
 * allocation's implicit device synchronisation is not acceptable, and
 * plug-in code running inside a host framework that owns all device
 * allocation.  It needs no handle and allocates nothing: no cudaMalloc,
 * cudaFree or allocating library call.
 *
 *   row_ptr [out_features+1], col [nnz], val [nnz]: a CSR layout of W in the
 *     caller's device memory, e.g. as exported by snack_export_segments()
 *     and snack_export().  Not validated: row_ptr must be non-decreasing
 *     with row_ptr[0] = 0 and row_ptr[out_features] = nnz, and every col
 *     must lie in [0, in_features).  col and val must be 16-byte aligned.
 *   X [batch][in_features] in, Y [batch][out_features] out (overwritten),
 *     16-byte aligned device memory, as for snack_forward().
 * Its only scratch is a fixed 8 MiB array (2^21 floats) in the library's
 * device memory, which every GPU that loads the library holds until the
 * process exits.  It holds the transposed X slice, so in_features times the
 * batch slice width (batch rounded up to a power of two, at most 64; no
 * scratch for batch 1) must not exceed 2^21, else SNACK_ERR_UNSUPPORTED.
 * The scratch is rewritten in full by every call.  All calls share it:
 * calls whose work overlaps on the GPU (other streams, other threads) race.
 * The first call on a device looks up the scratch's device address and
 * keeps it for the life of the process; make that first call before any
 * stream capture.  cudaDeviceReset() unloads the library's device code and
 * makes the kept address stale: do not call this entry point on a device
 * after resetting it.  Y must not overlap X (SNACK_ERR_INVALID_ARG).  Rows
 * are not split, so a few very long rows run slower than with
 * snack_forward().  Errors are reported through snack_last_error(NULL).
 * Asynchronous on `stream`.
 */
snack_status snack_forward_csr_static(int64_t out_features, int64_t in_features, int64_t nnz,
                                      const int32_t *row_ptr, const int32_t *col,
                                      const float *val, const float *X, float *Y,
                                      int64_t batch, void *stream);

/*
 * Read and clear the handle's device error flag: *flag = 1 if, since the
 * last read, a kernel of this handle gave up a bounded wait on one of its
 * own shared-memory copies (its outputs for that call are then not to be
 * trusted); 0 otherwise.  Kernels never trap or hang on such a failure.
 * Synchronises `stream`.
 */
snack_status snack_device_error(snack_handle h, int *flag, void *stream);

/*
 * Self-test of that failure path: one block waits, with a short bound, on a
 * device barrier that nothing completes, and records the time-out the way
 * the kernels record a failed wait.  *timed_out receives 1 when the wait
 * gave up as designed; the context stays usable afterwards.  The paper has
 * no counterpart to this call; it exists to test the bounded waits without
 * faulting or hanging the GPU.  Allocates a device int; synchronises
 * `stream`.  Errors report through snack_last_error(NULL).
 */
snack_status snack_selftest_wait(void *stream, int *timed_out);

/*
 * Kernel launches this library has issued in the process so far (all
 * handles, all threads).  Launches recorded into a CUDA graph count once,
 * at capture.  For accounting and tests.
 */
uint64_t snack_launch_count(void);

/*
 * Test hook for the out-of-memory paths: after `after` more device
 * allocations by this library (0 = the next one), one allocation reports
 * cudaErrorMemoryAllocation without allocating, and the hook disarms
 * itself; a negative value disarms it.  Process-wide (all handles and
 * threads).  A call that meets the failure returns SNACK_ERR_ALLOC, frees
 * what it had allocated and leaves an existing handle as it was.  The paper
 * has no counterpart; it exists so that those paths can be tested.
 */
void snack_debug_fail_alloc(int64_t after);

int64_t snack_nnz(snack_handle h);
int64_t snack_out_features(snack_handle h);
int64_t snack_in_features(snack_handle h);

/* Device bytes held by the handle (topology, values, workspace). */
size_t snack_device_bytes(snack_handle h);

/*
 * One-line text for the last failure on this handle; with h == NULL, the
 * last failure of snack_create / snack_create_random on the calling thread.
 * The string lives until the next call on the same handle / thread.
 */
const char *snack_last_error(snack_handle h);

const char *snack_status_string(snack_status s);

/* Free everything the handle owns (synchronises its device).  NULL is a no-op. */
void snack_destroy(snack_handle h);

#ifdef __cplusplus
}
#endif

#endif /* SNACK_H */
