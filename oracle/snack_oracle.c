/*
 * Plain CPU oracle for the SNACK truly-sparse linear layer.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library links, loads or
 * calls this file; only the test suite, the smoke check and the benchmark's
 * CPU-baseline leg do.  It shares no code, header, table or helper with the
 * CUDA library: every routine here is written straight from the paper
 * "Beyond Masked Sparsity: SNACK Enables Truly Sparse Neural Networks on GPU"
 * (Badour, van Keulen, Mocanu), cited per function by section, algorithm,
 * table or appendix.
 *
 * Conventions (the paper's §3.1 notation A = W, B = X^T, C = Y^T):
 *   W  : out x in, stored only as nonzeros (row, col, val), 0-based indices
 *   X  : [B][in]  row-major fp32      Y  : [B][out] row-major fp32
 *   dY : [B][out]                      dX : [B][in]
 *   dW : [nnz] in canonical order (rows ascending, then columns ascending)
 * Floating-point sums are formed in double and rounded once to float.  Each
 * numeric routine can also return S = sum of |term| per output element (in
 * double), the scale used by the parity tolerance |gpu - oracle| <= 1e-5 * S.
 *
 * Parity pins for every routine live in tests/test_oracle_pins.py.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_OK 0
#define ORACLE_ERR_RANGE 1
#define ORACLE_ERR_DUPLICATE 2
#define ORACLE_ERR_ALLOC 3
#define ORACLE_ERR_ARG 4

/* ------------------------------------------------------------------------ */
/* Canonical order and CSR / CSC segmentation                               */
/* Appendix B, Table 7 (COO, CSR, CSC of the same matrix).                  */
/* ------------------------------------------------------------------------ */

typedef struct {
  int64_t a; /* primary key   */
  int64_t b; /* secondary key */
  int64_t idx;
} key3;

static int cmp_key3(const void *p, const void *q) {
  const key3 *x = (const key3 *)p, *y = (const key3 *)q;
  if (x->a != y->a) return x->a < y->a ? -1 : 1;
  if (x->b != y->b) return x->b < y->b ? -1 : 1;
  if (x->idx != y->idx) return x->idx < y->idx ? -1 : 1;
  return 0;
}

/*
 * Sort the user's COO triple into canonical order (by row, then column),
 * reject out-of-range and repeated coordinates, and build:
 *   c_row, c_col, c_val [nnz]   canonical COO (c_val = 0 when val is NULL)
 *   c_src [nnz]                 user position of canonical entry k
 *   row_ptr [out+1]             CSR index pointer (Table 7 "CSR indptr")
 *   col_ptr [in+1]              CSC index pointer (Table 7 "CSC indptr")
 *   csc_row [nnz]               row of the s-th entry in column order
 *   csc_perm [nnz]              canonical k of the s-th entry in column order
 *                               (so val[csc_perm] is Table 7's "CSC data")
 * Column order is (col, row) ascending.  Returns ORACLE_OK, ORACLE_ERR_RANGE
 * (*bad = first offending user index) or ORACLE_ERR_DUPLICATE (*bad = user
 * index of the later copy in canonical order).
 */
int oracle_canonicalize(int64_t out, int64_t in, int64_t nnz,
                        const int32_t *row, const int32_t *col, const float *val,
                        int32_t *c_row, int32_t *c_col, float *c_val, int64_t *c_src,
                        int32_t *row_ptr, int32_t *col_ptr, int32_t *csc_row,
                        int32_t *csc_perm, int64_t *bad) {
  int64_t k, r, c;
  key3 *keys;
  *bad = -1;
  if (out < 0 || in < 0 || nnz < 0) return ORACLE_ERR_ARG;
  for (k = 0; k < nnz; ++k) {
    if (row[k] < 0 || row[k] >= out || col[k] < 0 || col[k] >= in) {
      *bad = k;
      return ORACLE_ERR_RANGE;
    }
  }
  keys = (key3 *)malloc(sizeof(key3) * (size_t)(nnz > 0 ? nnz : 1));
  if (!keys) return ORACLE_ERR_ALLOC;
  for (k = 0; k < nnz; ++k) {
    keys[k].a = row[k];
    keys[k].b = col[k];
    keys[k].idx = k;
  }
  qsort(keys, (size_t)nnz, sizeof(key3), cmp_key3);
  for (k = 1; k < nnz; ++k) {
    if (keys[k].a == keys[k - 1].a && keys[k].b == keys[k - 1].b) {
      *bad = keys[k].idx;
      free(keys);
      return ORACLE_ERR_DUPLICATE;
    }
  }
  for (k = 0; k < nnz; ++k) {
    c_row[k] = (int32_t)keys[k].a;
    c_col[k] = (int32_t)keys[k].b;
    c_val[k] = val ? val[keys[k].idx] : 0.0f;
    c_src[k] = keys[k].idx;
  }
  /* CSR index pointer: count entries per row, then exclusive prefix sum. */
  for (r = 0; r <= out; ++r) row_ptr[r] = 0;
  for (k = 0; k < nnz; ++k) row_ptr[c_row[k] + 1] += 1;
  for (r = 0; r < out; ++r) row_ptr[r + 1] += row_ptr[r];
  /* CSC: order canonical entries by (col, row). */
  for (k = 0; k < nnz; ++k) {
    keys[k].a = c_col[k];
    keys[k].b = c_row[k];
    keys[k].idx = k;
  }
  qsort(keys, (size_t)nnz, sizeof(key3), cmp_key3);
  for (k = 0; k < nnz; ++k) {
    csc_row[k] = (int32_t)keys[k].b;
    csc_perm[k] = (int32_t)keys[k].idx;
  }
  for (c = 0; c <= in; ++c) col_ptr[c] = 0;
  for (k = 0; k < nnz; ++k) col_ptr[c_col[k] + 1] += 1;
  for (c = 0; c < in; ++c) col_ptr[c + 1] += col_ptr[c];
  free(keys);
  return ORACLE_OK;
}

/* ------------------------------------------------------------------------ */
/* Forward SpMM, §3.1 Algorithm 1                                           */
/* ------------------------------------------------------------------------ */

/*
 * Y = X W^T.  In the paper's notation C = A B with A = W and B = X^T, so
 * C[i][l] = Y[l][i].  Algorithm 1: start from C = 0; for each stored
 * nonzero (i, j, A_z) and each batch column l, C[i][l] += A_z * B[j][l].
 * Entries are visited in the order given (canonical order in practice).
 */
int oracle_forward(int64_t out, int64_t in, int64_t nnz, const int32_t *row,
                   const int32_t *col, const float *val, int64_t B, const float *X,
                   float *Y, double *S) {
  int64_t k, l, n = B * out;
  double *acc = (double *)calloc((size_t)(n > 0 ? n : 1), sizeof(double));
  double *sabs = (double *)calloc((size_t)(n > 0 ? n : 1), sizeof(double));
  if (!acc || !sabs) {
    free(acc);
    free(sabs);
    return ORACLE_ERR_ALLOC;
  }
  for (k = 0; k < nnz; ++k) {
    const int64_t i = row[k], j = col[k];
    const double a = (double)val[k];
    for (l = 0; l < B; ++l) {
      const double t = a * (double)X[l * in + j];
      acc[l * out + i] += t;
      sabs[l * out + i] += fabs(t);
    }
  }
  for (k = 0; k < n; ++k) {
    Y[k] = (float)acc[k];
    if (S) S[k] = sabs[k];
  }
  free(acc);
  free(sabs);
  return ORACLE_OK;
}

/* ------------------------------------------------------------------------ */
/* Backward, §3.4 and Appendix F ("Full gradient derivation")               */
/* ------------------------------------------------------------------------ */

/*
 * dX = dY W, i.e. the input gradient W^T (dL/dA) of §3.4.  Appendix F: W^T
 * keeps W's support, obtained by swapping the row and column index arrays,
 * so this is Algorithm 1 with the roles of row and col exchanged.
 */
int oracle_backward_input(int64_t out, int64_t in, int64_t nnz, const int32_t *row,
                          const int32_t *col, const float *val, int64_t B,
                          const float *dY, float *dX, double *S) {
  int64_t k, l, n = B * in;
  double *acc = (double *)calloc((size_t)(n > 0 ? n : 1), sizeof(double));
  double *sabs = (double *)calloc((size_t)(n > 0 ? n : 1), sizeof(double));
  if (!acc || !sabs) {
    free(acc);
    free(sabs);
    return ORACLE_ERR_ALLOC;
  }
  for (k = 0; k < nnz; ++k) {
    const int64_t i = row[k], j = col[k];
    const double a = (double)val[k];
    for (l = 0; l < B; ++l) {
      const double t = a * (double)dY[l * out + i];
      acc[l * in + j] += t;
      sabs[l * in + j] += fabs(t);
    }
  }
  for (k = 0; k < n; ++k) {
    dX[k] = (float)acc[k];
    if (S) S[k] = sabs[k];
  }
  free(acc);
  free(sabs);
  return ORACLE_OK;
}

/*
 * Sparse outer-product weight gradient (§3.4; Appendix F, mini-batch form):
 * (dL/dW)[i][j] = sum over batch t of dY[t][i] * X[t][j], evaluated only at
 * the stored (i, j).  One value per stored entry, aligned with (row, col).
 * The batch sum runs t = 0, 1, ..., B-1.
 */
int oracle_backward_weight(int64_t out, int64_t in, int64_t nnz, const int32_t *row,
                           const int32_t *col, int64_t B, const float *X,
                           const float *dY, float *dW, double *S) {
  int64_t k, t;
  for (k = 0; k < nnz; ++k) {
    const int64_t i = row[k], j = col[k];
    double acc = 0.0, sabs = 0.0;
    for (t = 0; t < B; ++t) {
      const double p = (double)dY[t * out + i] * (double)X[t * in + j];
      acc += p;
      sabs += fabs(p);
    }
    dW[k] = (float)acc;
    if (S) S[k] = sabs;
  }
  return ORACLE_OK;
}

/*
 * The same weight gradient left in double (no rounding to float), for the
 * optimizer routines below: g[k] = sum over t of dY[t][row_k] * X[t][col_k].
 */
int oracle_weight_gradient64(int64_t out, int64_t in, int64_t nnz, const int32_t *row,
                             const int32_t *col, int64_t B, const float *X, const float *dY,
                             double *g, double *S) {
  int64_t k, t;
  for (k = 0; k < nnz; ++k) {
    const int64_t i = row[k], j = col[k];
    double acc = 0.0, sabs = 0.0;
    for (t = 0; t < B; ++t) {
      const double p = (double)dY[t * out + i] * (double)X[t * in + j];
      acc += p;
      sabs += fabs(p);
    }
    g[k] = acc;
    if (S) S[k] = sabs;
  }
  return ORACLE_OK;
}

/* ------------------------------------------------------------------------ */
/* Optimizer steps on the stored entries only                               */
/* ------------------------------------------------------------------------ */

/*
 * §3.4: the weight gradient exists only at supp(W), so the optimizer acts on
 * the nnz stored values alone (frozen cells see no gradient and no update);
 * §4.1 trains with SGD, Appendix G ("Optimization") with Adam.  The pages
 * give neither update rule, so these are the textbook ones in the
 * conventions of PyTorch's torch.optim.SGD and torch.optim.Adam, with L2
 * weight decay added to the gradient.
 *
 * SGD, momentum mu >= 0 (no dampening, no Nesterov), one entry:
 *   d = g + wd * w;  if mu > 0: buf = mu * buf + d, d = buf;  w = w - lr * d.
 * With buf starting at 0 the first step gives buf = d, as PyTorch does.
 * buf_in / buf_out may be NULL when mu == 0.
 */
int oracle_sgd_update(int64_t n, const float *val, const double *g, const float *buf_in,
                      double lr, double mu, double wd, double *val_out, double *buf_out) {
  int64_t k;
  if (mu != 0.0 && (!buf_in || !buf_out)) return ORACLE_ERR_ARG;
  for (k = 0; k < n; ++k) {
    double d = g[k] + wd * (double)val[k];
    if (mu != 0.0) {
      d = mu * (double)buf_in[k] + d;
      buf_out[k] = d;
    }
    val_out[k] = (double)val[k] - lr * d;
  }
  return ORACLE_OK;
}

/*
 * Adam (Kingma and Ba, "Adam: A Method for Stochastic Optimization", ICLR
 * 2015) with bias correction, step t >= 1, one entry:
 *   d = g + wd * w
 *   m = b1 * m + (1 - b1) * d
 *   v = b2 * v + (1 - b2) * d^2
 *   w = w - (lr / (1 - b1^t)) * m / (sqrt(v) / sqrt(1 - b2^t) + eps)
 * (eps added after the bias-corrected square root, as in torch.optim.Adam).
 */
int oracle_adam_update(int64_t n, const float *val, const double *g, const float *m_in,
                       const float *v_in, double lr, double b1, double b2, double eps, double wd,
                       int64_t t, double *val_out, double *m_out, double *v_out) {
  int64_t k;
  if (t < 1) return ORACLE_ERR_ARG;
  const double bc1 = 1.0 - pow(b1, (double)t), bc2 = 1.0 - pow(b2, (double)t);
  for (k = 0; k < n; ++k) {
    const double d = g[k] + wd * (double)val[k];
    const double m = b1 * (double)m_in[k] + (1.0 - b1) * d;
    const double v = b2 * (double)v_in[k] + (1.0 - b2) * d * d;
    m_out[k] = m;
    v_out[k] = v;
    val_out[k] = (double)val[k] - (lr / bc1) * m / (sqrt(v) / sqrt(bc2) + eps);
  }
  return ORACLE_OK;
}

/* ------------------------------------------------------------------------ */
/* getrand(): a counter-based SplitMix64 stream                             */
/* ------------------------------------------------------------------------ */

/*
 * Algorithm 2 leaves getrand() unspecified.  The stream used here is
 * SplitMix64 (Steele, Lea and Flood, "Fast splittable pseudorandom number
 * generators", OOPSLA 2014): the state advances by the golden-ratio gamma
 * 0x9E3779B97F4A7C15 and each output is the state passed through the
 * variant-13 finaliser (shift 30, multiply 0xBF58476D1CE4E5B9, shift 27,
 * multiply 0x94D049BB133111EB, shift 31).  Draw t (t = 0, 1, ...) is the
 * (t+1)-th output of a generator whose state starts at `seed`, i.e. the
 * finaliser applied to seed + (t+1) * gamma, so any draw can be computed
 * on its own.
 */
uint64_t oracle_splitmix64(uint64_t seed, uint64_t t) {
  uint64_t z = seed + (t + 1u) * 0x9E3779B97F4A7C15ull;
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

/*
 * Map a 64-bit draw x to a cell index in [0, n): floor(x * n / 2^64), the
 * multiply-shift reduction of Lemire ("Fast random integer generation in an
 * interval", ACM TOMACS 2019), without the rejection step.
 */
uint64_t oracle_cell_index(uint64_t x, uint64_t n) {
  unsigned __int128 p = (unsigned __int128)x * (unsigned __int128)n;
  return (uint64_t)(p >> 64);
}

/* Open-addressing set of 64-bit cell indices (the hash set S of Alg. 2). */
typedef struct {
  uint64_t *slot; /* value + 1; 0 = empty */
  uint64_t mask;
} cellset;

static int cellset_init(cellset *s, int64_t expected) {
  uint64_t cap = 16;
  while (cap < (uint64_t)(2 * expected + 16)) cap <<= 1;
  s->slot = (uint64_t *)calloc((size_t)cap, sizeof(uint64_t));
  s->mask = cap - 1;
  return s->slot != NULL;
}

static uint64_t cellset_hash(uint64_t v) {
  v ^= v >> 33;
  v *= 0xFF51AFD7ED558CCDull;
  v ^= v >> 33;
  return v;
}

/* Returns 1 if v was added, 0 if it was already present. */
static int cellset_add(cellset *s, uint64_t v) {
  uint64_t h = cellset_hash(v) & s->mask;
  for (;;) {
    if (s->slot[h] == 0) {
      s->slot[h] = v + 1;
      return 1;
    }
    if (s->slot[h] == v + 1) return 0;
    h = (h + 1) & s->mask;
  }
}

/* ------------------------------------------------------------------------ */
/* Uniform connection initializer, §3.3 Algorithm 2                         */
/* ------------------------------------------------------------------------ */

/*
 * Draw `count` distinct (i, j) cells of an m x k = out x in matrix uniformly
 * at random by rejection against a hash set S (Algorithm 2).  Candidate t is
 * cell p = cell_index(splitmix64(seed, t), out*in) with i = p / in and
 * j = p % in (0-based; the paper's "+1" is its 1-based indexing).  A
 * candidate already in S is rejected; otherwise it is added to S and
 * appended to the output, in acceptance order.  *trials = candidates drawn.
 * count must not exceed out*in.
 */
int oracle_uniform_init(int64_t out, int64_t in, int64_t count, uint64_t seed,
                        int32_t *row, int32_t *col, int64_t *trials) {
  cellset s;
  const uint64_t n = (uint64_t)out * (uint64_t)in;
  uint64_t t = 0;
  int64_t got = 0;
  if (out <= 0 || in <= 0 || count < 0 || (uint64_t)count > n) return ORACLE_ERR_ARG;
  if (!cellset_init(&s, count)) return ORACLE_ERR_ALLOC;
  while (got < count) {
    const uint64_t p = oracle_cell_index(oracle_splitmix64(seed, t), n);
    ++t;
    if (cellset_add(&s, p)) {
      row[got] = (int32_t)(p / (uint64_t)in);
      col[got] = (int32_t)(p % (uint64_t)in);
      ++got;
    }
  }
  *trials = (int64_t)t;
  free(s.slot);
  return ORACLE_OK;
}

/* ------------------------------------------------------------------------ */
/* Magnitude prune + uniform regrow, Appendix G ("Sparsity schedule and     */
/* DST") with the regrow draw of Algorithm 2                                 */
/* ------------------------------------------------------------------------ */

typedef struct {
  uint32_t mag; /* bits of |val| */
  int64_t k;
} magkey;

static int cmp_magkey(const void *p, const void *q) {
  const magkey *x = (const magkey *)p, *y = (const magkey *)q;
  if (x->mag != y->mag) return x->mag < y->mag ? -1 : 1;
  if (x->k != y->k) return x->k < y->k ? -1 : 1;
  return 0;
}

/* Number pruned: floor(frac * nnz), computed in double. */
int64_t oracle_prune_count(float frac, int64_t nnz) {
  double p;
  if (!(frac > 0.0f)) return 0;
  if (frac >= 1.0f) return nnz;
  p = floor((double)frac * (double)nnz);
  return (int64_t)p;
}

/*
 * One prune-and-regrow step on a canonical layer.
 *  1. Prune: the P = floor(frac * nnz) entries with the smallest |val|.  The
 *     order is by the bit pattern of |val| read as an unsigned integer
 *     (so -0 equals +0 and NaN sorts above +inf), ties by canonical k.
 *  2. Regrow: P fresh cells drawn by Algorithm 2's rejection loop, where S
 *     starts as the surviving cells (just-pruned cells are eligible again).
 *     Regrown entries get value 0.
 *  3. The survivors (values kept) and the regrown cells are put back into
 *     canonical order (row, then column).
 * Outputs n_row, n_col, n_val [nnz]; *pruned = P; *trials = candidates drawn.
 */
int oracle_prune_regrow(int64_t out, int64_t in, int64_t nnz, const int32_t *row,
                        const int32_t *col, const float *val, float frac, uint64_t seed,
                        int32_t *n_row, int32_t *n_col, float *n_val, int64_t *pruned,
                        int64_t *trials) {
  const int64_t P = oracle_prune_count(frac, nnz);
  const uint64_t n = (uint64_t)out * (uint64_t)in;
  magkey *mk;
  unsigned char *gone;
  key3 *all;
  cellset s;
  int64_t k, m, got = 0;
  uint64_t t = 0;
  *pruned = P;
  *trials = 0;
  mk = (magkey *)malloc(sizeof(magkey) * (size_t)(nnz > 0 ? nnz : 1));
  gone = (unsigned char *)calloc((size_t)(nnz > 0 ? nnz : 1), 1);
  all = (key3 *)malloc(sizeof(key3) * (size_t)(nnz > 0 ? nnz : 1));
  if (!mk || !gone || !all || !cellset_init(&s, nnz)) {
    free(mk);
    free(gone);
    free(all);
    return ORACLE_ERR_ALLOC;
  }
  for (k = 0; k < nnz; ++k) {
    uint32_t bits;
    memcpy(&bits, &val[k], sizeof(bits));
    mk[k].mag = bits & 0x7FFFFFFFu;
    mk[k].k = k;
  }
  qsort(mk, (size_t)nnz, sizeof(magkey), cmp_magkey);
  for (k = 0; k < P; ++k) gone[mk[k].k] = 1;
  for (k = 0; k < nnz; ++k)
    if (!gone[k]) cellset_add(&s, (uint64_t)row[k] * (uint64_t)in + (uint64_t)col[k]);
  /* all[]: a = cell index, b = source (k for survivors, -1 for regrown). */
  m = 0;
  for (k = 0; k < nnz; ++k) {
    if (gone[k]) continue;
    all[m].a = (int64_t)((uint64_t)row[k] * (uint64_t)in + (uint64_t)col[k]);
    all[m].b = k;
    all[m].idx = m;
    ++m;
  }
  while (got < P) {
    const uint64_t p = oracle_cell_index(oracle_splitmix64(seed, t), n);
    ++t;
    if (cellset_add(&s, p)) {
      all[m].a = (int64_t)p;
      all[m].b = -1;
      all[m].idx = m;
      ++m;
      ++got;
    }
  }
  *trials = (int64_t)t;
  qsort(all, (size_t)m, sizeof(key3), cmp_key3);
  for (k = 0; k < m; ++k) {
    n_row[k] = (int32_t)((uint64_t)all[k].a / (uint64_t)in);
    n_col[k] = (int32_t)((uint64_t)all[k].a % (uint64_t)in);
    n_val[k] = all[k].b >= 0 ? val[all[k].b] : 0.0f;
  }
  free(mk);
  free(gone);
  free(all);
  free(s.slot);
  return ORACLE_OK;
}
