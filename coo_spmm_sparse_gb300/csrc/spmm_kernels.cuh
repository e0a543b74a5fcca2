// Segmented SpMM / SDDMM kernels of the SNACK layer for sm_103a (CUDA cores).
//
// The paper's SNACK-COO kernel ("Beyond Masked Sparsity", §3.2 and Appendix F
// "Parallel-efficiency analysis") runs a (nnz-chunk x batch-column) grid with
// one global atomicAdd per (entry, batch column), re-reading the whole COO
// triple once per batch column.  Here the index/value stream is read ONCE per
// call whatever the batch:
//
//  * Entries are ordered by line (row for Y = X W^T and dW, column for
//    dX = dY W) and each line is cut into segments.  A TEAM of LPS lanes
//    owns one segment; inside a team, GROUPS of G lanes each take one entry
//    at a time, and the G lanes of a group split the batch slice (BW floats,
//    16-byte vectors).  Each group walks quads of 4 consecutive entries, each
//    from one 16-byte load of indices and one of values (aligned down to a
//    multiple of 4 and masked at the segment ends), two quads per step.
//    Gathering from global memory in canonical order (forward, dW), the
//    loads of the next step are issued before the gathers of this one.
//  * The dense operand is gathered from a transposed copy (line-major,
//    [lines][BW]) so that the BW batch values of one column are contiguous.
//    A group reads an entry's whole row (up to one 128-byte line) with ONE
//    instruction: the L1 data pipe spends a wavefront per (instruction,
//    line), so splitting a row across instructions multiplies its cost.
//  * Partial sums of the groups are combined with warp shuffles; only lines
//    split into several segments (long rows / columns) meet across warps,
//    and they do it deterministically: each segment stores its partial, the
//    last one to arrive (atomic ticket) adds them in segment order and
//    writes the output, then re-arms the ticket.  No floating-point atomics.
//  * Index and value streams bypass L1 (ld.global.nc.L1::no_allocate) so
//    that L1 keeps the gathered dense rows.
//  * Grids are persistent (resident blocks only) with a warp-uniform segment
//    loop.  A kernel may be launched as a programmatic dependent of the
//    transpose that feeds it: it waits (griddepcontrol.wait) before reading
//    anything, so only its launch and block start-up overlap the producer.
#pragma once

#include "snack_internal.cuh"

namespace snack {

__device__ __forceinline__ int4 ld_stream_i4(const int32_t *p) {
  int4 r;
  asm("ld.global.nc.L1::no_allocate.v4.s32 {%0, %1, %2, %3}, [%4];"
      : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
      : "l"(p));
  return r;
}

__device__ __forceinline__ float4 ld_stream_f4(const float *p) {
  float4 r;
  asm("ld.global.nc.L1::no_allocate.v4.f32 {%0, %1, %2, %3}, [%4];"
      : "=f"(r.x), "=f"(r.y), "=f"(r.z), "=f"(r.w)
      : "l"(p));
  return r;
}

// Bulk prefetch of [p, p + bytes) into L2 (16-byte aligned, multiple of 16).
__device__ __forceinline__ void l2_prefetch(const void *p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

// Each team's first lane asks L2 for the index (and value or permutation)
// ranges of every segment the team will process, so that the walk over them
// hits L2 instead of paying a DRAM round trip per step.  Segment ranges are
// rounded out to 16 bytes (the streams are padded).
__device__ __forceinline__ void prefetch_segments(const int4 *seg, int64_t nseg, const int32_t *a,
                                                  const void *b, int lps, int64_t block,
                                                  int64_t nblocks) {
  const int64_t teams_per_block = blockDim.x / lps;
  if ((threadIdx.x & (lps - 1)) != 0) return;
  for (int64_t t = block * teams_per_block + threadIdx.x / lps; t < nseg;
       t += nblocks * teams_per_block) {
    const int4 sg = seg[t];
    const int k0 = sg.y & ~3, k1 = (sg.z + 3) & ~3;
    if (k1 <= k0) continue;
    l2_prefetch(a + k0, (uint32_t)(k1 - k0) * 4);
    if (b) l2_prefetch(static_cast<const int32_t *>(b) + k0, (uint32_t)(k1 - k0) * 4);
  }
}

// Ask L2 for this block's share of a whole array (the values reached through
// the column permutation are read at random).
__device__ __forceinline__ void prefetch_share(const float *p, int64_t n, int64_t block,
                                               int64_t nblocks) {
  if (threadIdx.x != 0 || n <= 0) return;
  const int64_t per = (((n + nblocks - 1) / nblocks) + 3) & ~int64_t(3);
  const int64_t b0 = block * per;
  if (b0 >= n) return;
  const int64_t len = (b0 + per < n ? per : ((n - b0 + 3) & ~int64_t(3)));
  for (int64_t off = 0; off < len; off += 8192)
    l2_prefetch(p + b0 + off, (uint32_t)((len - off < 8192 ? len - off : 8192) * 4));
}

// Programmatic dependent launch: wait for the preceding grid (no-op when the
// kernel was launched without the attribute) / let the next grid launch.
// Every kernel here is launched as a programmatic dependent and waits before
// it reads or writes anything a preceding kernel may touch (operands,
// outputs, values, workspace), so only its launch, block start-up and the L2
// prefetch of the handle's immutable index streams run ahead.  Transposes
// trigger their dependents on entry; the segment kernels let theirs launch
// when they finish (triggering on entry measured slower in a replayed step:
// the early dependents hold block slots the running kernel could use).
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_launch() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Lanes per entry for a slice width: one 16-byte vector per lane and the
// whole row (up to 128 B) in one instruction; BW = 64 uses 8 lanes x 2, the
// wide slices (128, 256) a half or whole warp x 2.
__host__ __device__ constexpr int lanes_for(int bw) {
  return bw <= 4 ? 1 : (bw >= 128 ? bw / 8 : (bw >= 32 ? 8 : bw / 4));
}

// Shape of a batch slice: each lane holds NV vectors of VEC floats.
template <int BW>
struct SliceShape {
  static constexpr int G = lanes_for(BW);
  static constexpr int VEC = BW >= 4 ? 4 : BW;
  static constexpr int NV = BW >= 4 ? BW / (4 * G) : 1;
  static_assert(BW < 4 ? G == 1 : (BW % (4 * G) == 0), "bad slice shape");
};

template <int VEC>
__device__ __forceinline__ void load_vec(const float *p, float (&x)[VEC]);

template <>
__device__ __forceinline__ void load_vec<4>(const float *p, float (&x)[4]) {
  const float4 f = __ldg(reinterpret_cast<const float4 *>(p));
  x[0] = f.x;
  x[1] = f.y;
  x[2] = f.z;
  x[3] = f.w;
}

template <>
__device__ __forceinline__ void load_vec<2>(const float *p, float (&x)[2]) {
  const float2 f = __ldg(reinterpret_cast<const float2 *>(p));
  x[0] = f.x;
  x[1] = f.y;
}

template <>
__device__ __forceinline__ void load_vec<1>(const float *p, float (&x)[1]) {
  x[0] = __ldg(p);
}

// Operand row slice: from global memory through the read-only path, or (SM)
// from a copy in this block's shared memory.
template <int VEC, bool SM>
__device__ __forceinline__ void load_op(const float *p, float (&x)[VEC]) {
  if constexpr (SM) {
    if constexpr (VEC == 4) {
      const float4 f = *reinterpret_cast<const float4 *>(p);
      x[0] = f.x;
      x[1] = f.y;
      x[2] = f.z;
      x[3] = f.w;
    } else if constexpr (VEC == 2) {
      const float2 f = *reinterpret_cast<const float2 *>(p);
      x[0] = f.x;
      x[1] = f.y;
    } else {
      x[0] = *p;
    }
  } else {
    load_vec<VEC>(p, x);
  }
}

// Lane (group 0, sub) holds batch b = v*G*VEC + sub*VEC + i.
template <int BW>
__device__ __forceinline__ void store_line(float *dst, int64_t ld, int nb, int line, int sub,
                                           const float (&r)[SliceShape<BW>::NV]
                                                           [SliceShape<BW>::VEC]) {
  using S = SliceShape<BW>;
#pragma unroll
  for (int v = 0; v < S::NV; ++v)
#pragma unroll
    for (int i = 0; i < S::VEC; ++i) {
      const int b = v * S::G * S::VEC + sub * S::VEC + i;
      if (b < nb) dst[(int64_t)b * ld + line] = r[v][i];
    }
}

// Entries [kb, kb+4) of one group: indices / values from one 16-byte load
// each; values of a column-order stream come through the permutation.
template <bool PERM>
__device__ __forceinline__ void load_quad(const SpmmArgs &a, int kb, int k0, int k1, int (&c)[4],
                                          float (&w)[4]) {
  const int4 c4 = ld_stream_i4(a.idx + kb);
  c[0] = c4.x;
  c[1] = c4.y;
  c[2] = c4.z;
  c[3] = c4.w;
  if constexpr (PERM) {
    const int4 p4 = ld_stream_i4(a.perm + kb);
    const int pp[4] = {p4.x, p4.y, p4.z, p4.w};
#pragma unroll
    for (int e = 0; e < 4; ++e)
      w[e] = (kb + e >= k0 && kb + e < k1) ? __ldg(a.val + pp[e]) : 0.f;
  } else {
    const float4 v4 = ld_stream_f4(a.val + kb);
    w[0] = v4.x;
    w[1] = v4.y;
    w[2] = v4.z;
    w[3] = v4.w;
  }
}

// Gather the lane's slice of the dense rows of Q quads (all loads issued
// before any use), then accumulate.  Operand row c starts at src + c * ld.
template <int BW, int Q, bool SM = false>
__device__ __forceinline__ void gather_fma(const float *src, int ld, const int (&c)[Q][4],
                                           const float (&w)[Q][4], const bool (&ok)[Q][4],
                                           float (&acc)[SliceShape<BW>::NV][SliceShape<BW>::VEC]) {
  using S = SliceShape<BW>;
  constexpr int VEC = S::VEC, NV = S::NV, G = S::G;
  float x[Q][4][NV][VEC];
#pragma unroll
  for (int q = 0; q < Q; ++q)
#pragma unroll
    for (int e = 0; e < 4; ++e)
#pragma unroll
      for (int v = 0; v < NV; ++v) {
        if (ok[q][e]) {
          load_op<VEC, SM>(src + (int64_t)c[q][e] * ld + v * G * VEC, x[q][e][v]);
        } else {
#pragma unroll
          for (int i = 0; i < VEC; ++i) x[q][e][v][i] = 0.f;
        }
      }
#pragma unroll
  for (int q = 0; q < Q; ++q)
#pragma unroll
    for (int e = 0; e < 4; ++e)
#pragma unroll
      for (int v = 0; v < NV; ++v)
#pragma unroll
        for (int i = 0; i < VEC; ++i)
          // masked entries (a neighbouring line's) add exactly nothing, even
          // when their value is infinite or NaN
          acc[v][i] = fmaf(ok[q][e] ? w[q][e] : 0.f, x[q][e][v][i], acc[v][i]);
}

// The same for an operand whose rows are BW floats apart.
template <int BW, int Q, bool SM = false>
__device__ __forceinline__ void gather_fma(const float *src, const int (&c)[Q][4],
                                           const float (&w)[Q][4], const bool (&ok)[Q][4],
                                           float (&acc)[SliceShape<BW>::NV][SliceShape<BW>::VEC]) {
  gather_fma<BW, Q, SM>(src, BW, c, w, ok, acc);
}

// Index and value quads of one step (at kb and kb + 4 * npt, each only if
// it starts inside the segment), canonical-order streams only.
__device__ __forceinline__ void load_step(const SpmmArgs &a, int kb, int k1, int npt,
                                          int (&c)[2][4], float (&w)[2][4]) {
#pragma unroll
  for (int q = 0; q < 2; ++q) {
    const int kq = kb + q * 4 * npt;
    if (kq >= k1) continue;
    const int4 c4 = ld_stream_i4(a.idx + kq);
    const float4 v4 = ld_stream_f4(a.val + kq);
    c[q][0] = c4.x;
    c[q][1] = c4.y;
    c[q][2] = c4.z;
    c[q][3] = c4.w;
    w[q][0] = v4.x;
    w[q][1] = v4.y;
    w[q][2] = v4.z;
    w[q][3] = v4.w;
  }
}

// The entries of one group in steps of two quads, gathering the operand
// from global (SM = false) or shared memory, for canonical-order streams
// (rows).  The stream loads run one step ahead: while this step's operand
// rows are gathered, the next step's indices and values are in flight.  A quad past the segment end is
// not loaded and all its entries are masked.  (The column direction reads
// its values through the permutation, a load that depends on another; run
// ahead the same way it measured slower at 64-wide slices, so it keeps the
// plain loop.)
template <int BW, bool SM>
__device__ __forceinline__ void walk_pipelined(const SpmmArgs &a, const float *src, int ld, int kb,
                                               int k0, int k1, int npt,
                                               float (&acc)[SliceShape<BW>::NV]
                                                           [SliceShape<BW>::VEC]) {
  int c[2][4] = {};
  float w[2][4] = {};
  load_step(a, kb, k1, npt, c, w);
  for (; kb < k1; kb += 8 * npt) {
    bool ok[2][4];
#pragma unroll
    for (int q = 0; q < 2; ++q)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int k = kb + q * 4 * npt + e;
        ok[q][e] = k >= k0 && k < k1;
      }
    int cn[2][4] = {};
    float wn[2][4] = {};
    load_step(a, kb + 8 * npt, k1, npt, cn, wn);
    gather_fma<BW, 2, SM>(src, ld, c, w, ok, acc);
#pragma unroll
    for (int q = 0; q < 2; ++q)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        c[q][e] = cn[q][e];
        w[q][e] = wn[q][e];
      }
  }
}

// Segmented SpMM over blocks [block, ...) of a persistent grid of `nblocks`.
// PERM = values reached through a column-order -> canonical permutation
// (the dX = dY W direction while the column-ordered value copy is stale).
// PIPE = without a permutation, run the stream one step ahead
// (walk_pipelined).  SM = the operand is in shared memory.
template <int BW, int LPS, bool PERM, bool SM = false, bool PIPE = true>
__device__ __forceinline__ void spmm_part(const SpmmArgs &a, const float *op, int64_t block,
                                          int64_t nblocks) {
  using S = SliceShape<BW>;
  constexpr int VEC = S::VEC, NV = S::NV, G = S::G;
  constexpr int lps = LPS;  // lanes per team: power of two in [G, 32]
  constexpr int npt = lps / G;
  static_assert(LPS % G == 0 && LPS <= 32, "bad team");
  const int lane = threadIdx.x & 31;
  const int tlane = lane & (lps - 1);
  const int grp = tlane / G;
  const int sub = tlane % G;
  const int64_t teams_per_block = blockDim.x / lps;
  const int64_t stride = nblocks * teams_per_block;
  const int64_t my_team = block * teams_per_block + threadIdx.x / lps;
  const int64_t warp_team = block * teams_per_block + (threadIdx.x & ~31) / lps;
  // Batch sub-slice of this block (blockIdx.y, 0 unless the launch cuts the
  // slice into sub-slices; tables with split lines never are): columns
  // part_b * BW .. of an operand whose rows are a.stride floats apart.
  const int part_b = blockIdx.y;
  const int ld = SM ? BW : a.stride;
  const float *src = op + part_b * BW + sub * VEC;
  float *const dst = a.dst + (int64_t)part_b * BW * a.ld;
  const int nb = a.nb - part_b * BW;

  // Staged output (slices of 128+, one team per warp, no split lines): a
  // line's outputs are a column of the row-major output, BW scattered
  // 4-byte stores.  Instead the block's 8 warps, which hold 8 consecutive
  // lines in every round, park their results in shared memory (double
  // buffered, rows padded by 4 so the reads below are conflict-free) and the
  // block writes each output row's 8 consecutive lines as one 32-byte run.
  // The round count is then the block's, so every warp meets the barrier.
  // (At 64-wide slices the stores are too small a part of the work to pay
  // for the barrier: 10000x10000 @95% forward 93.6 -> 95.0 us.)
  constexpr bool kCanStage = BW >= 128 && LPS == 32 && !SM;
  constexpr int kStW = kCanStage ? BW + 4 : 1;
  __shared__ __align__(16) float stage_buf[kCanStage ? 2 : 1][kCanStage ? 8 : 1][kStW];
  const bool staged = kCanStage && a.stage;
  const int64_t block_team0 = block * teams_per_block;

  int64_t round = 0;
  for (int64_t t0 = 0; (staged ? block_team0 : warp_team) + t0 < a.nseg; t0 += stride, ++round) {
    const int64_t team = my_team + t0;
    const bool active = team < a.nseg;
    int4 sg = make_int4(0, 0, 0, -1);
    if (active) sg = a.seg[team];
    const int k0 = sg.y, k1 = sg.z;

    float acc[NV][VEC];
#pragma unroll
    for (int v = 0; v < NV; ++v)
#pragma unroll
      for (int i = 0; i < VEC; ++i) acc[v][i] = 0.f;

    int kb = (k0 & ~3) + 4 * grp;
    if constexpr (!PERM && PIPE) {
      walk_pipelined<BW, SM>(a, src, ld, kb, k0, k1, npt, acc);
    } else {
      for (; kb + 4 * npt < k1; kb += 8 * npt) {  // two quads in flight
        int c[2][4];
        float w[2][4];
        bool ok[2][4];
        load_quad<PERM>(a, kb, k0, k1, c[0], w[0]);
        load_quad<PERM>(a, kb + 4 * npt, k0, k1, c[1], w[1]);
#pragma unroll
        for (int q = 0; q < 2; ++q)
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int k = kb + q * 4 * npt + e;
            ok[q][e] = k >= k0 && k < k1;
          }
        gather_fma<BW, 2, SM>(src, ld, c, w, ok, acc);
      }
      if (kb < k1) {
        int c[1][4];
        float w[1][4];
        bool ok[1][4];
        load_quad<PERM>(a, kb, k0, k1, c[0], w[0]);
#pragma unroll
        for (int e = 0; e < 4; ++e) ok[0][e] = kb + e >= k0 && kb + e < k1;
        gather_fma<BW, 1, SM>(src, ld, c, w, ok, acc);
      }
    }

    // Combine the npt groups of the team (every lane of the warp is here).
#pragma unroll
    for (int off = G; off < lps; off <<= 1)
#pragma unroll
      for (int v = 0; v < NV; ++v)
#pragma unroll
        for (int i = 0; i < VEC; ++i) acc[v][i] += __shfl_xor_sync(0xffffffffu, acc[v][i], off);

    if constexpr (kCanStage) {
      if (staged) {
        float(*st)[kStW] = stage_buf[round & 1];
        const int w = threadIdx.x >> 5;
        if (grp == 0) {
#pragma unroll
          for (int v = 0; v < NV; ++v)
            *reinterpret_cast<float4 *>(&st[w][v * G * VEC + sub * VEC]) =
                make_float4(acc[v][0], acc[v][1], acc[v][2], acc[v][3]);
        }
        __syncthreads();
        const int64_t line0 = block_team0 + t0;  // segment s is line s
        for (int f = threadIdx.x; f < 8 * BW; f += blockDim.x) {
          const int b = f >> 3, j = f & 7;
          if (b < nb && line0 + j < a.nseg) dst[(int64_t)b * a.ld + line0 + j] = st[j][b];
        }
        continue;
      }
    }
    if (!active) continue;
    const int line = sg.x;
    if (sg.w < 0) {
      if (grp == 0) store_line<BW>(dst, a.ld, nb, line, sub, acc);
      continue;
    }

    // Line split over several segments: park the partial, last arrival sums.
    const int4 sp = a.split[sg.w];  // {first segment, parts, first slot, 0}
    const int part = (int)(team - sp.x);
    if (grp == 0) {
      float *mine = a.partial + (int64_t)(sp.z + part) * BW + sub * VEC;
#pragma unroll
      for (int v = 0; v < NV; ++v)
#pragma unroll
        for (int i = 0; i < VEC; ++i) mine[v * G * VEC + i] = acc[v][i];
    }
    if (a.counter == nullptr) continue;  // the parts are summed by split_sums
    __threadfence();
    const unsigned tmask = lps == 32 ? 0xffffffffu : (((1u << lps) - 1u) << (lane - tlane));
    __syncwarp(tmask);
    int last = 0;
    if (tlane == 0) last = atomicAdd(a.counter + sg.w, 1) == sp.y - 1;
    last = __shfl_sync(tmask, last, lane - tlane);
    if (!last) continue;
    __threadfence();
    // The team's npt groups each sum the parts grp, grp + npt, ... in order,
    // then meet by shuffle: a fixed order for a given plan (reproducible),
    // with up to npt parts' loads in flight at once.  The SpMM kernels of
    // slices of 1-4 floats (where the tickets stay in use) load four of a
    // group's parts at once: past the last part a group loads the last again
    // and leaves it out of the sum.  (Wider kernels and the fused backward
    // keep one part per load: the four would cost their main loop
    // registers.)
    float tot[NV][VEC];
#pragma unroll
    for (int v = 0; v < NV; ++v)
#pragma unroll
      for (int i = 0; i < VEC; ++i) tot[v][i] = 0.f;
    if constexpr (BW <= 4 && PIPE) {
#pragma unroll 1
      for (int p = grp; p < sp.y; p += 4 * npt) {
        float x[4][VEC];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const float *q =
              a.partial + (int64_t)(sp.z + min(p + u * npt, sp.y - 1)) * BW + sub * VEC;
#pragma unroll
          for (int i = 0; i < VEC; ++i) x[u][i] = __ldcg(q + i);
        }
#pragma unroll
        for (int u = 0; u < 4; ++u)
          if (p + u * npt < sp.y) {
#pragma unroll
            for (int i = 0; i < VEC; ++i) tot[0][i] += x[u][i];
          }
      }
    } else {
#pragma unroll 1
      for (int p = grp; p < sp.y; p += npt) {
        const float *q = a.partial + (int64_t)(sp.z + p) * BW + sub * VEC;
#pragma unroll
        for (int v = 0; v < NV; ++v)
#pragma unroll
          for (int i = 0; i < VEC; ++i) tot[v][i] += __ldcg(q + v * G * VEC + i);
      }
    }
#pragma unroll
    for (int off = G; off < lps; off <<= 1)
#pragma unroll
      for (int v = 0; v < NV; ++v)
#pragma unroll
        for (int i = 0; i < VEC; ++i) tot[v][i] += __shfl_xor_sync(tmask, tot[v][i], off);
    if (grp == 0) store_line<BW>(dst, a.ld, nb, line, sub, tot);
    if (tlane == 0) a.counter[sg.w] = 0;  // re-arm for the next call
  }
}

// Four consecutive floats at p (16-byte aligned): one vector access when the
// whole quad is in use, else only the entries whose bit is set in `mask`.
__device__ __forceinline__ void load4(const float *p, unsigned mask, float (&x)[4]) {
  if (mask == 15u) {
    const float4 f = *reinterpret_cast<const float4 *>(p);
    x[0] = f.x;
    x[1] = f.y;
    x[2] = f.z;
    x[3] = f.w;
  } else {
#pragma unroll
    for (int e = 0; e < 4; ++e) x[e] = (mask >> e) & 1u ? p[e] : 0.f;
  }
}

__device__ __forceinline__ void store4(float *p, unsigned mask, const float (&x)[4]) {
  if (mask == 15u) {
    *reinterpret_cast<float4 *>(p) = make_float4(x[0], x[1], x[2], x[3]);
  } else {
#pragma unroll
    for (int e = 0; e < 4; ++e)
      if ((mask >> e) & 1u) p[e] = x[e];
  }
}

// Operands of the optimizer step for one quad (entries whose bit is set in
// mask): values and state.  Loaded before the quad's gathers so that their
// latency overlaps them.
struct OptQuad {
  unsigned mask;
  float w[4], s0[4], s1[4];
};

__device__ __forceinline__ unsigned quad_mask(int kq, int k0, int k1) {
  unsigned mask = 0;
#pragma unroll
  for (int e = 0; e < 4; ++e)
    if (kq + e >= k0 && kq + e < k1) mask |= 1u << e;
  return mask;
}

__device__ __forceinline__ void opt_load(const OptArgs &o, int kq, unsigned mask, OptQuad &q) {
  q.mask = mask;
  load4(o.val + kq, mask, q.w);
  if (o.s0) load4(o.s0 + kq, mask, q.s0);
  if (o.s1) load4(o.s1 + kq, mask, q.s1);
}

// Optimizer step for one quad given its batch gradients res.  SGD: d = g + wd w, buf = mom buf + d (with a
// buffer), w -= lr d.  Adam: m = b1 m + (1-b1) d, v = b2 v + (1-b2) d^2,
// w -= step m / (sqrt(v) / sqrt(1 - b2^t) + eps).
__device__ __forceinline__ void opt_store(const OptArgs &o, int kq, OptQuad &q,
                                          const float (&res)[4]) {
  float d[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) d[e] = fmaf(o.wd, q.w[e], res[e]);
  if (o.kind == kOptSgd) {
    if (o.s0) {
#pragma unroll
      for (int e = 0; e < 4; ++e) d[e] = q.s0[e] = fmaf(o.mom, q.s0[e], d[e]);
      store4(o.s0 + kq, q.mask, q.s0);
    }
#pragma unroll
    for (int e = 0; e < 4; ++e) q.w[e] = fmaf(-o.lr, d[e], q.w[e]);
  } else {
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      q.s0[e] = fmaf(o.b1, q.s0[e], o.c1 * d[e]);
      q.s1[e] = fmaf(o.b2, q.s1[e], o.c2 * d[e] * d[e]);
      q.w[e] = q.w[e] - o.step * q.s0[e] / (sqrtf(q.s1[e]) / o.sbc2 + o.eps);
    }
    store4(o.s0 + kq, q.mask, q.s0);
    store4(o.s1 + kq, q.mask, q.s1);
  }
  store4(o.val + kq, q.mask, q.w);
}

// Column quads at kb (and kb + 4 * npt when QPS = 2), each only if it
// starts before k1.
template <int QPS>
__device__ __forceinline__ void load_col_step(const int32_t *col, int kb, int k1, int npt,
                                              int (&c)[2][4]) {
#pragma unroll
  for (int q = 0; q < QPS; ++q) {
    const int kq = kb + q * 4 * npt;
    if (kq >= k1) continue;
    const int4 c4 = ld_stream_i4(col + kq);
    c[q][0] = c4.x;
    c[q][1] = c4.y;
    c[q][2] = c4.z;
    c[q][3] = c4.w;
  }
}

// dW of one quad when its four dot products are spread over a group of G
// >= 2 lanes (d[e]: this lane's part of entry e): a butterfly over the
// group sums them and leaves one entry per lane at once.  The first level
// keeps entries 2-3 on the upper half of the group and 0-1 on the lower
// (two shuffles), the second one entry per lane (one shuffle), the rest
// finish that entry's sum; 2 / 3 / 4 / 5 / 6 shuffles per quad at G = 2 /
// 4 / 8 / 16 / 32, against log2(G) per entry when each entry is summed on
// its own (the shuffles go through the L1 data pipe the gathers need: at
// 64-wide slices they were 0.86 of its 3.6 wavefronts per entry).  With G
// = 2 each lane ends with two entries.
template <int G>
__device__ __forceinline__ void sddmm_store_spread(const SddmmArgs &a, int kq, int k0, int k1,
                                                   int sub, unsigned gmask, float (&d)[4]) {
  const bool up = (sub & (G / 2)) != 0;
  const float s0 = __shfl_xor_sync(gmask, up ? d[0] : d[2], G / 2);
  const float s1 = __shfl_xor_sync(gmask, up ? d[1] : d[3], G / 2);
  d[0] = (up ? d[2] : d[0]) + s0;
  d[1] = (up ? d[3] : d[1]) + s1;
  const int base = kq + (up ? 2 : 0);
  if constexpr (G == 2) {
#pragma unroll
    for (int e = 0; e < 2; ++e)
      if (base + e >= k0 && base + e < k1) {
        float *p = a.dw + base + e;
        *p = a.accumulate ? *p + d[e] : d[e];
      }
  } else {
    const bool up2 = (sub & (G / 4)) != 0;
    float r = (up2 ? d[1] : d[0]) + __shfl_xor_sync(gmask, up2 ? d[0] : d[1], G / 4);
#pragma unroll
    for (int off = G / 8; off >= 1; off >>= 1) r += __shfl_xor_sync(gmask, r, off);
    const int k = base + (up2 ? 1 : 0);
    if ((sub & (G / 4 - 1)) == 0 && k >= k0 && k < k1) {
      float *p = a.dw + k;
      *p = a.accumulate ? *p + r : r;
    }
  }
}

// dW for up to two quads of one group (columns already loaded): the G lanes
// of a group each form part of the batch dot product.  SPREAD: the quad's
// four sums meet in sddmm_store_spread; else each entry is summed over the
// group by shuffles and one lane stores the quad (the fused backward at
// slices of 64+ floats, where the butterfly measured slower) or applies the
// optimizer step (OPT, whose update reads all four sums in one lane).
template <int BW, bool SM, bool OPT, bool SPREAD>
__device__ __forceinline__ void sddmm_quads(const SddmmArgs &a, const float *xt, int kb, int k0,
                                            int k1, int npt, unsigned gmask, int sub,
                                            const float (&dy)[SliceShape<BW>::NV]
                                                             [SliceShape<BW>::VEC],
                                            const int (&c)[2][4], bool two) {
  using S = SliceShape<BW>;
  constexpr int VEC = S::VEC, NV = S::NV, G = S::G;
  OptQuad oq[OPT ? 2 : 1];
  if constexpr (OPT) {
    if (sub == 0) {
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        const int kq = kb + q * 4 * npt;
        opt_load(a.opt, kq, (q == 0 || two) ? quad_mask(kq, k0, k1) : 0u, oq[q]);
      }
    }
  }
  float x[2][4][NV][VEC];
#pragma unroll
  for (int q = 0; q < 2; ++q)
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int k = kb + q * 4 * npt + e;
      const bool ok = (q == 0 || two) && k >= k0 && k < k1;
#pragma unroll
      for (int v = 0; v < NV; ++v) {
        if (ok) {
          load_op<VEC, SM>(xt + (int64_t)c[q][e] * BW + v * G * VEC, x[q][e][v]);
        } else {
#pragma unroll
          for (int i = 0; i < VEC; ++i) x[q][e][v][i] = 0.f;
        }
      }
    }
#pragma unroll
  for (int q = 0; q < 2; ++q) {
    if (q == 1 && !two) break;
    const int kq = kb + q * 4 * npt;
    float res[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      float s = 0.f;
#pragma unroll
      for (int v = 0; v < NV; ++v)
#pragma unroll
        for (int i = 0; i < VEC; ++i) s = fmaf(dy[v][i], x[q][e][v][i], s);
      if constexpr (OPT || !SPREAD) {
#pragma unroll
        for (int off = 1; off < G; off <<= 1) s += __shfl_xor_sync(gmask, s, off);
      }
      res[e] = s;
    }
    if constexpr (SPREAD && !OPT && G >= 2) {
      sddmm_store_spread<G>(a, kq, k0, k1, sub, gmask, res);
      continue;
    }
    if (sub == 0) {
      if constexpr (OPT) {
        opt_store(a.opt, kq, oq[q], res);
        continue;
      }
      float *d = a.dw + kq;
      if (kq >= k0 && kq + 3 < k1) {
        float4 o = make_float4(res[0], res[1], res[2], res[3]);
        if (a.accumulate) {
          const float4 old = *reinterpret_cast<const float4 *>(d);
          o.x += old.x;
          o.y += old.y;
          o.z += old.z;
          o.w += old.w;
        }
        *reinterpret_cast<float4 *>(d) = o;
      } else {
#pragma unroll
        for (int e = 0; e < 4; ++e)
          if (kq + e >= k0 && kq + e < k1) d[e] = a.accumulate ? d[e] + res[e] : res[e];
      }
    }
  }
}

// dW[k] = sum_b dY[b][row_k] X[b][col_k] over the row segments (persistent
// grid of `nblocks`; a team's lanes stay together, groups never diverge).
// OPT: apply the optimizer step of a.opt instead of writing dW (compiled
// separately, so the plain kernels keep their registers).
template <int BW, int LPS, bool SM = false, bool OPT = false, bool FUSED = false>
__device__ __forceinline__ void sddmm_part(const SddmmArgs &a, const float *op, int64_t block,
                                           int64_t nblocks) {
  using S = SliceShape<BW>;
  constexpr int VEC = S::VEC, NV = S::NV, G = S::G;
  constexpr int lps = LPS;
  constexpr int npt = lps / G;
  static_assert(LPS % G == 0 && LPS <= 32, "bad team");
  const int lane = threadIdx.x & 31;
  const int tlane = lane & (lps - 1);
  const int grp = tlane / G;
  const int sub = tlane % G;
  const unsigned gmask = G == 32 ? 0xffffffffu
                                 : (G == 1 ? (1u << lane) : (((1u << G) - 1u) << (lane & ~(G - 1))));
  const int64_t teams_per_block = blockDim.x / lps;
  const int64_t stride = nblocks * teams_per_block;
  const float *xt = op + sub * VEC;
  // Entry sub-ranges (nsub > 1): team t takes part t / nseg of segment
  // t % nseg (the entries are independent, nothing to combine).
  const int64_t nteams = a.nseg * a.nsub;
  for (int64_t team = block * teams_per_block + threadIdx.x / lps; team < nteams; team += stride) {
    const int part = a.nsub > 1 ? (int)(team / a.nseg) : 0;
    const int4 sg = a.seg[team - (int64_t)part * a.nseg];
    const int r = sg.x;
    int k0 = sg.y, k1 = sg.z;
    if (a.nsub > 1) {
      const int64_t len = k1 - k0;
      k1 = sg.y + (int)((part + 1) * len / a.nsub);
      k0 = sg.y + (int)(part * len / a.nsub);
    }
    float dy[NV][VEC];
    {
      const float *p = a.dyt + (int64_t)r * BW + sub * VEC;
#pragma unroll
      for (int v = 0; v < NV; ++v) load_vec<VEC>(p + v * G * VEC, dy[v]);
    }
    // The column loads run one step ahead of the gathers (as in
    // walk_pipelined).  Two quads per step; one with the optimizer step (its
    // operands take the registers of the second quad), and one for rows of
    // 64+ floats, where the second quad's gathered rows cost resident warps:
    // 96 -> 64 registers, 2 -> 4 blocks per SM (10000x10000 @95% batch 256 dW
    // 353 -> 343 us, the decoder workload's fused backward step +7 %; batch
    // 64 dW over halved rows at 95 % 93.2 -> 87.3 us, at 99 % 33.5 -> 31.1,
    // at 90 % 167.9 -> 168.1).
    constexpr int QPS = (OPT || BW >= 64) ? 1 : 2;
    int kb = (k0 & ~3) + 4 * grp;
    int c[2][4] = {};
    load_col_step<QPS>(a.col, kb, k1, npt, c);
    for (; kb < k1; kb += 4 * QPS * npt) {
      int cn[2][4] = {};
      load_col_step<QPS>(a.col, kb + 4 * QPS * npt, k1, npt, cn);
      sddmm_quads<BW, SM, OPT, !(FUSED && BW >= 64)>(a, xt, kb, k0, k1, npt, gmask, sub, dy, c,
                                                     QPS == 2 && kb + 4 * npt < k1);
#pragma unroll
      for (int q = 0; q < 2; ++q)
#pragma unroll
        for (int e = 0; e < 4; ++e) c[q][e] = cn[q][e];
    }
  }
}

// Second pass of an SpMM whose split lines only parked their parts'
// partials (launched with a.counter null).  Each split line takes TPL x pl
// threads: TPL = BW / VEC over its batch rows (VEC rows each) times pl over
// its parts, thread j of those adding parts j, j + pl, ... in order, eight
// loads at once (past the last part it loads the last again and leaves it
// out of the sum).  pl = 1 for lines of a few parts, so a 64-wide slice's
// 10000 quartered lines fit one wave; lines of many parts (the parts of a
// heavy-tailed table's longest lines) take up to a warp, their pl sums
// meeting by a butterfly of shuffles (a fixed order).  Its grid-dependency
// wait makes the first pass's partials visible.
template <int BW>
__host__ __device__ constexpr int split_sum_vec() {
  return BW >= 4 ? 4 : BW;
}

template <int BW>
__global__ void __launch_bounds__(256) split_sums(const SpmmArgs a, int64_t nsplit, int pl) {
  constexpr int VEC = split_sum_vec<BW>(), TPL = BW / VEC;
  griddep_wait();
  const int tpl = TPL * pl;  // a power of two; at most 32 when pl > 1
  const int64_t t = (int64_t)blockIdx.x * 256 + threadIdx.x;
  const int64_t w = t / tpl;
  const int r = (int)(t % tpl);
  const int b0 = (r % TPL) * VEC;
  const int j = r / TPL;
  const bool live = w < nsplit && b0 < a.nb;
  // With pl > 1 every lane of the warp meets the shuffles below: the lanes
  // past the last line read the last line's parts and store nothing.
  if (!live && pl == 1) return;
  const int4 sp = a.split[w < nsplit ? w : nsplit - 1];
  const float *q = a.partial + (int64_t)sp.z * BW + b0;  // b0 < BW
  float s[VEC];
#pragma unroll
  for (int i = 0; i < VEC; ++i) s[i] = 0.f;
  for (int p = j; p < sp.y; p += 8 * pl) {
    float x[8][VEC];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const float *rp = q + (int64_t)min(p + u * pl, sp.y - 1) * BW;
      if constexpr (VEC == 4) {
        const float4 f = __ldcg(reinterpret_cast<const float4 *>(rp));
        x[u][0] = f.x;
        x[u][1] = f.y;
        x[u][2] = f.z;
        x[u][3] = f.w;
      } else {
#pragma unroll
        for (int i = 0; i < VEC; ++i) x[u][i] = __ldcg(rp + i);
      }
    }
#pragma unroll
    for (int u = 0; u < 8; ++u)
      if (p + u * pl < sp.y) {
#pragma unroll
        for (int i = 0; i < VEC; ++i) s[i] += x[u][i];
      }
  }
  for (int off = TPL; off < tpl; off <<= 1)
#pragma unroll
    for (int i = 0; i < VEC; ++i) s[i] += __shfl_xor_sync(0xffffffffu, s[i], off);
  if (!live || j != 0) return;
  float *d = a.dst + (int64_t)b0 * a.ld + a.seg[sp.x].x;
#pragma unroll
  for (int i = 0; i < VEC; ++i)
    if (b0 + i < a.nb) d[(int64_t)i * a.ld] = s[i];
}

template <int BW, int LPS, bool PERM>
__global__ void __launch_bounds__(256) spmm_segments(const SpmmArgs a) {
  // Index / value streams do not depend on the transpose this kernel may
  // follow: pull them into L2 while waiting for it (without one to wait
  // for, the prefetch only delays the kernel's own loads).
  if (a.prefetch) {
    prefetch_segments(a.seg, a.nseg, a.idx, PERM ? (const void *)a.perm : (const void *)a.val,
                      LPS, blockIdx.x, gridDim.x);
    if (PERM) prefetch_share(a.val, a.nval, blockIdx.x, gridDim.x);
  }
  griddep_wait();
  spmm_part<BW, LPS, PERM>(a, a.src, blockIdx.x, gridDim.x);
}

template <int BW, int LPS, bool OPT = false>
__global__ void __launch_bounds__(256) sddmm_segments(const SddmmArgs a) {
  if (a.prefetch) prefetch_segments(a.seg, a.nseg, a.col, nullptr, LPS, blockIdx.x, gridDim.x);
  griddep_wait();
  sddmm_part<BW, LPS, false, OPT>(a, a.xt, blockIdx.x, gridDim.x);
}

// Both backward products in one launch: the first `cols_blocks` blocks run
// dX over the column segments, the rest run dW over the row segments (one
// team size for both parts).  PERM: dX reads the values through the
// column permutation (else from the column-ordered copy).  dX keeps the
// plain loop here: the look-ahead's registers would cost the shared grid a
// resident block per SM.
template <int BW, int LPS, bool PERM>
__global__ void __launch_bounds__(256) backward_segments(const SpmmArgs cols, const SddmmArgs rows,
                                                         int cols_blocks) {
  if (cols.prefetch) {  // waiting on the transpose: pull the streams into L2
    if ((int)blockIdx.x < cols_blocks) {
      prefetch_segments(cols.seg, cols.nseg, cols.idx,
                        PERM ? (const void *)cols.perm : (const void *)cols.val, LPS, blockIdx.x,
                        cols_blocks);
      if (PERM) prefetch_share(cols.val, cols.nval, blockIdx.x, cols_blocks);
    } else {
      prefetch_segments(rows.seg, rows.nseg, rows.col, nullptr, LPS, blockIdx.x - cols_blocks,
                        gridDim.x - cols_blocks);
    }
  }
  griddep_wait();
  if ((int)blockIdx.x < cols_blocks)
    spmm_part<BW, LPS, PERM, false, false>(cols, cols.src, blockIdx.x, cols_blocks);
  else
    sddmm_part<BW, LPS, false, false, true>(rows, rows.xt, blockIdx.x - cols_blocks,
                                            gridDim.x - cols_blocks);
}

// Rows of the slice per transpose tile (tiles are 32 columns by this many
// rows, so that wide slices still spread over many blocks).
template <int BW>
__host__ __device__ constexpr int transpose_rows() {
  return BW < 32 ? BW : 32;
}

// Tiles of one transpose: 32-column tiles times row tiles.
template <int BW>
inline int64_t transpose_tiles(int64_t ncols) {
  return (ncols + 31) / 32 * (BW / transpose_rows<BW>());
}

// dst[c * BW + b] = b < nb ? src[b * ld + c] : 0 for one tile of 32 columns
// by transpose_rows<BW>() rows (the row tile varies fastest with `tile`).
template <int BW>
__device__ __forceinline__ void transpose_tile(const float *__restrict__ src, int64_t ld, int nb,
                                               int64_t ncols, float *__restrict__ dst, int64_t tile,
                                               float (*buf)[33]) {
  constexpr int RT = transpose_rows<BW>(), NRT = BW / RT;
  const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;
  const int64_t c0 = tile / NRT * 32;
  const int r0 = (int)(tile % NRT) * RT;
  for (int b = ty; b < RT; b += 8) {
    const int64_t c = c0 + tx;
    buf[b][tx] = (r0 + b < nb && c < ncols) ? src[(int64_t)(r0 + b) * ld + c] : 0.f;
  }
  __syncthreads();
  for (int f = threadIdx.x; f < 32 * RT; f += 256) {
    const int cc = f / RT, b = f % RT;
    if (c0 + cc < ncols) dst[(c0 + cc) * BW + r0 + b] = buf[b][cc];
  }
}

template <int BW>
__global__ void __launch_bounds__(256) transpose_pad(const float *__restrict__ src, int64_t ld,
                                                     int nb, int64_t ncols,
                                                     float *__restrict__ dst) {
  __shared__ float buf[transpose_rows<BW>()][33];
  griddep_launch();
  griddep_wait();
  transpose_tile<BW>(src, ld, nb, ncols, dst, blockIdx.x, buf);
}

// Two transposes in one launch (X for dW, dY for dX and dW): the first
// `a_tiles` blocks handle a, the rest b.
template <int BW>
__global__ void __launch_bounds__(256) transpose_pair(const float *__restrict__ a, int64_t a_ld,
                                                      int64_t a_cols, float *__restrict__ at,
                                                      const float *__restrict__ b, int64_t b_ld,
                                                      int64_t b_cols, float *__restrict__ bt,
                                                      int nb, int64_t a_tiles) {
  __shared__ float buf[transpose_rows<BW>()][33];
  griddep_launch();
  griddep_wait();
  if ((int64_t)blockIdx.x < a_tiles)
    transpose_tile<BW>(a, a_ld, nb, a_cols, at, blockIdx.x, buf);
  else
    transpose_tile<BW>(b, b_ld, nb, b_cols, bt, blockIdx.x - a_tiles, buf);
}

}  // namespace snack
