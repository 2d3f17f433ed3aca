// Speculative accept step ("Speculative Decoding이란?", section 3 Steps 3-4,
// section 6; greedy equivalence in section 5).
//
// Stochastic sequence mode, three launches:
//  1. accept_stats_kernel, persistent warps: every p / q logit row is cut
//     into items of 1024 logits; a warp holds an item in registers (one HBM
//     pass, the next item's loads in flight meanwhile), takes the exact item
//     maximum and the sum of exp(l - max) (pairwise fp32 per lane,
//     double-float across lanes). When the caller supplies the target
//     rows' statistics per 32-logit slice (spec_accept_prestat, from the
//     fused lm_head), the pass reads the draft rows only and merges the
//     supplied slices, 512 to an item, into the same item statistics.
//  2. accept_decide_kernel, one block per batch row: merges each row's item
//     statistics (one warp per row), evaluates alpha_i = min(1, P(d_i) /
//     Q(d_i)) for every draft, finds the first rejection r and records r
//     with the normalisers of row r.
//  3. accept_resid_kernel, grid (chunk, batch row): each block sums the
//     distribution to draw from — max(0, P_r - Q_r), or P_{n+1} after full
//     acceptance — over its vocabulary chunk. The last block of the batch row
//     finds the chunk that holds u * S with a warp scan of the chunk sums,
//     re-scans that chunk with a double-float block scan, and writes
//     accepted_len and next_token.
// Greedy modes, one launch: accept_argmax_kernel reduces chunks to
// (max, smallest index); the last block of a batch row merges them and walks
// the chain or tree.
//
// Every per-element value that decides a draw (P, Q, max(0, P - Q)) is formed
// with explicit rn intrinsics so that the block that sums a chunk and the
// block that re-scans it compute bit-identical values.
#include <float.h>

#include <atomic>
#include <cooperative_groups.h>

#include "common.cuh"
#include "internal.h"

namespace w4a16 {

namespace cg = cooperative_groups;

constexpr int kAccThreads = 256;
constexpr int kAccWarps = kAccThreads / 32;
constexpr int kArgPT = 64;                           // logits a thread holds in the argmax pass
constexpr int kArgChunk = kAccThreads * kArgPT;      // 16384
constexpr int kStatPT = 32;                          // logits a lane holds per statistics item
constexpr int kStatItem = 32 * kStatPT;              // 1024 logits: one warp's item
constexpr int kSliceItem = 32 * kStatPT / 2;         // 512 caller-supplied slice statistics: one warp's item
constexpr int kStatBlocksPerSm = 2;                  // statistics blocks resident per SM (launch bounds)
constexpr int kDecThreads = 512;                     // decide kernel: 15 merging warps + 1 loading warp
constexpr int kMaxStatRows = 2 * 1024 + 1;           // statistics rows of one batch row (n <= 1024)
constexpr int kMaxNodes = 1025;                      // rows of one batch element in greedy mode (n <= 1024)
constexpr int kCounterBank2 = 32768;                 // second bank of completion counters (B <= 32768)
constexpr int kResidPT = 16;                         // logits a thread holds in the residual pass and re-scan
constexpr int kMaxChunk2 = kAccThreads * kResidPT;   // 4096
constexpr int kMinChunk2 = 1024;
constexpr int kMaxCh2 = 256;                         // residual chunks per batch row (V <= 2^20 fits)

// Double-float value hi + lo (two fp32 words). GB300 executes only a couple
// of fp64 operations per clock per SM, so sums that need more than fp32 are
// carried in this form with error-free transformations on the fp32 pipe:
// TwoSum (Knuth, TAOCP vol. 2, 4.2.2) and FastTwoSum (Dekker 1971), and the
// fma-based exact product.
struct DF {
  float hi, lo;
};

__device__ __forceinline__ DF two_sum(float a, float b) {
  const float s = __fadd_rn(a, b);
  const float bb = __fsub_rn(s, a);
  const float e = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb));
  return DF{s, e};
}
__device__ __forceinline__ DF fast_two_sum(float a, float b) {  // |a| >= |b|
  const float s = __fadd_rn(a, b);
  return DF{s, __fsub_rn(b, __fsub_rn(s, a))};
}
__device__ __forceinline__ DF df_add(DF a, DF b) {
  const DF s = two_sum(a.hi, b.hi);
  return fast_two_sum(s.hi, __fadd_rn(s.lo, __fadd_rn(a.lo, b.lo)));
}
__device__ __forceinline__ DF df_add_f(DF a, float b) {
  const DF s = two_sum(a.hi, b);
  return fast_two_sum(s.hi, __fadd_rn(s.lo, a.lo));
}
__device__ __forceinline__ DF df_mul_f(DF a, float b) {
  const float p = __fmul_rn(a.hi, b);
  const float e = __fmaf_rn(a.hi, b, -p);
  return fast_two_sum(p, __fmaf_rn(a.lo, b, e));
}
__device__ __forceinline__ float df_val(DF a) { return __fadd_rn(a.hi, a.lo); }
// sign of a - b
__device__ __forceinline__ bool df_gt(DF a, DF b) {
  const DF d = df_add(a, DF{-b.hi, -b.lo});
  return d.hi > 0.0f || (d.hi == 0.0f && d.lo > 0.0f);
}

struct RowStat {
  float m;
  float pad;
  DF s;
};

struct Decision {  // first rejection r and the normalisers of the rows the final draw uses
  int r;
  float mp, mq;
  float izp, izq;  // 1 / Z
  int pad[3];
};

struct ChunkSum {
  DF r;  // sum of the distribution being sampled
  DF p;  // sum of P_r (fallback when the corrected distribution is all zero)
};

struct ArgPart {
  float v;
  int idx;
};

// ---------------------------------------------------------- block helpers
// Block-wide max / sums, result returned to every thread.
__device__ float block_max(float v) {
  __shared__ float sm[kAccWarps];
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  if ((threadIdx.x & 31) == 0) sm[threadIdx.x >> 5] = v;
  __syncthreads();
  float r = sm[0];
#pragma unroll
  for (int i = 1; i < kAccWarps; ++i) r = fmaxf(r, sm[i]);
  __syncthreads();
  return r;
}

__device__ __forceinline__ DF shfl_xor_df(DF v, int o) {
  return DF{__shfl_xor_sync(0xffffffffu, v.hi, o), __shfl_xor_sync(0xffffffffu, v.lo, o)};
}

// Block-wide double-float sum, returned to every thread.
__device__ DF block_sum(DF v) {
  __shared__ DF sm[kAccWarps];
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = df_add(v, shfl_xor_df(v, o));
  if ((threadIdx.x & 31) == 0) sm[threadIdx.x >> 5] = v;
  __syncthreads();
  DF r = sm[0];
#pragma unroll
  for (int i = 1; i < kAccWarps; ++i) r = df_add(r, sm[i]);
  __syncthreads();
  return r;
}

// Exclusive prefix sum over the block (thread order), double-float.
__device__ DF block_exclusive_scan(DF v) {
  __shared__ DF wsum[kAccWarps];
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  DF incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const DF y{__shfl_up_sync(0xffffffffu, incl.hi, o), __shfl_up_sync(0xffffffffu, incl.lo, o)};
    if (lane >= o) incl = df_add(incl, y);
  }
  if (lane == 31) wsum[w] = incl;
  __syncthreads();
  DF before{0.0f, 0.0f};
  for (int i = 0; i < w; ++i) before = df_add(before, wsum[i]);
  __syncthreads();
  return df_add(before, df_add(incl, DF{-v.hi, -v.lo}));
}

// Statistics row rr of a batch row's 2n+1 rows: target rows 0..n, then draft
// rows; with q_only (target statistics supplied by the caller) the rows are
// the draft rows alone, rr = b * n + i.
__device__ __forceinline__ const float* stat_row_ptr(const float* p, const float* q, int n, int64_t V, int rr,
                                                     bool q_only) {
  if (q_only) return q + (int64_t)rr * V;
  const int per = 2 * n + 1;
  const int b = rr / per, i = rr % per;
  if (i <= n) return p + ((int64_t)b * (n + 1) + i) * V;
  return q + ((int64_t)b * n + (i - n - 1)) * V;
}

// Merge a row's chunk statistics with one warp: M = max m_c,
// Z = sum_c s_c exp(m_c - M); every lane returns the same M and Z (df_add is
// commutative bit for bit, so the butterfly leaves one value in all lanes).
// The statistics (written by an earlier kernel) are read through L2; the
// first kMergeRegs per lane are held in registers between the two passes.
constexpr int kMergeRegs = 8;
__device__ void warp_merge_row(const RowStat* st, int ch, float& M, DF& Z) {
  const int lane = threadIdx.x & 31;
  float4 e[kMergeRegs];
  float m = -FLT_MAX;
#pragma unroll
  for (int k = 0; k < kMergeRegs; ++k) {
    const int c = lane + 32 * k;
    e[k] = c < ch ? __ldcg(reinterpret_cast<const float4*>(st + c)) : make_float4(-FLT_MAX, 0.0f, 0.0f, 0.0f);
    m = fmaxf(m, e[k].x);
  }
  for (int c = lane + 32 * kMergeRegs; c < ch; c += 32) m = fmaxf(m, __ldcg(&st[c].m));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  DF z{0.0f, 0.0f};
#pragma unroll
  for (int k = 0; k < kMergeRegs; ++k)
    if (lane + 32 * k < ch) z = df_add(z, df_mul_f(DF{e[k].z, e[k].w}, expf(__fsub_rn(e[k].x, m))));
  for (int c = lane + 32 * kMergeRegs; c < ch; c += 32) {
    const float4 f = __ldcg(reinterpret_cast<const float4*>(st + c));
    z = df_add(z, df_mul_f(DF{f.z, f.w}, expf(__fsub_rn(f.x, m))));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) z = df_add(z, shfl_xor_df(z, o));
  M = m;
  Z = z;
}

// Inclusive prefix sum over the warp (lane order), double-float.
__device__ __forceinline__ DF warp_inclusive_scan(DF v) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const DF y{__shfl_up_sync(0xffffffffu, v.hi, o), __shfl_up_sync(0xffffffffu, v.lo, o)};
    if (lane >= o) v = df_add(y, v);
  }
  return v;
}

// Load this thread's share of [x0, x1) into registers (missing slots: -FLT_MAX).
template <bool VEC, int PT>
__device__ __forceinline__ void load_chunk(const float* row, int x0, int x1, float (&v)[PT]) {
  if (VEC) {
#pragma unroll
    for (int j = 0; j < PT / 4; ++j) {
      const int xi = x0 + (j * kAccThreads + (int)threadIdx.x) * 4;
      float4 t = make_float4(-FLT_MAX, -FLT_MAX, -FLT_MAX, -FLT_MAX);
      if (xi < x1) t = ldg_stream_f4(reinterpret_cast<const float4*>(row + xi));
      v[4 * j] = t.x;
      v[4 * j + 1] = t.y;
      v[4 * j + 2] = t.z;
      v[4 * j + 3] = t.w;
    }
  } else {
#pragma unroll
    for (int j = 0; j < PT; ++j) {
      const int xi = x0 + j * kAccThreads + (int)threadIdx.x;
      v[j] = xi < x1 ? ldg_stream_f(row + xi) : -FLT_MAX;
    }
  }
}

// ------------------------------------------------------- pass 1: row stats
// Items are (statistics row, chunk of kStatItem logits); one warp takes one
// item, its lanes holding kStatPT logits each, and the warps are persistent
// (item it, it + warps, ...).

// Exact maximum m of the item and sum of exp(l - m) (pairwise fp32 per lane,
// double-float across lanes); lane 0 stores them. Padding (-FLT_MAX) adds 0.
// exp via ex2.approx (__expf): its relative error grows with |l - m|, so it is
// smallest on the terms that carry the sum; about 1e-7 of the total.
__device__ __forceinline__ void item_stats(const float (&v)[kStatPT], RowStat* out, bool store) {
  float m = -FLT_MAX;
#pragma unroll
  for (int j = 0; j < kStatPT; ++j) m = fmaxf(m, v[j]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  float t[kStatPT / 4];
#pragma unroll
  for (int j = 0; j < kStatPT / 4; ++j)
    t[j] = (__expf(v[4 * j] - m) + __expf(v[4 * j + 1] - m)) + (__expf(v[4 * j + 2] - m) + __expf(v[4 * j + 3] - m));
#pragma unroll
  for (int w = kStatPT / 8; w >= 1; w >>= 1)
#pragma unroll
    for (int j = 0; j < w; ++j) t[j] += t[j + w];
  DF s{t[0], 0.0f};
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) s = df_add(s, shfl_xor_df(s, o));
  if (store && (threadIdx.x & 31) == 0) *out = RowStat{m, 0.0f, s};
}

__device__ __forceinline__ void item_range(int n, int V, int ch, int it, int& rr, int& x0, int& x1) {
  rr = it / ch;
  x0 = (it - rr * ch) * kStatItem;
  x1 = min(V, x0 + kStatItem);
}

// A warp's item goes into registers (float4 loads when V % 4 == 0: rows are
// then 16-byte aligned and every float4 lies wholly inside or outside the
// row). Each warp keeps the next item's loads in flight while it reduces the
// current one, so the HBM stream does not stop while the exponentials run.
template <bool VEC>
__device__ __forceinline__ void load_item(const float* p, const float* q, int n, int V, int ch, int it, bool q_only,
                                          float (&v)[kStatPT]) {
  int rr, x0, x1;
  item_range(n, V, ch, it, rr, x0, x1);
  const float* row = stat_row_ptr(p, q, n, V, rr, q_only);
  const int lane = threadIdx.x & 31;
  if (VEC) {
#pragma unroll
    for (int j = 0; j < kStatPT / 4; ++j) {
      const int xi = x0 + (j * 32 + lane) * 4;
      float4 t = make_float4(-FLT_MAX, -FLT_MAX, -FLT_MAX, -FLT_MAX);
      if (xi < x1) t = ldg_stream_f4(reinterpret_cast<const float4*>(row + xi));
      v[4 * j] = t.x;
      v[4 * j + 1] = t.y;
      v[4 * j + 2] = t.z;
      v[4 * j + 3] = t.w;
    }
  } else {
#pragma unroll
    for (int j = 0; j < kStatPT; ++j) {
      const int xi = x0 + j * 32 + lane;
      v[j] = xi < x1 ? ldg_stream_f(row + xi) : -FLT_MAX;
    }
  }
}

// Items over the caller-supplied statistics of the target rows (the fused
// lm_head's (max, sum exp(l - max)) per 32-logit slice, V / 32 per row): an
// item is kSliceItem consecutive slices of one row, a lane holding
// kStatPT / 2 (max, sum) pairs; missing slices are (-FLT_MAX, 0).
__device__ __forceinline__ void load_slice_item(const float2* ps, int V, int chs, int it, float (&v)[kStatPT]) {
  const int ns = V / 32;
  const int row = it / chs;
  const int s0 = (it - row * chs) * kSliceItem;
  const float2* src = ps + (int64_t)row * ns;
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int j = 0; j < kStatPT / 2; ++j) {
    const int si = s0 + j * 32 + lane;
    float2 t = make_float2(-FLT_MAX, 0.0f);
    if (si < ns) t = __ldcs(src + si);
    v[2 * j] = t.x;
    v[2 * j + 1] = t.y;
  }
}

// Merged statistics of an item of slices: m = max of the slice maxima,
// sum of s_j exp(m_j - m) (fp32 per lane, pairwise; double-float across
// lanes), as item_stats does for raw logits.
__device__ __forceinline__ void slice_item_stats(const float (&v)[kStatPT], RowStat* out, bool store) {
  float m = -FLT_MAX;
#pragma unroll
  for (int j = 0; j < kStatPT / 2; ++j) m = fmaxf(m, v[2 * j]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  float t[kStatPT / 4];
#pragma unroll
  for (int j = 0; j < kStatPT / 4; ++j)
    t[j] = __fmul_rn(v[4 * j + 1], __expf(v[4 * j] - m)) + __fmul_rn(v[4 * j + 3], __expf(v[4 * j + 2] - m));
#pragma unroll
  for (int w = kStatPT / 8; w >= 1; w >>= 1)
#pragma unroll
    for (int j = 0; j < w; ++j) t[j] += t[j + w];
  DF s{t[0], 0.0f};
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) s = df_add(s, shfl_xor_df(s, o));
  if (store && (threadIdx.x & 31) == 0) *out = RowStat{m, 0.0f, s};
}

template <bool VEC>
__global__ void __launch_bounds__(kAccThreads, kStatBlocksPerSm) accept_stats_kernel(const float* __restrict__ p,
                                                                       const float* __restrict__ q, int n, int V,
                                                                       int ch, int items, int q_only,
                                                                       const float2* __restrict__ p_stats, int chs,
                                                                       int slice_items, RowStat* __restrict__ stats,
                                                                       int64_t stats_cap, unsigned* err) {
  grid_launch_dependents();
  grid_dependency_wait();
  // items [0, items): logit chunks; [items, items + slice_items): slices of
  // the supplied target statistics (q_only mode), written after them
  const int all = items + slice_items;
  auto load = [&](int i, float (&v)[kStatPT]) {
    if (i < items)
      load_item<VEC>(p, q, n, V, ch, i, q_only, v);
    else
      load_slice_item(p_stats, V, chs, i - items, v);
  };
  auto reduce = [&](int i, const float (&v)[kStatPT]) {
    const bool ok = in_bounds(err, i, stats_cap);
    if (i < items)
      item_stats(v, stats + i, ok);
    else
      slice_item_stats(v, stats + i, ok);
  };
  const int nw = gridDim.x * kAccWarps;
  int it = blockIdx.x * kAccWarps + (threadIdx.x >> 5);
  float va[kStatPT], vb[kStatPT];
  if (it < all) load(it, va);
  while (it < all) {  // two items per trip: the buffers swap roles
    const int i1 = it + nw;
    if (i1 < all) load(i1, vb);
    reduce(it, va);
    if (i1 >= all) break;
    const int i2 = i1 + nw;
    if (i2 < all) load(i2, va);
    reduce(i1, vb);
    it = i2;
  }
}

// Decision of batch row b by one 512-thread block (kDecThreads): merge each
// statistics row's chunks (one warp per row, 15 merging warps; the last warp
// fetches the drafts' own logits meanwhile), evaluate alpha_i = min(1,
// P_i(d_i) / Q_i(d_i)) for every draft, find the first rejection r and return
// r with the normalisers of row r (the same value in every thread).
struct DecideShared {
  float sM[kMaxStatRows];
  DF sZ[kMaxStatRows];
  float sLp[kMaxNodes], sLq[kMaxNodes];  // P_i / Q_i logits at d_i (n <= 1024)
  int first_reject;
};

__device__ Decision decide_batch_row(const float* __restrict__ p, const float* __restrict__ q,
                                     const int32_t* __restrict__ d, const float* __restrict__ u, int n, int V, int ch,
                                     const RowStat* __restrict__ stats, int prestat, int chs, int B, int b,
                                     DecideShared& ds, unsigned* err) {
  constexpr int kMergeWarps = kDecThreads / 32 - 1;
  const int per = 2 * n + 1;
  // row statistics: all 2n + 1 rows from the statistics pass (ch items a
  // row), or (prestat) the draft rows (ch items a row) followed, after all
  // batch rows' draft rows, by the target rows merged from the caller's
  // slices (chs items a row)
  const RowStat* st = prestat ? stats + (int64_t)b * n * ch : stats + (int64_t)b * per * ch;
  const RowStat* st_p = stats + (int64_t)B * n * ch + (int64_t)b * (n + 1) * chs;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (warp == kMergeWarps) {
    // the drafts' own logits, fetched while the other warps merge
    for (int i = lane; i < n; i += 32) {
      const int di = d[(int64_t)b * n + i];
      float lp = 0.0f, lq = 0.0f;
      if (di < 0 || di >= V) {
        report_error(err, kErrInput);
        lp = -FLT_MAX;  // marks the draft rejected
      } else {
        lp = p[((int64_t)b * (n + 1) + i) * V + di];
        lq = q[((int64_t)b * n + i) * V + di];
      }
      ds.sLp[i] = lp;
      ds.sLq[i] = lq;
    }
  } else {
    for (int row = warp; row < per; row += kMergeWarps) {
      float M;
      DF Z;
      if (!prestat)
        warp_merge_row(st + (int64_t)row * ch, ch, M, Z);
      else if (row <= n)
        warp_merge_row(st_p + (int64_t)row * chs, chs, M, Z);
      else
        warp_merge_row(st + (int64_t)(row - n - 1) * ch, ch, M, Z);
      if (lane == 0) {
        ds.sM[row] = M;
        ds.sZ[row] = Z;
      }
    }
  }
  if (threadIdx.x == 0) ds.first_reject = n;
  __syncthreads();
  for (int i = threadIdx.x; i < n; i += kDecThreads) {
    bool reject;
    if (ds.sLp[i] == -FLT_MAX) {
      reject = true;
    } else {
      // alpha = min(1, P / Q) = min(1, (e_p * Z_q) / (e_q * Z_p)), fp32 (a few ulp)
      const float ep = exp_of_diff(ds.sLp[i], ds.sM[i]);
      const float eq = exp_of_diff(ds.sLq[i], ds.sM[n + 1 + i]);
      const float num = __fmul_rn(ep, df_val(ds.sZ[n + 1 + i])), den = __fmul_rn(eq, df_val(ds.sZ[i]));
      const float alpha = den > 0.0f ? fminf(1.0f, __fdiv_rn(num, den)) : 1.0f;
      reject = !(u[(int64_t)b * (n + 1) + i] < alpha);
    }
    if (reject) atomicMin(&ds.first_reject, i);
  }
  __syncthreads();
  Decision D;
  D.r = ds.first_reject;
  D.pad[0] = D.pad[1] = D.pad[2] = 0;
  D.mp = ds.sM[D.r];
  D.izp = __frcp_rn(df_val(ds.sZ[D.r]));
  if (D.r < n) {
    D.mq = ds.sM[n + 1 + D.r];
    D.izq = __frcp_rn(df_val(ds.sZ[n + 1 + D.r]));
  } else {
    D.mq = 0.0f;
    D.izq = 0.0f;
  }
  return D;
}

// One block per batch row: the decision, for the residual pass.
__global__ void __launch_bounds__(kDecThreads) accept_decide_kernel(
    const float* __restrict__ p, const float* __restrict__ q, const int32_t* __restrict__ d,
    const float* __restrict__ u, int n, int V, int ch, const RowStat* __restrict__ stats, int prestat, int chs,
    Decision* __restrict__ dec, unsigned* err) {
  grid_launch_dependents();
  grid_dependency_wait();
  __shared__ DecideShared ds;
  const Decision D = decide_batch_row(p, q, d, u, n, V, ch, stats, prestat, chs, (int)gridDim.x, (int)blockIdx.x, ds,
                                      err);
  if (threadIdx.x == 0) dec[blockIdx.x] = D;
}

// --------------------------------------------- pass 2: residual and draw
// Value of the distribution being sampled at x (bit-identical wherever computed).
struct ResidFn {
  const float* prow;  // P_r row logits (or P_{n+1} after full acceptance)
  const float* qrow;  // Q_r row logits, NULL after full acceptance
  float mp, ip, mq, iq;
  __device__ __forceinline__ float pv_of(float lp) const { return __fmul_rn(exp_of_diff(lp, mp), ip); }
  __device__ __forceinline__ float rv_of(float lp, float lq) const {
    const float pv = pv_of(lp);
    if (!qrow) return pv;
    const float qv = __fmul_rn(exp_of_diff(lq, mq), iq);
    return fmaxf(__fsub_rn(pv, qv), 0.0f);
  }
  __device__ __forceinline__ float pval(int x) const { return pv_of(prow[x]); }
  __device__ __forceinline__ float rval(int x) const { return rv_of(prow[x], qrow ? qrow[x] : 0.0f); }
};

// VEC: V and chunk2 multiples of 4, so the chunk is whole float4s.
template <int RS, bool VEC>  // values per thread in a chunk: chunk2 <= RS * kAccThreads
__global__ void __launch_bounds__(kAccThreads, 4) accept_resid_kernel(
    const float* __restrict__ p, const float* __restrict__ q, const float* __restrict__ u, int n, int V,
    int chunk2, const Decision* __restrict__ dec, ChunkSum* __restrict__ csum, int* __restrict__ counters,
    int32_t* __restrict__ acc_out, int32_t* __restrict__ next_out, int32_t* __restrict__ node_out, int64_t csum_cap,
    unsigned* err) {
  grid_launch_dependents();
  grid_dependency_wait();
  const int b = blockIdx.y;
  const int r = __ldcg(&dec[b].r);
  ResidFn f;
  f.prow = p + ((int64_t)b * (n + 1) + r) * V;
  f.mp = __ldcg(&dec[b].mp);
  f.ip = __ldcg(&dec[b].izp);
  if (r < n) {
    f.qrow = q + ((int64_t)b * n + r) * V;
    f.mq = __ldcg(&dec[b].mq);
    f.iq = __ldcg(&dec[b].izq);
  } else {
    f.qrow = nullptr;
    f.mq = 0.0f;
    f.iq = 0.0f;
  }
  const int x0 = blockIdx.x * chunk2, x1 = min(V, x0 + chunk2);
  const uint64_t pol = policy_evict_first();
  // all of this thread's logits are loaded before any is used (one latency)
  float lp[RS], lq[RS];
  auto index_of = [&](int j) {
    return VEC ? x0 + ((j / 4) * kAccThreads + (int)threadIdx.x) * 4 + (j % 4) : x0 + j * kAccThreads + (int)threadIdx.x;
  };
  if (VEC) {
#pragma unroll
    for (int j = 0; j < RS / 4; ++j) {
      const int xi = x0 + (j * kAccThreads + (int)threadIdx.x) * 4;
      float4 tp = make_float4(0.f, 0.f, 0.f, 0.f), tq = tp;
      if (xi < x1) {  // the rows' last read: evict-first
        tp = ldg_hint_f4(reinterpret_cast<const float4*>(f.prow + xi), pol);
        if (f.qrow) tq = ldg_hint_f4(reinterpret_cast<const float4*>(f.qrow + xi), pol);
      }
      lp[4 * j] = tp.x, lp[4 * j + 1] = tp.y, lp[4 * j + 2] = tp.z, lp[4 * j + 3] = tp.w;
      lq[4 * j] = tq.x, lq[4 * j + 1] = tq.y, lq[4 * j + 2] = tq.z, lq[4 * j + 3] = tq.w;
    }
  } else {
#pragma unroll
    for (int j = 0; j < RS; ++j) {
      const int x = index_of(j);
      lp[j] = x < x1 ? f.prow[x] : 0.0f;
      lq[j] = (x < x1 && f.qrow) ? f.qrow[x] : 0.0f;
    }
  }
  float sr = 0.0f, sp = 0.0f;
#pragma unroll
  for (int j = 0; j < RS; ++j) {
    if (index_of(j) < x1) {
      const float pv = f.pv_of(lp[j]);
      if (f.qrow) {
        sr += fmaxf(__fsub_rn(pv, __fmul_rn(exp_of_diff(lq[j], f.mq), f.iq)), 0.0f);  // as rv_of
        sp += pv;
      } else {
        sr += pv;
      }
    }
  }
  const DF SR = block_sum(DF{sr, 0.0f});
  const DF SP = block_sum(DF{sp, 0.0f});
  __shared__ int last;
  if (threadIdx.x == 0) {
    const int64_t ci = (int64_t)b * gridDim.x + blockIdx.x;
    if (in_bounds(err, ci, csum_cap)) csum[ci] = ChunkSum{SR, SP};
    __threadfence();
    last = in_bounds(err, kCounterBank2 + b, kMaxCounters) && atomicAdd(&counters[b], 1) == (int)gridDim.x - 1;
  }
  __syncthreads();
  if (!last) return;
  __threadfence();

  // ---- the last block of batch row b draws the next token
  __shared__ DF sh_t, sh_before;
  __shared__ int sh_chunk, sh_usep, sh_found;
  __shared__ ChunkSum sh_cs[kMaxCh2];  // gridDim.x <= kMaxCh2
  for (int c = threadIdx.x; c < (int)gridDim.x; c += kAccThreads) {
    const ChunkSum* cs = csum + (int64_t)b * gridDim.x + c;
    sh_cs[c].r = DF{__ldcg(&cs->r.hi), __ldcg(&cs->r.lo)};
    sh_cs[c].p = DF{__ldcg(&cs->p.hi), __ldcg(&cs->p.lo)};
  }
  __syncthreads();
  if (threadIdx.x < 32) {
    // warp 0 finds the chunk holding u * S: each lane sums a contiguous run
    // of chunk sums, a warp scan gives the prefix at each run, and the first
    // lane whose prefix passes u * S walks its run
    const int lane = threadIdx.x, C = gridDim.x;
    const int per_l = (C + 31) / 32;
    const int c0 = min(C, lane * per_l), c1 = min(C, c0 + per_l);
    DF mine{0.0f, 0.0f};
    for (int c = c0; c < c1; ++c) mine = df_add(mine, sh_cs[c].r);
    DF incl = warp_inclusive_scan(mine);
    DF S{__shfl_sync(0xffffffffu, incl.hi, 31), __shfl_sync(0xffffffffu, incl.lo, 31)};
    int usep = 0;
    if (f.qrow && S.hi == 0.0f) {  // corrected distribution is all zero: draw from P_r
      usep = 1;
      mine = DF{0.0f, 0.0f};
      for (int c = c0; c < c1; ++c) mine = df_add(mine, sh_cs[c].p);
      incl = warp_inclusive_scan(mine);
      S = DF{__shfl_sync(0xffffffffu, incl.hi, 31), __shfl_sync(0xffffffffu, incl.lo, 31)};
    }
    const DF t = df_mul_f(S, u[(int64_t)b * (n + 1) + n]);
    const unsigned passed = __ballot_sync(0xffffffffu, c1 > c0 && df_gt(incl, t));
    const DF excl{__shfl_up_sync(0xffffffffu, incl.hi, 1), __shfl_up_sync(0xffffffffu, incl.lo, 1)};
    if (passed == 0u) {
      if (lane == 0) {  // u * S is not below the total: no chunk holds it
        sh_t = t;
        sh_before = S;
        sh_chunk = -1;
      }
    } else if (lane == __ffs(passed) - 1) {
      DF cum = lane == 0 ? DF{0.0f, 0.0f} : excl;
      int cstar = c1 - 1;  // the run's prefix passes u * S; rounding may place the step at its end
      for (int c = c0; c < c1; ++c) {
        const DF nxt = df_add(cum, usep ? sh_cs[c].p : sh_cs[c].r);
        if (df_gt(nxt, t)) {
          cstar = c;
          break;
        }
        if (c + 1 < c1) cum = nxt;
      }
      sh_t = t;
      sh_before = cum;
      sh_chunk = cstar;
    }
    if (lane == 0) {
      sh_usep = usep;
      sh_found = INT_MAX;
      counters[b] = 0;
    }
  }
  __syncthreads();
  const int usep = sh_usep;
  auto val = [&](int x) { return usep ? f.pval(x) : f.rval(x); };
  if (sh_chunk >= 0) {
    // coalesced loads of the chunk (stride kAccThreads) into shared memory,
    // then a contiguous sub-range per thread (at most RS values) for the
    // double-float running sums from a block scan
    __shared__ float sv[RS * kAccThreads + RS * kAccThreads / 32];  // one pad word per 32: conflict-free row reads
    const int c0 = sh_chunk * chunk2, c1 = min(V, c0 + chunk2);
    {
      float lp[RS], lq[RS];
#pragma unroll
      for (int j = 0; j < RS; ++j) {
        const int x = min(c0 + j * kAccThreads + (int)threadIdx.x, V - 1);
        lp[j] = f.prow[x];
        lq[j] = f.qrow ? f.qrow[x] : 0.0f;
      }
#pragma unroll
      for (int j = 0; j < RS; ++j) {
        const int o = j * kAccThreads + (int)threadIdx.x;
        if (c0 + o < c1) sv[o + (o >> 5)] = usep ? f.pv_of(lp[j]) : f.rv_of(lp[j], lq[j]);
      }
    }
    __syncthreads();
    const int per_t = (c1 - c0 + kAccThreads - 1) / kAccThreads;
    const int a0 = min(c1, c0 + (int)threadIdx.x * per_t), a1 = min(c1, a0 + per_t);
    float vals[RS];
#pragma unroll
    for (int j = 0; j < RS; ++j) {
      const int k = a0 + j - c0;
      vals[j] = (a0 + j < a1) ? sv[k + (k >> 5)] : 0.0f;
    }
    DF mine{0.0f, 0.0f};
#pragma unroll
    for (int j = 0; j < RS; ++j) mine = df_add_f(mine, vals[j]);
    DF run = df_add(sh_before, block_exclusive_scan(mine));
    const DF t = sh_t;
    int hit = INT_MAX;
#pragma unroll
    for (int j = 0; j < RS; ++j) {
      if (a0 + j < a1 && hit == INT_MAX) {
        run = df_add_f(run, vals[j]);
        if (df_gt(run, t)) hit = a0 + j;
      }
    }
    if (hit != INT_MAX) atomicMin(&sh_found, hit);
  }
  __syncthreads();
  if (sh_found == INT_MAX) {
    // rounding left no crossing: first positive index after the chosen chunk,
    // else the last positive index of the row
    const int start = sh_chunk >= 0 ? min(V, (sh_chunk + 1) * chunk2) : V;
    int first_after = INT_MAX, last_pos = -1;
    for (int x = threadIdx.x; x < V; x += kAccThreads) {
      if (val(x) > 0.0f) {
        if (x >= start) first_after = min(first_after, x);
        last_pos = max(last_pos, x);
      }
    }
    __shared__ int sh_fa, sh_lp;
    if (threadIdx.x == 0) {
      sh_fa = INT_MAX;
      sh_lp = -1;
    }
    __syncthreads();
    if (first_after != INT_MAX) atomicMin(&sh_fa, first_after);
    if (last_pos >= 0) atomicMax(&sh_lp, last_pos);
    __syncthreads();
    if (threadIdx.x == 0) sh_found = sh_fa != INT_MAX ? sh_fa : (sh_lp >= 0 ? sh_lp : 0);
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    acc_out[b] = r;
    next_out[b] = sh_found;
    if (node_out) node_out[b] = r;  // a sequence draft's node index is its depth
  }
}

// -------------------------------------------------------------- greedy
__device__ __forceinline__ ArgPart arg_better(ArgPart a, ArgPart b) {
  if (a.idx < 0) return b;
  if (b.idx < 0) return a;
  if (a.v > b.v) return a;
  if (b.v > a.v) return b;
  return a.idx < b.idx ? a : b;
}

struct GreedyShared {
  int amax[kMaxNodes];
  int par[kMaxNodes];    // parents of the batch row's nodes (tree mode)
  int draft[kMaxNodes];  // its draft ids
  short depth[kMaxNodes];
  unsigned char ok[kMaxNodes];
};

template <bool VEC>
__global__ void __launch_bounds__(kAccThreads) accept_argmax_kernel(
    const float* __restrict__ p, const int32_t* __restrict__ d, const int32_t* __restrict__ parents, int n,
    int rows_per_b, int V, int chunk, ArgPart* __restrict__ parts, int* __restrict__ counters,
    int32_t* __restrict__ acc_out, int32_t* __restrict__ next_out, int32_t* __restrict__ node_out, unsigned* err,
    int64_t parts_cap) {
  grid_launch_dependents();
  grid_dependency_wait();
  const int rr = blockIdx.y;  // row index over all batch rows
  const int b = rr / rows_per_b;
  const float* row = p + (int64_t)rr * V;
  const int x0 = blockIdx.x * chunk, x1 = min(V, x0 + chunk);
  float v[kArgPT];
  load_chunk<VEC, kArgPT>(row, x0, x1, v);
  // this thread's indices increase with j (and within a float4), so a strict
  // comparison keeps the smallest index among equal values
  ArgPart best{-FLT_MAX, -1};
#pragma unroll
  for (int j = 0; j < kArgPT; ++j) {
    const int xi = VEC ? x0 + ((j / 4) * kAccThreads + (int)threadIdx.x) * 4 + (j % 4)
                       : x0 + j * kAccThreads + (int)threadIdx.x;
    if (xi < x1 && (v[j] > best.v || best.idx < 0)) best = ArgPart{v[j], xi};
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    ArgPart other;
    other.v = __shfl_xor_sync(0xffffffffu, best.v, o);
    other.idx = __shfl_xor_sync(0xffffffffu, best.idx, o);
    best = arg_better(best, other);
  }
  __shared__ ArgPart wbest[kAccWarps];
  __shared__ int last;
  if ((threadIdx.x & 31) == 0) wbest[threadIdx.x >> 5] = best;
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int i = 1; i < kAccWarps; ++i) best = arg_better(best, wbest[i]);
    const int64_t pi = (int64_t)rr * gridDim.x + blockIdx.x;
    if (in_bounds(err, pi, parts_cap)) parts[pi] = best;
    __threadfence();
    last = in_bounds(err, b, kCounterBank2) && atomicAdd(&counters[b], 1) == rows_per_b * (int)gridDim.x - 1;
  }
  __syncthreads();
  if (!last) return;
  __threadfence();

  __shared__ GreedyShared gs;
  // the row's draft ids (and parents) into shared memory with all threads:
  // the walk below then reads no global memory
  for (int j = threadIdx.x; j < n; j += kAccThreads) {
    gs.draft[j] = d[(int64_t)b * n + j];
    if (parents) gs.par[j] = parents[(int64_t)b * n + j];
  }
  for (int j = threadIdx.x; j < rows_per_b; j += kAccThreads) {
    const ArgPart* pp = parts + ((int64_t)b * rows_per_b + j) * gridDim.x;
    ArgPart a{-FLT_MAX, -1};
    for (int c = 0; c < (int)gridDim.x; ++c) {
      ArgPart w;
      w.v = __ldcg(&pp[c].v);
      w.idx = __ldcg(&pp[c].idx);
      a = arg_better(a, w);
    }
    gs.amax[j] = a.idx < 0 ? 0 : a.idx;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    counters[b] = 0;
    int acc = 0, best_node = 0;
    if (!parents) {  // chain: rows 0..n, drafts d_1..d_n
      acc = n;
      for (int i = 0; i < n; ++i) {
        const int di = gs.draft[i];
        if (di < 0 || di >= V) report_error(err, kErrInput);
        if (di != gs.amax[i]) {
          acc = i;
          break;
        }
      }
      best_node = acc;
    } else {  // tree: rows 0..n-1, node 0 is the root
      const int* par = gs.par;
      const int* dd = gs.draft;
      gs.depth[0] = 0;
      gs.ok[0] = 1;
      bool bad = par[0] != -1;
      for (int j = 1; j < n && !bad; ++j) {
        const int pj = par[j];
        if (pj < 0 || pj >= j) {
          bad = true;
          break;
        }
        const int dj = dd[j];
        if (dj < 0 || dj >= V) report_error(err, kErrInput);
        gs.depth[j] = (short)(gs.depth[pj] + 1);
        gs.ok[j] = (unsigned char)(gs.ok[pj] && dj == gs.amax[pj]);
        if (gs.ok[j] && gs.depth[j] > gs.depth[best_node]) best_node = j;
      }
      if (bad) {
        report_error(err, kErrInput);
        best_node = 0;
      }
      acc = gs.depth[best_node];
    }
    acc_out[b] = acc;
    next_out[b] = gs.amax[best_node];
    if (node_out) node_out[b] = best_node;
  }
}

// ------------------------------------------------- stochastic token tree
// Multi-step speculative sampling over a token tree (SpecInfer, section 4.2;
// the pages give the rule for a sequence draft only): at node u the
// children are tried in ascending index, child s with token x accepted iff
// u_s < min(1, R(x) / Q_u(x)); a rejection replaces R by the normalised
// max(0, R - Q_u); with no child left the next token is drawn from R.
// R after k rejections at u equals max(0, P_u - c_k Q_u) / T_k with
// c_0 = 0, T_0 = 1, c_{k+1} = c_k + T_k and T_{k+1} the sum of
// max(0, P_u - c_{k+1} Q_u) (induction on the update), so each rejection
// costs one vocabulary-wide sum.
//
// One cluster of kTreeCtas CTAs per batch row; CTA r holds logits
// [r kTreeSlice, (r + 1) kTreeSlice) of the visited node's target and draft
// rows in registers (kTreePT contiguous logits per thread), so every sum
// over the vocabulary is a register pass; partial results meet through
// distributed shared memory, each CTA adding the kTreeCtas partials in rank
// order (every CTA holds the same totals and takes the same decisions).
constexpr int kTreeCtas = 8;
constexpr int kTreeThreads = 512;
constexpr int kTreeWarps = kTreeThreads / 32;
constexpr int kTreePT = 32;
constexpr int kTreeSlice = kTreeThreads * kTreePT;  // 16384
static_assert(kTreeCtas * kTreeSlice == kAcceptTreeMaxV, "vocabulary limit of the cluster kernels");

struct TreeShared {
  int par[kMaxNodes];
  int draft[kMaxNodes];
  DF red[2][2];      // this CTA's partials for the cluster (double-buffered): two quantities
  DF warp_part[kTreeWarps][2];
  DF total[2];
  int found, last_pos;
};

__device__ __forceinline__ DF shfl_df(DF v, int src) {
  return DF{__shfl_sync(0xffffffffu, v.hi, src), __shfl_sync(0xffffffffu, v.lo, src)};
}

// Sum (kind 0) or max (kind 1, in .hi) of two values over the cluster.
template <int KIND>
__device__ void cluster_reduce2(cg::cluster_group& cluster, TreeShared& sh, int& phase, DF a, DF b, DF& ra, DF& rb) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    if (KIND == 0) {
      a = df_add(a, shfl_xor_df(a, o));
      b = df_add(b, shfl_xor_df(b, o));
    } else {
      a.hi = fmaxf(a.hi, __shfl_xor_sync(0xffffffffu, a.hi, o));
      b.hi = fmaxf(b.hi, __shfl_xor_sync(0xffffffffu, b.hi, o));
    }
  }
  if (lane == 0) {
    sh.warp_part[w][0] = a;
    sh.warp_part[w][1] = b;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    DF x = sh.warp_part[0][0], y = sh.warp_part[0][1];
    for (int i = 1; i < kTreeWarps; ++i) {
      if (KIND == 0) {
        x = df_add(x, sh.warp_part[i][0]);
        y = df_add(y, sh.warp_part[i][1]);
      } else {
        x.hi = fmaxf(x.hi, sh.warp_part[i][0].hi);
        y.hi = fmaxf(y.hi, sh.warp_part[i][1].hi);
      }
    }
    sh.red[phase][0] = x;
    sh.red[phase][1] = y;
  }
  cluster.sync();
  if (threadIdx.x < 32) {  // lane r fetches rank r's partials; lane 0 combines them in rank order
    DF ox{0.0f, 0.0f}, oy{0.0f, 0.0f};
    if (lane < kTreeCtas) {
      const TreeShared* o = cluster.map_shared_rank(&sh, lane);
      ox = o->red[phase][0];
      oy = o->red[phase][1];
    }
    DF x = KIND == 0 ? DF{0.0f, 0.0f} : DF{-FLT_MAX, 0.0f}, y = x;
#pragma unroll
    for (int r = 0; r < kTreeCtas; ++r) {
      const DF rx = shfl_df(ox, r), ry = shfl_df(oy, r);
      if (KIND == 0) {
        x = df_add(x, rx);
        y = df_add(y, ry);
      } else {
        x.hi = fmaxf(x.hi, rx.hi);
        y.hi = fmaxf(y.hi, ry.hi);
      }
    }
    if (lane == 0) {
      sh.total[0] = x;
      sh.total[1] = y;
    }
  }
  __syncthreads();
  ra = sh.total[0];
  rb = sh.total[1];
  __syncthreads();
  phase ^= 1;
}

// Inverse-CDF draw over the cluster's vocabulary slices: rv holds this
// thread's kTreePT values at x0, x0 + 1, ... (zero past V). The smallest x
// whose ascending running sum exceeds u * S (double-float sums: the thread's
// own run, the CTA's warps, the CTAs of lower rank); if rounding leaves no
// such x, the last x with positive mass. Returns the index in rank 0's
// thread 0; the caller writes its outputs there and synchronises the
// cluster once more before any CTA exits.
__device__ int cluster_draw(cg::cluster_group& cluster, TreeShared& sh, int phase, int rank, int x0, int V,
                            const float (&rv)[kTreePT], float uval) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  DF mine{0.0f, 0.0f};
  int lastp = -1;
#pragma unroll
  for (int k = 0; k < kTreePT; ++k) {
    if (rv[k] > 0.0f) lastp = x0 + k;
    mine = df_add_f(mine, rv[k]);
  }
  // this thread's exclusive prefix within the CTA, then the CTAs before it
  DF incl = mine;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const DF y{__shfl_up_sync(0xffffffffu, incl.hi, o), __shfl_up_sync(0xffffffffu, incl.lo, o)};
    if (lane >= o) incl = df_add(y, incl);
  }
  if (lane == 31) sh.warp_part[w][0] = incl;
  __syncthreads();
  DF before{0.0f, 0.0f};
  for (int i = 0; i < w; ++i) before = df_add(before, sh.warp_part[i][0]);
  DF cta_total{0.0f, 0.0f};
  for (int i = 0; i < kTreeWarps; ++i) cta_total = df_add(cta_total, sh.warp_part[i][0]);
  const DF excl_thread = df_add(before, df_add(incl, DF{-mine.hi, -mine.lo}));
  if (threadIdx.x == 0) {
    sh.red[phase][0] = cta_total;
    sh.found = INT_MAX;
    sh.last_pos = -1;
  }
  cluster.sync();
  if (threadIdx.x < 32) {  // lane r fetches rank r's total; the sums in rank order go to every thread
    const DF o = lane < kTreeCtas ? cluster.map_shared_rank(&sh, lane)->red[phase][0] : DF{0.0f, 0.0f};
    DF bl{0.0f, 0.0f}, tot{0.0f, 0.0f};
#pragma unroll
    for (int r = 0; r < kTreeCtas; ++r) {
      const DF x = shfl_df(o, r);
      if (r < rank) bl = df_add(bl, x);
      tot = df_add(tot, x);
    }
    if (lane == 0) {
      sh.total[0] = tot;
      sh.total[1] = bl;
    }
  }
  __syncthreads();
  const DF S = sh.total[0], below = sh.total[1];
  const DF tt = df_mul_f(S, uval);
  DF run = df_add(below, excl_thread);
  int hit = INT_MAX;
#pragma unroll
  for (int k = 0; k < kTreePT; ++k) {
    run = df_add_f(run, rv[k]);
    if (hit == INT_MAX && x0 + k < V && df_gt(run, tt)) hit = x0 + k;
  }
  // one shared-memory atomic per warp (512 threads on one address serialise)
  hit = __reduce_min_sync(0xffffffffu, hit);
  lastp = __reduce_max_sync(0xffffffffu, lastp);
  if (lane == 0) {
    if (hit != INT_MAX) atomicMin(&sh.found, hit);
    if (lastp >= 0) atomicMax(&sh.last_pos, lastp);
  }
  cluster.sync();  // every CTA's candidates are in
  int best = 0;
  if (rank == 0 && threadIdx.x == 0) {
    int found = INT_MAX, lastv = -1;
    for (int r = 0; r < kTreeCtas; ++r) {
      const TreeShared* o = cluster.map_shared_rank(&sh, r);
      found = min(found, o->found);
      lastv = max(lastv, o->last_pos);
    }
    best = found != INT_MAX ? found : (lastv >= 0 ? lastv : 0);
  }
  return best;
}

template <bool VEC>
__global__ void __cluster_dims__(kTreeCtas, 1, 1) __launch_bounds__(kTreeThreads, 1) accept_tree_kernel(
    const float* __restrict__ p, const float* __restrict__ q, const int32_t* __restrict__ d,
    const int32_t* __restrict__ parents, const float* __restrict__ u, int n, int V, int32_t* __restrict__ acc_out,
    int32_t* __restrict__ next_out, int32_t* __restrict__ node_out, unsigned* err) {
  grid_launch_dependents();
  grid_dependency_wait();
  cg::cluster_group cluster = cg::this_cluster();
  __shared__ TreeShared sh;
  const int rank = (int)cluster.block_rank();
  const int b = blockIdx.x / kTreeCtas;
  const int x0 = rank * kTreeSlice + (int)threadIdx.x * kTreePT;  // this thread's logits
  int phase = 0;
  for (int j = threadIdx.x; j < n; j += kTreeThreads) {
    int pj = parents[(int64_t)b * n + j];
    const int dj = d[(int64_t)b * n + j];
    if (j == 0 ? pj != -1 : (pj < 0 || pj >= j)) {
      if (rank == 0) report_error(err, kErrInput);
      pj = -2;  // never anyone's child
    }
    if (j > 0 && (dj < 0 || dj >= V)) {
      if (rank == 0) report_error(err, kErrInput);
      pj = -2;
    }
    sh.par[j] = pj;
    sh.draft[j] = dj;
  }
  __syncthreads();
  const float* ub = u + (int64_t)b * n;
  float lp[kTreePT], lq[kTreePT];
  int node = 0, depth = 0, s = 1;
  float mp = 0.0f, mq = 0.0f, izp = 0.0f, izq = 0.0f, c = 0.0f, T = 1.0f;
  bool load = true;
  for (;;) {
    if (load) {  // the node's rows into registers, their maxima and normalisers
      const float* prow = p + ((int64_t)b * n + node) * V;
      const float* qrow = q + ((int64_t)b * n + node) * V;
      if (VEC) {
#pragma unroll
        for (int k = 0; k < kTreePT; k += 4) {
          float4 a = make_float4(-FLT_MAX, -FLT_MAX, -FLT_MAX, -FLT_MAX), e = a;
          if (x0 + k < V) {
            a = ldg_stream_f4(reinterpret_cast<const float4*>(prow + x0 + k));
            e = ldg_stream_f4(reinterpret_cast<const float4*>(qrow + x0 + k));
          }
          lp[k] = a.x, lp[k + 1] = a.y, lp[k + 2] = a.z, lp[k + 3] = a.w;
          lq[k] = e.x, lq[k + 1] = e.y, lq[k + 2] = e.z, lq[k + 3] = e.w;
        }
      } else {
#pragma unroll
        for (int k = 0; k < kTreePT; ++k) {
          lp[k] = x0 + k < V ? ldg_stream_f(prow + x0 + k) : -FLT_MAX;
          lq[k] = x0 + k < V ? ldg_stream_f(qrow + x0 + k) : -FLT_MAX;
        }
      }
      float a = -FLT_MAX, e = -FLT_MAX;
#pragma unroll
      for (int k = 0; k < kTreePT; ++k) {
        a = fmaxf(a, lp[k]);
        e = fmaxf(e, lq[k]);
      }
      DF M1, M2;
      cluster_reduce2<1>(cluster, sh, phase, DF{a, 0.0f}, DF{e, 0.0f}, M1, M2);
      mp = M1.hi;
      mq = M2.hi;
      // the registers now hold exp(l - max), then the probabilities
      DF zp{0.0f, 0.0f}, zq{0.0f, 0.0f};
#pragma unroll
      for (int k = 0; k < kTreePT; ++k) {
        const bool in = x0 + k < V;
        lp[k] = in ? exp_of_diff(lp[k], mp) : 0.0f;
        lq[k] = in ? exp_of_diff(lq[k], mq) : 0.0f;
        zp = df_add_f(zp, lp[k]);
        zq = df_add_f(zq, lq[k]);
      }
      DF Zp, Zq;
      cluster_reduce2<0>(cluster, sh, phase, zp, zq, Zp, Zq);
      izp = __frcp_rn(df_val(Zp));
      izq = __frcp_rn(df_val(Zq));
#pragma unroll
      for (int k = 0; k < kTreePT; ++k) {
        lp[k] = __fmul_rn(lp[k], izp);
        lq[k] = __fmul_rn(lq[k], izq);
      }
      c = 0.0f;
      T = 1.0f;
      s = node + 1;
      load = false;
    }
    while (s < n && sh.par[s] != node) ++s;  // the node's next child
    if (s >= n) break;
    // the child's test (every thread of the cluster computes the same value)
    const int x = sh.draft[s];
    const float px = __fmul_rn(exp_of_diff(__ldg(p + ((int64_t)b * n + node) * V + x), mp), izp);
    const float qx = __fmul_rn(exp_of_diff(__ldg(q + ((int64_t)b * n + node) * V + x), mq), izq);
    const float rx = fmaxf(__fsub_rn(px, __fmul_rn(c, qx)), 0.0f);
    const float alpha = qx > 0.0f ? fminf(1.0f, __fdiv_rn(__fdiv_rn(rx, T), qx)) : 1.0f;
    if (ub[s] < alpha) {
      node = s;
      ++depth;
      load = true;
      continue;
    }
    // rejected: R <- max(0, P - c' Q) / T' with c' = c + T
    const float c1 = __fadd_rn(c, T);
    DF t{0.0f, 0.0f};
#pragma unroll
    for (int k = 0; k < kTreePT; ++k) t = df_add_f(t, fmaxf(__fsub_rn(lp[k], __fmul_rn(c1, lq[k])), 0.0f));
    DF T1, unused;
    cluster_reduce2<0>(cluster, sh, phase, t, DF{0.0f, 0.0f}, T1, unused);
    const float tv = df_val(T1);
    if (tv > 0.0f) {  // else the residual keeps its previous value
      c = c1;
      T = tv;
    }
    ++s;
  }
  // ---- the next token: inverse CDF of r(x) = max(0, P - c Q) (P itself when c = 0), ascending x
  float rv[kTreePT];
#pragma unroll
  for (int k = 0; k < kTreePT; ++k) rv[k] = c == 0.0f ? lp[k] : fmaxf(__fsub_rn(lp[k], __fmul_rn(c, lq[k])), 0.0f);
  const int best = cluster_draw(cluster, sh, phase, rank, x0, V, rv, ub[0]);
  if (rank == 0 && threadIdx.x == 0) {
    acc_out[b] = depth;
    next_out[b] = best;
    if (node_out) node_out[b] = node;
  }
  cluster.sync();  // no CTA leaves while rank 0 may still read its shared memory
}

cudaError_t launch_accept_tree(const float* p, const float* q, const int32_t* d, const int32_t* parents,
                               const float* u, int B, int n, int V, int32_t* acc, int32_t* next, int32_t* node,
                               unsigned* err, cudaStream_t stream) {
  if (V % 4 == 0)
    return launch_pdl(accept_tree_kernel<true>, dim3((unsigned)(B * kTreeCtas)), dim3(kTreeThreads), 0, stream, p, q,
                      d, parents, u, n, V, acc, next, node, err);
  return launch_pdl(accept_tree_kernel<false>, dim3((unsigned)(B * kTreeCtas)), dim3(kTreeThreads), 0, stream, p, q,
                    d, parents, u, n, V, acc, next, node, err);
}

// ------------------------------------------------------------------ host
static inline size_t align256(size_t v) { return (v + 255) / 256 * 256; }

AcceptPlan accept_plan(int B, int n, int V) {
  AcceptPlan pl;
  const int rows = B * (2 * n + 1);  // upper bound over modes (greedy reads B*(n+1) or B*n rows)
  pl.rows = rows;
  pl.rows_seq = rows;
  // statistics items: chunks of kStatItem logits
  const int ch = (V + kStatItem - 1) / kStatItem;
  pl.ch = ch;
  pl.chunk = kStatItem;
  // argmax chunks (greedy modes): at most kArgChunk logits, about 1024
  // blocks in all, at most 64 per row, at least ~2048 logits each
  int cha = (V + kArgChunk - 1) / kArgChunk;
  const int want = (1024 + rows - 1) / rows;
  const int cap_v = (V + 2047) / 2048;
  int more = want < cap_v ? want : cap_v;
  if (more > 64) more = 64;
  if (cha < more) cha = more;
  int chunka = (V + cha - 1) / cha;
  chunka = (chunka + 3) / 4 * 4;
  if (chunka > kArgChunk) chunka = kArgChunk;
  cha = (V + chunka - 1) / chunka;
  pl.cha = cha;
  pl.chunka = chunka;
  // residual chunks per batch row: the launch picks ch2 in [lo, hi] so the
  // grid fits the resident blocks (one wave); the workspace holds hi
  const int lo = (V + kMaxChunk2 - 1) / kMaxChunk2;  // <= kMaxCh2 for V <= 2^20
  int hi = (V + kMinChunk2 - 1) / kMinChunk2;
  if (hi > kMaxCh2) hi = kMaxCh2;
  if (hi < lo) hi = lo;
  pl.ch2_lo = lo;
  pl.ch2 = hi;
  pl.chunk2 = (V + hi - 1) / hi;
  size_t stats_bytes = align256((size_t)rows * ch * sizeof(RowStat));
  const size_t parts_bytes = align256((size_t)rows * cha * sizeof(ArgPart));
  if (parts_bytes > stats_bytes) stats_bytes = parts_bytes;
  const size_t dec_bytes = align256((size_t)B * sizeof(Decision));
  const size_t csum_bytes = align256((size_t)B * hi * sizeof(ChunkSum));
  pl.stats_off = kCounterRegionBytes;
  pl.dec_off = pl.stats_off + stats_bytes;
  pl.csum_off = pl.dec_off + dec_bytes;
  pl.total = pl.csum_off + csum_bytes;
  return pl;
}

cudaError_t launch_accept_seq(const float* p, const float* q, const int32_t* d, const float* u, int B, int n, int V,
                              int32_t* acc, int32_t* next, void* ws, const AcceptPlan& pl, int num_sms, unsigned* err,
                              cudaStream_t stream, const float2* p_stats, int32_t* node) {
  uint8_t* w = static_cast<uint8_t*>(ws);
  RowStat* stats = reinterpret_cast<RowStat*>(w + pl.stats_off);
  Decision* dec = reinterpret_cast<Decision*>(w + pl.dec_off);
  ChunkSum* csum = reinterpret_cast<ChunkSum*>(w + pl.csum_off);
  int* cnt2 = reinterpret_cast<int*>(w) + kCounterBank2;
  const int64_t stats_cap = (int64_t)((pl.dec_off - pl.stats_off) / sizeof(RowStat));
  const int64_t csum_cap = (int64_t)((pl.total - pl.csum_off) / sizeof(ChunkSum));
  cudaError_t e;
  // statistics grid: persistent warps, one wave of resident blocks (the
  // kernel's launch bounds give two per SM); with the target statistics
  // supplied, the draft rows only
  const int q_only = p_stats ? 1 : 0;
  const int items = (q_only ? B * n : pl.rows_seq) * pl.ch;
  // supplied target statistics: V / 32 slices a row, kSliceItem an item
  const int chs = q_only ? (V / 32 + kSliceItem - 1) / kSliceItem : 0;
  const int slice_items = B * (n + 1) * chs;  // fits: chs <= ch, so the total stays within rows_seq * ch
  int g1 = (items + slice_items + kAccWarps - 1) / kAccWarps;
  if (g1 > kStatBlocksPerSm * num_sms) g1 = kStatBlocksPerSm * num_sms;
  if (V % 4 == 0)
    e = launch_pdl(accept_stats_kernel<true>, dim3(g1), dim3(kAccThreads), 0, stream, p, q, n, V, pl.ch, items, q_only,
                   p_stats, chs, slice_items, stats, stats_cap, err);
  else
    e = launch_pdl(accept_stats_kernel<false>, dim3(g1), dim3(kAccThreads), 0, stream, p, q, n, V, pl.ch, items, q_only,
                   p_stats, chs, slice_items, stats, stats_cap, err);
  if (e != cudaSuccess) return e;
  e = launch_pdl(accept_decide_kernel, dim3(B), dim3(kDecThreads), 0, stream, p, q, d, u, n, V, pl.ch,
                 (const RowStat*)stats, q_only, chs, dec, err);
  if (e != cudaSuccess) return e;
  // residual grid: as many chunks per batch row as one wave of resident
  // blocks allows, within [ch2_lo, ch2]
  static std::atomic<int> resid_per_sm{0};
  int per_sm = resid_per_sm.load(std::memory_order_relaxed);
  if (per_sm == 0) {
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, accept_resid_kernel<kResidPT, true>, kAccThreads, 0);
    if (e != cudaSuccess) return e;
    if (per_sm < 1) per_sm = 1;
    resid_per_sm.store(per_sm, std::memory_order_relaxed);
  }
  int ch2 = (int)(((int64_t)per_sm * num_sms) / B);
  if (ch2 > pl.ch2) ch2 = pl.ch2;
  if (ch2 < pl.ch2_lo) ch2 = pl.ch2_lo;
  int chunk2 = (V + ch2 - 1) / ch2;
  if (V % 4 == 0) chunk2 = (chunk2 + 3) / 4 * 4;  // whole float4s (still <= kMaxChunk2)
  ch2 = (V + chunk2 - 1) / chunk2;
  if (V % 4 == 0)
    return launch_pdl(accept_resid_kernel<kResidPT, true>, dim3(ch2, B), dim3(kAccThreads), 0, stream, p, q, u, n, V,
                      chunk2, (const Decision*)dec, csum, cnt2, acc, next, node, csum_cap, err);
  return launch_pdl(accept_resid_kernel<kResidPT, false>, dim3(ch2, B), dim3(kAccThreads), 0, stream, p, q, u, n, V,
                    chunk2, (const Decision*)dec, csum, cnt2, acc, next, node, csum_cap, err);
}

cudaError_t launch_accept_greedy(const float* p, const int32_t* d, const int32_t* parents, int B, int n, int V,
                                 int32_t* acc, int32_t* next, void* ws, const AcceptPlan& pl, unsigned* err,
                                 cudaStream_t stream, int32_t* node) {
  uint8_t* w = static_cast<uint8_t*>(ws);
  ArgPart* parts = reinterpret_cast<ArgPart*>(w + pl.stats_off);
  int* cnt = reinterpret_cast<int*>(w);
  const int rows_per_b = parents ? n : n + 1;
  const dim3 g(pl.cha, B * rows_per_b);
  const int64_t parts_cap = (int64_t)((pl.dec_off - pl.stats_off) / sizeof(ArgPart));
  if (V % 4 == 0)
    return launch_pdl(accept_argmax_kernel<true>, g, dim3(kAccThreads), 0, stream, p, d, parents, n, rows_per_b, V,
                      pl.chunka, parts, cnt, acc, next, node, err, parts_cap);
  return launch_pdl(accept_argmax_kernel<false>, g, dim3(kAccThreads), 0, stream, p, d, parents, n, rows_per_b, V,
                    pl.chunka, parts, cnt, acc, next, node, err, parts_cap);
}

}  // namespace w4a16
