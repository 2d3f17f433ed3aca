// Speculative accept step ("Speculative Decoding이란?", section 3 Steps 3-4,
// section 6; greedy equivalence in section 5).
//
// Stochastic sequence mode, two launches:
//  1. accept_stats_kernel: every p / q logit row is cut into chunks; a block
//     reduces one chunk to (max, sum of exp(l - max)) — one HBM pass over
//     all logits, fp32 exponentials, per-thread fp32 sums folded into fp64.
//  2. accept_resid_kernel, grid (chunk, batch row): each block merges the
//     row statistics of its batch row, evaluates alpha_i = min(1, P/Q) for
//     the drafts (fp64), finds the first rejection r, then sums the corrected
//     distribution max(0, P_r - Q_r) (or P_{n+1} after full acceptance) over
//     its vocabulary chunk. The last block of the batch row (atomic count)
//     walks the chunk sums, re-scans the one chunk that holds u * S, and
//     writes accepted_len and next_token.
// Greedy modes, one launch: accept_argmax_kernel reduces chunks to
// (max, smallest index); the last block of a batch row merges them and walks
// the chain or tree.
//
// Every per-element value that decides a draw (P, Q, max(0, P - Q)) is formed
// with explicit rn intrinsics so that the block that sums a chunk and the
// block that re-scans it compute bit-identical values.
#include <float.h>

#include "common.cuh"
#include "internal.h"

namespace w4a16 {

constexpr int kAccThreads = 256;
constexpr int kAccWarps = kAccThreads / 32;
constexpr int kMaxNodes = 1025;  // rows of one batch element in greedy mode (n <= 1024)

struct RowStat {
  float m;
  float pad;
  double s;
};

struct ChunkSum {
  double r;  // sum of the distribution being sampled
  double p;  // sum of P_r (fallback when the corrected distribution is all zero)
};

struct ArgPart {
  float v;
  int idx;
};

__device__ __forceinline__ void merge_stat(float& m, double& s, float m2, double s2) {
  if (s2 == 0.0 && m2 == -FLT_MAX) return;
  if (m2 > m) {
    s = s * (double)expf(m - m2) + s2;
    m = m2;
  } else {
    s += s2 * (double)expf(m2 - m);
  }
}

// Block-wide merge of (max, sum-of-exp) pairs; result valid in thread 0.
__device__ void block_merge_stat(float& m, double& s) {
  __shared__ float sm_m[kAccWarps];
  __shared__ double sm_s[kAccWarps];
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float m2 = __shfl_xor_sync(0xffffffffu, m, o);
    const double s2 = __shfl_xor_sync(0xffffffffu, s, o);
    merge_stat(m, s, m2, s2);
  }
  if (lane == 0) {
    sm_m[w] = m;
    sm_s[w] = s;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int i = 1; i < kAccWarps; ++i) merge_stat(m, s, sm_m[i], sm_s[i]);
  }
  __syncthreads();
}

__device__ __forceinline__ double block_sum_double(double v) {
  __shared__ double sm[kAccWarps];
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  if (lane == 0) sm[w] = v;
  __syncthreads();
  double t = 0.0;
  if (threadIdx.x == 0)
    for (int i = 0; i < kAccWarps; ++i) t += sm[i];
  __syncthreads();
  return t;  // valid in thread 0
}

// Row pointer for statistics row rr: batch b's n+1 target rows, then its n draft rows.
__device__ __forceinline__ const float* stat_row_ptr(const float* p, const float* q, int n, int64_t V, int rr) {
  const int per = 2 * n + 1;
  const int b = rr / per, i = rr % per;
  if (i <= n) return p + ((int64_t)b * (n + 1) + i) * V;
  return q + ((int64_t)b * n + (i - n - 1)) * V;
}

// ------------------------------------------------------- pass 1: row stats
template <bool VEC>
__global__ void __launch_bounds__(kAccThreads) accept_stats_kernel(const float* __restrict__ p,
                                                                   const float* __restrict__ q, int n, int V,
                                                                   int chunk, RowStat* __restrict__ stats) {
  const int rr = blockIdx.y;
  const float* row = stat_row_ptr(p, q, n, V, rr);
  const int x0 = blockIdx.x * chunk;
  const int x1 = min(V, x0 + chunk);
  float m = -FLT_MAX;
  double s = 0.0;
  if (VEC) {
    constexpr int U = 4;
    for (int base = x0 + threadIdx.x * 4; base < x1; base += kAccThreads * 4 * U) {
      float4 v[U];
      float bm = -FLT_MAX;
#pragma unroll
      for (int k = 0; k < U; ++k) {
        const int xi = base + k * kAccThreads * 4;
        if (xi < x1) {
          v[k] = ldg_stream_f4(reinterpret_cast<const float4*>(row + xi));
          bm = fmaxf(bm, fmaxf(fmaxf(v[k].x, v[k].y), fmaxf(v[k].z, v[k].w)));
        } else {
          v[k] = make_float4(-FLT_MAX, -FLT_MAX, -FLT_MAX, -FLT_MAX);
        }
      }
      if (bm > m) {
        if (s != 0.0) s *= (double)expf(m - bm);
        m = bm;
      }
      float fs = 0.0f;
#pragma unroll
      for (int k = 0; k < U; ++k)
        if (base + k * kAccThreads * 4 < x1)
          fs += (expf(v[k].x - m) + expf(v[k].y - m)) + (expf(v[k].z - m) + expf(v[k].w - m));
      s += (double)fs;
    }
  } else {
    for (int xi = x0 + threadIdx.x; xi < x1; xi += kAccThreads) {
      const float v = ldg_stream_f(row + xi);
      if (v > m) {
        if (s != 0.0) s *= (double)expf(m - v);
        m = v;
      }
      s += (double)expf(v - m);
    }
  }
  block_merge_stat(m, s);
  if (threadIdx.x == 0) {
    RowStat r;
    r.m = m;
    r.pad = 0.0f;
    r.s = s;
    stats[(int64_t)rr * gridDim.x + blockIdx.x] = r;
  }
}

// --------------------------------------- pass 2: decide, residual, sample
struct SeqShared {
  float mp[kMaxNodes];
  double zp[kMaxNodes];
  float mq[kMaxNodes];
  double zq[kMaxNodes];
  int reject[kMaxNodes];
  int r;
};

// Value of the distribution being sampled at x (bit-identical wherever computed).
struct ResidFn {
  const float* prow;  // P_r row logits (or P_{n+1} after full acceptance)
  const float* qrow;  // Q_r row logits, NULL after full acceptance
  float mp, ip, mq, iq;
  __device__ __forceinline__ float pval(int x) const { return __fmul_rn(expf(__fsub_rn(prow[x], mp)), ip); }
  __device__ __forceinline__ float rval(int x) const {
    const float pv = pval(x);
    if (!qrow) return pv;
    const float qv = __fmul_rn(expf(__fsub_rn(qrow[x], mq)), iq);
    return fmaxf(__fsub_rn(pv, qv), 0.0f);
  }
};

__global__ void __launch_bounds__(kAccThreads) accept_resid_kernel(
    const float* __restrict__ p, const float* __restrict__ q, const int32_t* __restrict__ d,
    const float* __restrict__ u, int n, int V, int ch, int chunk2, const RowStat* __restrict__ stats,
    ChunkSum* __restrict__ csum, int* __restrict__ counters, int32_t* __restrict__ acc_out,
    int32_t* __restrict__ next_out, unsigned* err) {
  __shared__ SeqShared sh;
  const int b = blockIdx.y;
  const int per = 2 * n + 1;
  // merge the chunk statistics of this batch row's 2n+1 rows
  for (int i = threadIdx.x; i < per; i += kAccThreads) {
    const RowStat* st = stats + ((int64_t)b * per + i) * ch;
    float m = -FLT_MAX;
    double s = 0.0;
    for (int c = 0; c < ch; ++c) merge_stat(m, s, st[c].m, st[c].s);
    if (i <= n) {
      sh.mp[i] = m;
      sh.zp[i] = s;
    } else {
      sh.mq[i - n - 1] = m;
      sh.zq[i - n - 1] = s;
    }
  }
  __syncthreads();
  // acceptance test for each draft position (in parallel), first rejection after
  for (int i = threadIdx.x; i < n; i += kAccThreads) {
    const int di = d[(int64_t)b * n + i];
    int rej;
    if (di < 0 || di >= V) {
      report_error(err, kErrInput);
      rej = 1;
    } else {
      const double ep = (double)expf(__fsub_rn(p[((int64_t)b * (n + 1) + i) * V + di], sh.mp[i]));
      const double eq = (double)expf(__fsub_rn(q[((int64_t)b * n + i) * V + di], sh.mq[i]));
      const double P = ep / sh.zp[i], Q = eq / sh.zq[i];
      const double alpha = Q > 0.0 ? fmin(1.0, P / Q) : 1.0;
      rej = ((double)u[(int64_t)b * (n + 1) + i] < alpha) ? 0 : 1;
    }
    sh.reject[i] = rej;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    int r = n;
    for (int i = 0; i < n; ++i)
      if (sh.reject[i]) {
        r = i;
        break;
      }
    sh.r = r;
  }
  __syncthreads();
  const int r = sh.r;
  ResidFn f;
  f.prow = p + ((int64_t)b * (n + 1) + r) * V;
  f.mp = sh.mp[r];
  f.ip = (float)(1.0 / sh.zp[r]);
  if (r < n) {
    f.qrow = q + ((int64_t)b * n + r) * V;
    f.mq = sh.mq[r];
    f.iq = (float)(1.0 / sh.zq[r]);
  } else {
    f.qrow = nullptr;
    f.mq = 0.0f;
    f.iq = 0.0f;
  }
  // this block's chunk sums
  const int x0 = blockIdx.x * chunk2, x1 = min(V, x0 + chunk2);
  double sr = 0.0, sp = 0.0;
  for (int x = x0 + threadIdx.x; x < x1; x += kAccThreads) {
    sr += (double)f.rval(x);
    if (f.qrow) sp += (double)f.pval(x);
  }
  sr = block_sum_double(sr);
  sp = block_sum_double(sp);
  __shared__ int last;
  if (threadIdx.x == 0) {
    csum[(int64_t)b * gridDim.x + blockIdx.x] = ChunkSum{sr, sp};
    __threadfence();
    const int old = atomicAdd(&counters[b], 1);
    last = (old == (int)gridDim.x - 1);
  }
  __syncthreads();
  if (!last) return;
  __threadfence();

  // ---- the last block of batch row b draws the next token
  __shared__ double sh_t, sh_before;
  __shared__ int sh_chunk, sh_usep;
  __shared__ ChunkSum sh_cs[64];  // gridDim.x <= 64
  for (int c = threadIdx.x; c < (int)gridDim.x; c += kAccThreads) {
    const ChunkSum* cs = csum + (int64_t)b * gridDim.x + c;
    sh_cs[c].r = __ldcg(&cs->r);
    sh_cs[c].p = __ldcg(&cs->p);
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    double S = 0.0;
    for (int c = 0; c < (int)gridDim.x; ++c) S += sh_cs[c].r;
    int usep = 0;
    if (f.qrow && S == 0.0) {  // corrected distribution is all zero: draw from P_r
      usep = 1;
      S = 0.0;
      for (int c = 0; c < (int)gridDim.x; ++c) S += sh_cs[c].p;
    }
    const double t = (double)u[(int64_t)b * (n + 1) + n] * S;
    double cum = 0.0;
    int cstar = -1;
    for (int c = 0; c < (int)gridDim.x; ++c) {
      const double v = usep ? sh_cs[c].p : sh_cs[c].r;
      if (cum + v > t) {
        cstar = c;
        break;
      }
      cum += v;
    }
    sh_t = t;
    sh_before = cum;
    sh_chunk = cstar;
    sh_usep = usep;
    counters[b] = 0;
  }
  __syncthreads();
  const int usep = sh_usep;
  auto val = [&](int x) { return usep ? f.pval(x) : f.rval(x); };
  int found = INT_MAX;
  if (sh_chunk >= 0) {
    // contiguous sub-range per thread, exclusive scan of thread sums (fp64)
    const int c0 = sh_chunk * chunk2, c1 = min(V, c0 + chunk2);
    const int len = c1 - c0;
    const int per_t = (len + kAccThreads - 1) / kAccThreads;
    const int a0 = c0 + threadIdx.x * per_t, a1 = min(c1, a0 + per_t);
    double mine = 0.0;
    for (int x = a0; x < a1; ++x) mine += (double)val(x);
    __shared__ double scan[kAccThreads];
    scan[threadIdx.x] = mine;
    __syncthreads();
    if (threadIdx.x == 0) {
      double run = sh_before;
      for (int i = 0; i < kAccThreads; ++i) {
        const double v = scan[i];
        scan[i] = run;
        run += v;
      }
    }
    __syncthreads();
    double run = scan[threadIdx.x];
    for (int x = a0; x < a1; ++x) {
      run += (double)val(x);
      if (run > sh_t) {
        found = x;
        break;
      }
    }
  }
  // smallest crossing index in the block
  __shared__ int sh_found;
  if (threadIdx.x == 0) sh_found = INT_MAX;
  __syncthreads();
  if (found != INT_MAX) atomicMin(&sh_found, found);
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
  short depth[kMaxNodes];
  unsigned char ok[kMaxNodes];
};

template <bool VEC>
__global__ void __launch_bounds__(kAccThreads) accept_argmax_kernel(
    const float* __restrict__ p, const int32_t* __restrict__ d, const int32_t* __restrict__ parents, int n,
    int rows_per_b, int V, int chunk, ArgPart* __restrict__ parts, int* __restrict__ counters,
    int32_t* __restrict__ acc_out, int32_t* __restrict__ next_out, unsigned* err) {
  const int rr = blockIdx.y;  // row index over all batch rows
  const int b = rr / rows_per_b;
  const float* row = p + (int64_t)rr * V;
  const int x0 = blockIdx.x * chunk, x1 = min(V, x0 + chunk);
  ArgPart best{-FLT_MAX, -1};
  if (VEC) {
    for (int base = x0 + threadIdx.x * 4; base < x1; base += kAccThreads * 4) {
      const float4 v = ldg_stream_f4(reinterpret_cast<const float4*>(row + base));
      if (v.x > best.v || best.idx < 0) best = ArgPart{v.x, base};
      if (v.y > best.v) best = ArgPart{v.y, base + 1};
      if (v.z > best.v) best = ArgPart{v.z, base + 2};
      if (v.w > best.v) best = ArgPart{v.w, base + 3};
    }
  } else {
    for (int x = x0 + threadIdx.x; x < x1; x += kAccThreads) {
      const float v = ldg_stream_f(row + x);
      if (v > best.v || best.idx < 0) best = ArgPart{v, x};
    }
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
    parts[(int64_t)rr * gridDim.x + blockIdx.x] = best;
    __threadfence();
    const int old = atomicAdd(&counters[b], 1);
    last = (old == rows_per_b * (int)gridDim.x - 1);
  }
  __syncthreads();
  if (!last) return;
  __threadfence();

  __shared__ GreedyShared gs;
  for (int j = threadIdx.x; j < rows_per_b; j += kAccThreads) {
    const ArgPart* pp = parts + ((int64_t)b * rows_per_b + j) * gridDim.x;
    ArgPart a{-FLT_MAX, -1};
    for (int c = 0; c < (int)gridDim.x; ++c) {
      ArgPart v;
      v.v = __ldcg(&pp[c].v);
      v.idx = __ldcg(&pp[c].idx);
      a = arg_better(a, v);
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
        const int di = d[(int64_t)b * n + i];
        if (di < 0 || di >= V) report_error(err, kErrInput);
        if (di != gs.amax[i]) {
          acc = i;
          break;
        }
      }
      best_node = acc;
    } else {  // tree: rows 0..n-1, node 0 is the root
      const int32_t* par = parents + (int64_t)b * n;
      const int32_t* dd = d + (int64_t)b * n;
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
  }
}

// ------------------------------------------------------------------ host
static inline size_t align256(size_t v) { return (v + 255) / 256 * 256; }

AcceptPlan accept_plan(int B, int n, int V) {
  AcceptPlan pl;
  const int rows = B * (2 * n + 1);  // upper bound over modes (greedy reads B*(n+1) or B*n rows)
  pl.rows = rows;
  int ch = (1024 + rows - 1) / rows;
  const int max_ch_v = V / 2048 > 1 ? V / 2048 : 1;
  ch = ch < 1 ? 1 : ch;
  ch = ch > 64 ? 64 : ch;
  ch = ch > max_ch_v ? max_ch_v : ch;
  int chunk = (V + ch - 1) / ch;
  chunk = (chunk + 3) / 4 * 4;
  ch = (V + chunk - 1) / chunk;
  pl.ch = ch;
  pl.chunk = chunk;
  int ch2 = (1024 + B - 1) / B;
  ch2 = ch2 > 64 ? 64 : ch2;
  ch2 = ch2 > max_ch_v ? max_ch_v : ch2;
  ch2 = ch2 < 1 ? 1 : ch2;
  int chunk2 = (V + ch2 - 1) / ch2;
  ch2 = (V + chunk2 - 1) / chunk2;
  pl.ch2 = ch2;
  pl.chunk2 = chunk2;
  const size_t stats_bytes = align256((size_t)rows * ch * (sizeof(RowStat) > sizeof(ArgPart) ? sizeof(RowStat)
                                                                                              : sizeof(ArgPart)));
  const size_t csum_bytes = align256((size_t)B * ch2 * sizeof(ChunkSum));
  pl.stats_off = kCounterRegionBytes;
  pl.csum_off = pl.stats_off + stats_bytes;
  pl.total = pl.csum_off + csum_bytes;
  return pl;
}

cudaError_t launch_accept_seq(const float* p, const float* q, const int32_t* d, const float* u, int B, int n, int V,
                              int32_t* acc, int32_t* next, void* ws, const AcceptPlan& pl, unsigned* err,
                              cudaStream_t stream) {
  uint8_t* w = static_cast<uint8_t*>(ws);
  RowStat* stats = reinterpret_cast<RowStat*>(w + pl.stats_off);
  ChunkSum* csum = reinterpret_cast<ChunkSum*>(w + pl.csum_off);
  int* cnt = reinterpret_cast<int*>(w);
  const dim3 g1(pl.ch, B * (2 * n + 1));
  if (V % 4 == 0)
    accept_stats_kernel<true><<<g1, kAccThreads, 0, stream>>>(p, q, n, V, pl.chunk, stats);
  else
    accept_stats_kernel<false><<<g1, kAccThreads, 0, stream>>>(p, q, n, V, pl.chunk, stats);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const dim3 g2(pl.ch2, B);
  accept_resid_kernel<<<g2, kAccThreads, 0, stream>>>(p, q, d, u, n, V, pl.ch, pl.chunk2, stats, csum, cnt, acc,
                                                       next, err);
  return cudaGetLastError();
}

cudaError_t launch_accept_greedy(const float* p, const int32_t* d, const int32_t* parents, int B, int n, int V,
                                 int32_t* acc, int32_t* next, void* ws, const AcceptPlan& pl, unsigned* err,
                                 cudaStream_t stream) {
  uint8_t* w = static_cast<uint8_t*>(ws);
  ArgPart* parts = reinterpret_cast<ArgPart*>(w + pl.stats_off);
  int* cnt = reinterpret_cast<int*>(w);
  const int rows_per_b = parents ? n : n + 1;
  const dim3 g(pl.ch, B * rows_per_b);
  if (V % 4 == 0)
    accept_argmax_kernel<true><<<g, kAccThreads, 0, stream>>>(p, d, parents, n, rows_per_b, V, pl.chunk, parts, cnt,
                                                               acc, next, err);
  else
    accept_argmax_kernel<false><<<g, kAccThreads, 0, stream>>>(p, d, parents, n, rows_per_b, V, pl.chunk, parts,
                                                                cnt, acc, next, err);
  return cudaGetLastError();
}

}  // namespace w4a16
