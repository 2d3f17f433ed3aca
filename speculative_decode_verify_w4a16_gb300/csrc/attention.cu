// Tree-masked attention of the verify pass and compaction of the accepted
// path's keys and values ("Speculative Decoding이란?", section 10.1: Medusa's
// tree-based attention checks all candidate continuations of a token tree in
// one target pass; section 10.4: ReDrafter's dynamic tree attention; section
// 8.7: how a serving stack reuses the KV cache across accepted and rejected
// tokens).
//
// tree_attention_tc_kernel: the query rows of a KV head are its G = H / Hkv
// query heads at every tree node, row r = node * G + head-in-group, in tiles
// of 128 (the tcgen05 MMA's M). S = Q K^T and O += P V run on the tensor
// cores with S, P and O in tensor memory; the keys and values stream through
// a shared-memory ring of 64-key blocks (2-D TMA, 128-byte swizzle). Each row
// is masked (the committed prefix: every key; the tree's own keys: the node's
// ancestors and itself, a 64-bit mask per node), keeps the running maximum
// and sum of the online softmax in the log2 domain (the sum over the fp32
// weights), and accumulates P V with P rounded to bf16. With one
// piece per sequence the rows are normalised and stored as bf16; a sequence
// cut into several pieces (CTAs) leaves fp32 (m, l, O) per piece and
// tree_attention_combine_kernel merges them.
//
// kv_compact_kernel: per (batch row, layer), the keys and values of the
// accepted root path move to the positions right after the committed prefix.
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <float.h>
#include <math.h>

#include "common.cuh"
#include "internal.h"
#include "tcgen05.cuh"

namespace w4a16 {

constexpr int kAttD = 128;                     // head width
constexpr int kAttKeys = 64;                   // keys per block
constexpr int kAttMaxNodes = 64;

struct AttnParams {
  const __nv_bfloat16* q;  // [B][n][H][D]
  const int32_t* lens;     // [B]
  const int32_t* parents;  // [B][n] or null (chain)
  __nv_bfloat16* out;      // [B][n][H][D]
  float* part_o;           // cut: [ctas][unit_rows][D] unnormalised sums, one slot per piece
  float2* part_ml;         // and [ctas][unit_rows] (running max, sum), log2 domain
  unsigned* err;
  int B, n, H, Hkv, G, Lcap, max_len;
  int rows;        // n * G query rows per KV head
  int unit_rows;   // query rows per CTA: 128 * tiles
  int row_blocks;  // CTAs along the rows of a KV head
  int ctas;        // CTAs the pieces are cut for (one wave)
  int pieces_max;  // grid size: max(ctas, B * Hkv * row_blocks)
  int cut;         // 1: sequences may be cut into several pieces (partials and the combine)
  int2* seq_pieces;  // cut: per sequence (first piece, pieces)
  float scale_log2;  // softmax scale * log2(e)
};

// 2^x by the hardware approximation (a few ulp; 2^-inf = 0)
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
// two fp32 lanes in one 64-bit register (low half = first), for the paired
// fp32 instructions of sm_100 and later
__device__ __forceinline__ uint64_t f2_pack(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void f2_unpack(uint64_t v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
// the largest of three fp32 values
__device__ __forceinline__ float max3f(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}
// two fp32 values rounded to a bf16 pair (low half = first)
__device__ __forceinline__ uint32_t pack_bf16_rn(float lo, float hi) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}


// Ancestor-or-self mask of every node of sequence b (node j is bit j) into
// anc. All threads of the CTA take part: the parents are loaded and checked
// at once (a parent precedes its node, the root's is -1; a bad one is
// reported and taken as -1) into par, then each node's chain is walked. The
// caller synchronises before reading the masks.
__device__ void attn_ancestors(const AttnParams& p, int b, uint64_t* anc, int* par) {
  for (int j = threadIdx.x; j < p.n; j += blockDim.x) {
    int q = p.parents ? p.parents[(int64_t)b * p.n + j] : j - 1;
    if (j == 0 ? q != -1 : (q < 0 || q >= j)) {
      report_error(p.err, kErrInput);
      q = -1;
    }
    par[j] = q;
  }
  __syncthreads();
  for (int j = threadIdx.x; j < p.n; j += blockDim.x) {
    uint64_t a = 1ull << j;
    for (int k = par[j]; k >= 0; k = par[k]) a |= 1ull << k;
    anc[j] = a;
  }
}

// ------------------------------------------------ tcgen05 tree attention
// One CTA per SM and per piece: a block of TILES x 128 query rows of a KV
// head of a sequence against a run of its key blocks (all of them, or a piece
// of a sequence cut to fill one wave of CTAs); the TILES tiles of 128 rows
// share every key block.
// TILES = 2 (more than 128 query rows per KV head: tree drafts): 12 warps, a
// 4-stage ring, all 512 TMEM columns. TILES = 1 (up to 128 rows: sequence
// drafts and small trees, where streaming the keys and values is the cost):
// 6 warps, a 6-stage ring, Q in TMEM beside the scores and O (S = Q K^T then
// takes its A operand from TMEM).
//   warp 0        2-D TMA of the 64-key blocks of K and V into the ring
//   warps 1 ..    the MMAs of tile 0 (and tile 1) (whole warp in the loop, the
//                 elect.sync lane issuing): S = Q K^T (M = 128 query rows,
//                 N = 64 keys, K = 128; A = Q from shared memory with two
//                 tiles, from TMEM with one; B = K from shared memory) into
//                 the tile's TMEM score buffer, and O += P V (M = 128, N = 128
//                 head columns, K = 64 keys; P from TMEM, V from shared
//                 memory as it was loaded: key rows of head columns, the
//                 MN-major B operand) into the tile's TMEM accumulator. Each
//                 tile has two TMEM score buffers: S for block i + 2 goes out
//                 once the P V of block i, whose P sits in the same buffer,
//                 is complete, so the scores of the next block are ready
//                 when the softmax reaches it; the two tiles' MMAs
//                 interleave on the tensor pipe.
//   warp 3        idle (TILES = 2)
//   4 per tile    the softmax warps from warp 4 (TILES = 2) or 2 (TILES = 1):
//                 one query row per thread, TMEM lane quadrant warp % 4:
//                 the row's scores from TMEM, the mask as one 64-bit word
//                 per block (committed prefix: every key; tree keys: the
//                 node's ancestors and itself; skipped on blocks of the
//                 prefix), the
//                 online softmax in the log2 domain (the row sum over the
//                 fp32 weights) and P (rounded to bf16) back into TMEM,
//                 over the first half of the scores just read;
//                 at the end the normalised row (or a piece's partial)
// While one tile's softmax runs, the tensor pipe works on the other tile.
// The running maximum is raised only when a block's maximum exceeds it by
// more than 8 (a factor 256: P stays well inside bf16 and fp32), so the
// accumulator in TMEM is rescaled rarely; the result O / l does not depend on
// which maximum the weights were taken against.
constexpr int kTaRows = 128;   // query rows per tile (UMMA M)
constexpr float kTaLazy = 8.0f;  // log2 of the largest weight before the maximum is raised

template <int TILES>
struct TaConfig {
  static constexpr int kStages = TILES == 2 ? 4 : 6;
  static constexpr int kSoftWarp0 = TILES == 2 ? 4 : 2;  // first softmax warp
  static constexpr int kThreads = 32 * (kSoftWarp0 + 4 * TILES);
  // two score buffers per tile (S(i + 2) waits for P V (i), whose P sits in
  // its buffer). One tile: Q in TMEM too (S = Q K^T then reads its A operand
  // there, 33 instead of ~50 cycles an MMA, and the ring takes Q's shared
  // memory); two tiles fill the TMEM with scores and O, Q stays in shared
  // memory (a single score buffer with Q in TMEM measured 158 against 111 us:
  // S(i + 1) then waits for P V (i))
  static constexpr uint32_t kTmemCols = 512u;
  static constexpr int kSBufs = 2;
  static constexpr bool kQInTmem = TILES == 1;
};

template <int TILES>
struct TaLayout {
  static constexpr int S = TaConfig<TILES>::kStages;
  static constexpr int kKHalf = kAttKeys * 128;       // 64 keys x 64 head columns
  static constexpr int kStage = 4 * kKHalf;          // K halves, V halves
  static constexpr int kQHalf = kTaRows * 128;  // 128 rows x 64 head columns (bf16)
  static constexpr int kQOff = 0;               // Q in shared memory: tile t's halves at 2 t kQHalf
  static constexpr int kStageOff = TaConfig<TILES>::kQInTmem ? 0 : TILES * 2 * kQHalf;
  static constexpr int kAncOff = kStageOff + S * kStage;
  static constexpr int kBarOff = kAncOff + kAttMaxNodes * 8;
  // kv_full[S], kv_free[S]; per tile s_full[2], p_full[2], pv_done[2], mma_fin; q_ready
  static constexpr int kNumBars = 2 * S + TILES * 7 + 1;
  static constexpr int kTotal = kBarOff + kNumBars * 8 + 16 + 1024;  // + TMEM base, alignment
  static_assert(kStage % 1024 == 0 && kQHalf % 1024 == 0 && kKHalf % 1024 == 0, "swizzle atoms");
  static_assert(kTotal + 512 <= 227 * 1024, "shared memory (with the static words and parents)");
};
// TMEM columns of tile t: score buffer sb at 128 t + 64 sb .. + 63 (the
// block's P, bf16 pairs, over its first 32 columns); O 128 TILES + 128 t ..
// + 127; one tile's Q (bf16 pairs) at 256 .. 319
template <int TILES>
__device__ __forceinline__ uint32_t ta_s_col(int t, int sb) {
  return 128u * (uint32_t)t + 64u * (uint32_t)sb;
}
constexpr uint32_t kTaQCol = 256u;
template <int TILES>
__device__ __forceinline__ uint32_t ta_o_col(int t) {
  return 128u * (uint32_t)TILES + 128u * (uint32_t)t;
}

// lane 0 waits (bounded), every lane gets the outcome. The hand-offs of
// this kernel are short and on its critical path, so the first tests do not
// ask the hardware to suspend the thread (a suspended waiter wakes up late:
// 382 -> 287 us for 16 sequences x 64-node trees, measured).
__device__ __forceinline__ bool ta_wait(uint64_t* bar, uint32_t parity, unsigned* err) {
  int ok = 1;
  if ((threadIdx.x & 31) == 0) {
    int k = 0;
    while (k < 64 && !mbar_try_wait(bar, parity)) ++k;
    if (k == 64) ok = mbar_wait(bar, parity, err) ? 1 : 0;
  }
  ok = __shfl_sync(0xffffffffu, ok, 0);
  __syncwarp();
  return ok != 0;
}

// The work of one CTA: the query rows of row block rb of KV head kvh of
// sequence b, against key blocks blk0 .. blk0 + nb - 1 of that sequence, one
// of the np pieces the sequence was cut into (np = 1: the rows are finished
// here; otherwise the CTA leaves a partial in its slot). b < 0: no work.
struct TaWork {
  int b, kvh, rb, blk0, nb, np, len;
};

// Warp-collective (one warp): the piece of CTA x. With up to 64 sequences
// every (sequence, KV head, row block) unit is cut into np pieces of about
// the same number of key blocks, np = ceil(nblk / Q) for a sequence of nblk
// blocks, Q the smallest length for which all pieces fit p.ctas CTAs (one
// wave; when the units alone fill them, np = 1); pieces are numbered in
// decreasing blocks per piece (ties by sequence), a sequence's pieces unit by
// unit and piece by piece, so that the longest start first. Above 64
// sequences: one piece per unit, in order.
__device__ TaWork ta_assign(const AttnParams& p, int x, int lane) {
  const int units = p.Hkv * p.row_blocks;
  const int hi = min(p.max_len, p.Lcap - p.n);
  TaWork w{-1, 0, 0, 0, 0, 1, 0};
  if (p.B > 64) {
    const int b = x / units;
    if (b < p.B) {
      const int u = x - b * units;
      int len = p.lens[b];
      if (len < 0 || len > hi) {
        if (lane == 0) report_error(p.err, kErrInput);
        len = len < 0 ? 0 : hi;
      }
      w = TaWork{b, u / p.row_blocks, u % p.row_blocks, 0, (len + p.n + kAttKeys - 1) / kAttKeys, 1, len};
    }
    return w;
  }
  int len[2], nbk[2], np[2], ps[2], off[2] = {0, 0};
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int c = lane + 32 * h;
    int l = c < p.B ? p.lens[c] : 0;
    l = l < 0 ? 0 : (l > hi ? hi : l);
    len[h] = l;
    nbk[h] = c < p.B ? (l + p.n + kAttKeys - 1) / kAttKeys : 0;
  }
  int qhi = __reduce_max_sync(0xffffffffu, max(nbk[0], nbk[1]));
  int q = p.cut ? 1 : qhi;  // not cut: one piece per unit
  while (q < qhi) {  // the smallest piece length whose pieces fit the CTAs
    const int mid = (q + qhi) >> 1;
    const int cnt = __reduce_add_sync(0xffffffffu, (nbk[0] + mid - 1) / mid + (nbk[1] + mid - 1) / mid);
    if ((int64_t)cnt * units <= p.ctas)
      qhi = mid;
    else
      q = mid + 1;
  }
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    np[h] = (nbk[h] + q - 1) / q;
    ps[h] = np[h] > 0 ? (nbk[h] + np[h] - 1) / np[h] : 0;
  }
  for (int c2 = 0; c2 < p.B; ++c2) {  // pieces numbered before each sequence's first
    const int ps2 = __shfl_sync(0xffffffffu, c2 < 32 ? ps[0] : ps[1], c2 & 31);
    const int np2 = __shfl_sync(0xffffffffu, c2 < 32 ? np[0] : np[1], c2 & 31);
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int c = lane + 32 * h;
      if (c < p.B && (ps2 > ps[h] || (ps2 == ps[h] && c2 < c))) off[h] += np2 * units;
    }
  }
  int found = -1;
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int c = lane + 32 * h;
    if (c < p.B && x >= off[h] && x < off[h] + np[h] * units) {
      const int li = x - off[h], u = li / np[h], k = li - u * np[h];
      const int blk0 = k * ps[h];
      w = TaWork{c, u / p.row_blocks, u % p.row_blocks, blk0, min(nbk[h], blk0 + ps[h]) - blk0, np[h], len[h]};
      found = h;
      if (li == 0) {  // the sequence's first piece reports a bad length and records its pieces
        const int raw = p.lens[c];
        if (raw < 0 || raw > hi) report_error(p.err, kErrInput);
        if (p.cut) p.seq_pieces[c] = make_int2(off[h], np[h]);
      }
    }
  }
  const int src = __ffs(__ballot_sync(0xffffffffu, found >= 0)) - 1;
  if (src < 0) return TaWork{-1, 0, 0, 0, 0, 1, 0};
  return TaWork{__shfl_sync(0xffffffffu, w.b, src),   __shfl_sync(0xffffffffu, w.kvh, src),
                __shfl_sync(0xffffffffu, w.rb, src),  __shfl_sync(0xffffffffu, w.blk0, src),
                __shfl_sync(0xffffffffu, w.nb, src),  __shfl_sync(0xffffffffu, w.np, src),
                __shfl_sync(0xffffffffu, w.len, src)};
}

template <int TILES>
__global__ void __launch_bounds__(TaConfig<TILES>::kThreads, 1)
    tree_attention_tc_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
                             const AttnParams p) {
  using L = TaLayout<TILES>;
  using C = TaConfig<TILES>;
  constexpr int S = C::kStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* anc = reinterpret_cast<uint64_t*>(smem + L::kAncOff);
  uint64_t* kv_full = reinterpret_cast<uint64_t*>(smem + L::kBarOff);
  uint64_t* kv_free = kv_full + S;  // both tiles' P V of the block are complete: K and V are free
  uint64_t* tb = kv_free + S;       // per tile: s_full[2], p_full[2], pv_done[2], mma_fin
  auto s_full = [&](int t, int sb) { return tb + 7 * t + sb; };
  auto p_full = [&](int t, int pb) { return tb + 7 * t + 2 + pb; };
  auto pv_done = [&](int t, int pb) { return tb + 7 * t + 4 + pb; };
  auto mma_fin = [&](int t) { return tb + 7 * t + 6; };
  uint64_t* q_ready = tb + 7 * TILES;
  uint32_t* tmem_base_s = reinterpret_cast<uint32_t*>(q_ready + 1);
  __shared__ TaWork s_w;
  __shared__ int s_par[kAttMaxNodes];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  grid_launch_dependents();
  grid_dependency_wait();  // q, the caches and lens may come from the preceding kernels
  if (warp == 0) {
    const TaWork w = ta_assign(p, (int)blockIdx.x, lane);
    if (lane == 0) s_w = w;
  }
  __syncthreads();
  const TaWork w = s_w;
  if (w.b < 0) return;  // the whole CTA: no piece left for it
  const int b = w.b, kvh = w.kvh, rb = w.rb, len = w.len, blk0 = w.blk0, nb = w.nb;
  // tiles holding query rows (the last row block of a head may need one)
  const int ntiles = min(TILES, (p.rows - rb * TILES * kTaRows + kTaRows - 1) / kTaRows);
  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&kv_full[s], 1);
      mbar_init(&kv_free[s], (uint32_t)ntiles);  // each tile's last P V commit
    }
    for (int t = 0; t < TILES; ++t) {
      for (int pb = 0; pb < 2; ++pb) {
        mbar_init(s_full(t, pb), 1);
        mbar_init(p_full(t, pb), 4);  // the tile's four softmax warps
        mbar_init(pv_done(t, pb), 1);
      }
      mbar_init(mma_fin(t), 1);
    }
    mbar_init(q_ready, 4 * TILES);
    fence_mbarrier_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_base_s, C::kTmemCols);
    tmem_relinquish();
  }
  attn_ancestors(p, b, anc, s_par);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_base_s;
  const int64_t kv_row0 = ((int64_t)b * p.Hkv + kvh) * p.Lcap;
  int mma_issued = 0;

  if (warp == 0) {
    // ---------------------------------------------------------- producer
    if (lane == 0) {
      int i = 0;
      for (; i < nb; ++i) {
        const int s = i % S;
        if (i >= S && !mbar_wait(&kv_free[s], (uint32_t)(i / S - 1) & 1u, p.err)) break;
        uint8_t* st = smem + L::kStageOff + s * L::kStage;
        const int32_t y = (int32_t)(kv_row0 + (int64_t)(blk0 + i) * kAttKeys);
        mbar_arrive_expect_tx(&kv_full[s], (uint32_t)(4 * L::kKHalf));
        tma_load_2d(st, &kmap, 0, y, &kv_full[s]);
        tma_load_2d(st + L::kKHalf, &kmap, 64, y, &kv_full[s]);
        tma_load_2d(st + 2 * L::kKHalf, &vmap, 0, y, &kv_full[s]);
        tma_load_2d(st + 3 * L::kKHalf, &vmap, 64, y, &kv_full[s]);
      }
      if (i < nb)  // a wait ran out: let the copies in flight land before the CTA exits
        for (int k = i > S ? i - S : 0; k < i; ++k) mbar_wait(&kv_full[k % S], (uint32_t)(k / S) & 1u, p.err);
    }
  } else if (warp >= 1 && warp <= TILES) {
    // ------------------------------------------------------ MMA, tile t
    const int t = warp - 1;
    const uint32_t idesc_s = umma_idesc_bf16((uint32_t)kAttKeys), idesc_o = umma_idesc_bf16_bmn((uint32_t)kAttD);
    bool ok = ta_wait(q_ready, 0u, p.err);
    tc_fence_after();
    constexpr int lag = C::kSBufs;
    // S(i) = Q K(i)^T into the tile's score buffer i % kSBufs, once P V
    // (i - kSBufs) (its P in the same buffer) is complete
    auto issue_s = [&](int i) {
      const int s = i % S, sb = i & 1;
      if (!ta_wait(&kv_full[s], (uint32_t)(i / S) & 1u, p.err)) return false;
      if (i >= lag && !ta_wait(pv_done(t, (i - lag) & 1), (uint32_t)((i - lag) / 2) & 1u, p.err)) return false;
      tc_fence_after();
      const uint32_t k0 = smem_u32(smem + L::kStageOff + s * L::kStage);
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        const uint32_t koff = (uint32_t)((kk >> 2) * L::kKHalf + 32 * (kk & 3));
        if constexpr (C::kQInTmem) {
          umma_bf16_ts_warp(tmem + ta_s_col<TILES>(t, sb), tmem + kTaQCol + 8u * (uint32_t)kk,
                            umma_desc_sw128_kmajor(k0 + koff), idesc_s, kk > 0 ? 1u : 0u);
        } else {
          const uint32_t q0 = smem_u32(smem + L::kQOff + t * 2 * L::kQHalf);
          umma_bf16_ss_warp(tmem + ta_s_col<TILES>(t, sb),
                            umma_desc_sw128_kmajor(q0 + (uint32_t)((kk >> 2) * L::kQHalf + 32 * (kk & 3))),
                            umma_desc_sw128_kmajor(k0 + koff), idesc_s, kk > 0 ? 1u : 0u);
        }
      }
      umma_commit_warp(s_full(t, sb));
      mma_issued = 1;
      return true;
    };
    if (t >= ntiles) ok = false;  // no rows in this tile
    for (int i = 0; ok && i < lag && i < nb; ++i) ok = issue_s(i);
    for (int i = 0; ok && i < nb; ++i) {
      const int s = i % S, pb = i & 1;
      if (!ta_wait(p_full(t, pb), (uint32_t)(i / 2) & 1u, p.err)) break;
      tc_fence_after();
      // V half h: keys 0 .. 63 x head columns 64 h .. 64 h + 63, 128-byte rows;
      // 16 keys (two 8-row atoms) per MMA, the second head-column half kKHalf on
      const uint32_t v0 = smem_u32(smem + L::kStageOff + s * L::kStage + 2 * L::kKHalf);
#pragma unroll
      for (int kk = 0; kk < 4; ++kk)
        umma_bf16_ts_warp(tmem + ta_o_col<TILES>(t), tmem + ta_s_col<TILES>(t, pb) + 8u * (uint32_t)kk,
                          umma_desc_sw128_mnmajor(v0 + 2048u * (uint32_t)kk, (uint32_t)L::kKHalf, 1024u), idesc_o,
                          (i > 0 || kk > 0) ? 1u : 0u);
      umma_commit_warp(pv_done(t, pb));
      umma_commit_warp(&kv_free[s]);
      if (i + lag < nb && !issue_s(i + lag)) break;
    }
    if (mma_issued) umma_commit_warp(mma_fin(t));  // tracks all of this warp's MMAs
  } else if (warp < C::kSoftWarp0) {
    // idle
  } else {
    // --------------------------------------------------------- softmax
    const int t = (warp - C::kSoftWarp0) >> 2;  // tile
    const int qd = warp & 3;        // TMEM lane quadrant
    const int rl = qd * 32 + lane;
    const int R = rb * TILES * kTaRows + t * kTaRows + rl;
    const bool valid = R < p.rows;
    const int j = valid ? R / p.G : 0, g = R - j * p.G;
    // this row of Q: into TMEM with one tile (the row's lane, 64 columns of
    // bf16 pairs), else into shared memory (128-byte swizzle, K-major, two
    // 64-column halves)
    {
      const int64_t qi = (((int64_t)b * p.n + j) * p.H + kvh * p.G + g) * kAttD;
      const bool qok = valid && in_bounds(p.err, qi + kAttD - 1, (int64_t)p.B * p.n * p.H * kAttD);
      // all 16 loads in flight before the first store (a store between two
      // loads would make each load wait for the one before it)
      uint4 v[16];
#pragma unroll
      for (int c = 0; c < 16; ++c)
        v[c] = qok ? *reinterpret_cast<const uint4*>(p.q + qi + c * 8) : make_uint4(0u, 0u, 0u, 0u);
      if constexpr (C::kQInTmem) {
        const uint32_t qrow = tmem + ((uint32_t)(32 * qd) << 16) + kTaQCol;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          uint32_t w[32];
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            w[4 * c] = v[8 * h + c].x;
            w[4 * c + 1] = v[8 * h + c].y;
            w[4 * c + 2] = v[8 * h + c].z;
            w[4 * c + 3] = v[8 * h + c].w;
          }
          tmem_st_32x32b_x32(qrow + 32u * (uint32_t)h, w);
        }
        tmem_wait_st();
        tc_fence_before();
      } else {
        uint8_t* qt = smem + L::kQOff + t * 2 * L::kQHalf;
#pragma unroll
        for (int c = 0; c < 16; ++c)
          *reinterpret_cast<uint4*>(qt + (c >> 3) * L::kQHalf + rl * 128 + (((c & 7) ^ (rl & 7)) << 4)) = v[c];
        fence_proxy_async_smem();
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(q_ready);
    }
    const uint64_t an = valid ? anc[j] : 0ull;
    const uint32_t trow = tmem + ((uint32_t)(32 * qd) << 16);
    const int nbt = t < ntiles ? nb : 0;
    float m_used = -INFINITY, l = 0.0f;
    bool ok = true;
    // a warp without query rows (padding of the last tile) only keeps the
    // hand-offs' counts: its Q rows are zero, so are its scores, and the P
    // it leaves in TMEM (those scores' bits) is zero as well
    const bool any_row = __any_sync(0xffffffffu, valid);
    for (int i = 0; i < nbt; ++i) {
      const int pb = i & 1;
      if (!ta_wait(s_full(t, pb), (uint32_t)(i / 2) & 1u, p.err)) {
        ok = false;
        break;
      }
      if (!any_row) {
        __syncwarp();
        if (lane == 0) mbar_arrive(p_full(t, pb));
        continue;
      }
      tc_fence_after();
      uint32_t sv[2][32];
      tmem_ld_32x32b_x32(trow + ta_s_col<TILES>(t, pb), sv[0]);
      tmem_ld_32x32b_x32(trow + ta_s_col<TILES>(t, pb) + 32u, sv[1]);
      tmem_wait_ld();
      // the mask (keys the row does not see: -inf), then the block's maximum
      // on the raw scores (the positive scale commutes with it), in the log2
      // domain. A block of the committed prefix alone needs no mask (every
      // key is seen by every row); nor does a padding row (never stored).
      const int key0 = (blk0 + i) * kAttKeys;
      if (key0 + kAttKeys > len) {
        // the block's visible keys as a word (bit k: key key0 + k): the
        // committed prefix below d, then node t of the tree at bit d + t for
        // each of the row's ancestors and itself
        const int d = len - key0;  // < 64 here
        uint64_t vis = d > 0 ? (1ull << d) - 1ull : 0ull;
        if (d >= 0)
          vis |= an << d;
        else if (d > -64)
          vis |= an >> (-d);
        const uint32_t vw[2] = {(uint32_t)vis, (uint32_t)(vis >> 32)};
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
          for (int c = 0; c < 32; ++c)
            if (!((vw[h] >> c) & 1u)) sv[h][c] = __float_as_uint(-INFINITY);
      }
      float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
      for (int h = 0; h < 2; ++h)
#pragma unroll
        for (int c = 0; c < 16; ++c)
          m4[c & 3] = max3f(m4[c & 3], __uint_as_float(sv[h][2 * c]), __uint_as_float(sv[h][2 * c + 1]));
      const float mx = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3])) * p.scale_log2;
      // raise the running maximum only by more than kTaLazy; rescale l and O then
      float cf = 1.0f;
      if (mx > m_used + kTaLazy) {
        cf = m_used == -INFINITY ? 0.0f : ex2(m_used - mx);
        m_used = mx;
        l *= cf;
      }
      if (__any_sync(0xffffffffu, cf < 1.0f && i > 0)) {
        // O holds the sums of blocks 0 .. i - 1: wait for the last of them
        if (!ta_wait(pv_done(t, (i - 1) & 1), (uint32_t)((i - 1) / 2) & 1u, p.err)) {
          ok = false;
          break;
        }
        tc_fence_after();
#pragma unroll 1
        for (int c0 = 0; c0 < kAttD; c0 += 32) {
          uint32_t ov[32];
          tmem_ld_32x32b_x32(trow + ta_o_col<TILES>(t) + (uint32_t)c0, ov);
          tmem_wait_ld();
#pragma unroll
          for (int c = 0; c < 32; ++c) ov[c] = __float_as_uint(__uint_as_float(ov[c]) * cf);
          tmem_st_32x32b_x32(trow + ta_o_col<TILES>(t) + (uint32_t)c0, ov);
        }
        tmem_wait_st();
      }
      // P = 2^(s scale - m), rounded to bf16 for P V; l over the fp32 values.
      // The exponents' arguments and the sums go two lanes per instruction.
      const float u = m_used == -INFINITY ? 0.0f : m_used;
      const uint64_t sc2 = f2_pack(p.scale_log2, p.scale_log2), nu2 = f2_pack(-u, -u);
      uint64_t la = f2_pack(0.0f, 0.0f), lb = la;
      uint32_t pr[32];
#pragma unroll
      for (int h = 0; h < 2; ++h)
#pragma unroll
        for (int c = 0; c < 16; ++c) {
          float x0, x1;
          f2_unpack(f2_fma(f2_pack(__uint_as_float(sv[h][2 * c]), __uint_as_float(sv[h][2 * c + 1])), sc2, nu2), x0, x1);
          const float e0 = ex2(x0), e1 = ex2(x1);
          pr[16 * h + c] = pack_bf16_rn(e0, e1);
          const uint64_t r2 = f2_pack(e0, e1);
          if (c & 1)
            lb = f2_add(lb, r2);
          else
            la = f2_add(la, r2);
        }
      {
        float a0, a1, b0, b1;
        f2_unpack(la, a0, a1);
        f2_unpack(lb, b0, b1);
        l += (a0 + a1) + (b0 + b1);
      }
      tmem_st_32x32b_x32(trow + ta_s_col<TILES>(t, pb), pr);  // over the scores just read
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(p_full(t, pb));
    }
    // ---- the row: O / l (the sequence in one piece) or the piece's
    // (m, l, O) in the CTA's slot; a piece without keys leaves (-inf, 0)
    const int64_t base = (int64_t)blockIdx.x * p.unit_rows;
    const int64_t rows_cap = (int64_t)p.ctas * p.unit_rows;
    const int Ru = R - rb * p.unit_rows;  // the row within the CTA's rows
    if (ok && nb == 0 && valid && w.np > 1 && p.cut && in_bounds(p.err, base + Ru, rows_cap))
      p.part_ml[base + Ru] = make_float2(-INFINITY, 0.0f);
    if (ok && nbt > 0 && any_row && ta_wait(pv_done(t, (nb - 1) & 1), (uint32_t)((nb - 1) / 2) & 1u, p.err)) {
      tc_fence_after();
      const float il = l > 0.0f ? 1.0f / l : 0.0f;
      const int64_t out_cap = (int64_t)p.B * p.n * p.H * kAttD;
      const int64_t oi = (((int64_t)b * p.n + j) * p.H + kvh * p.G + g) * kAttD;
      const bool st_ok = valid && (w.np == 1 ? in_bounds(p.err, oi + kAttD - 1, out_cap)
                                             : p.cut && in_bounds(p.err, base + Ru, rows_cap));
#pragma unroll 1
      for (int c0 = 0; c0 < kAttD; c0 += 32) {
        uint32_t ov[32];
        tmem_ld_32x32b_x32(trow + ta_o_col<TILES>(t) + (uint32_t)c0, ov);
        tmem_wait_ld();
        if (!st_ok) continue;
        if (w.np == 1) {
#pragma unroll
          for (int c = 0; c < 32; c += 8) {
            uint4 w;
            w.x = pack_bf16_rn(__uint_as_float(ov[c]) * il, __uint_as_float(ov[c + 1]) * il);
            w.y = pack_bf16_rn(__uint_as_float(ov[c + 2]) * il, __uint_as_float(ov[c + 3]) * il);
            w.z = pack_bf16_rn(__uint_as_float(ov[c + 4]) * il, __uint_as_float(ov[c + 5]) * il);
            w.w = pack_bf16_rn(__uint_as_float(ov[c + 6]) * il, __uint_as_float(ov[c + 7]) * il);
            *reinterpret_cast<uint4*>(p.out + oi + c0 + c) = w;
          }
        } else {
          float* dst = p.part_o + (base + Ru) * kAttD + c0;
#pragma unroll
          for (int c = 0; c < 32; c += 4)
            *reinterpret_cast<float4*>(dst + c) = make_float4(__uint_as_float(ov[c]), __uint_as_float(ov[c + 1]),
                                                              __uint_as_float(ov[c + 2]), __uint_as_float(ov[c + 3]));
        }
      }
      if (st_ok && w.np > 1) p.part_ml[base + Ru] = make_float2(m_used, l);
    }
  }

  // ---------------------------------------------------------- teardown
  tc_fence_before();
  __syncthreads();
  if (warp >= 1 && warp <= TILES && lane == 0 && mma_issued)
    mbar_wait(mma_fin(warp - 1), 0u, p.err);  // no MMA in flight when TMEM is freed
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

// One warp per query row of a sequence that was cut into pieces: the
// pieces' (m, l, O), in the slots the sequence's first piece recorded, merged
// and stored as bf16 (lane k: columns 4k .. 4k + 3); a sequence in one piece
// was finished by its CTA.
__global__ void __launch_bounds__(256) tree_attention_combine_kernel(const AttnParams p) {
  grid_launch_dependents();
  grid_dependency_wait();
  const int64_t row = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  const int64_t per_b = (int64_t)p.Hkv * p.rows;
  if (row >= (int64_t)p.B * per_b) return;
  const int b = (int)(row / per_b);
  const int kvh = (int)((row - b * per_b) / p.rows);
  const int R = (int)(row - b * per_b - (int64_t)kvh * p.rows);
  const int j = R / p.G, g = R - j * p.G;
  const int2 sp = __ldcg(&p.seq_pieces[b]);  // (first piece, pieces)
  if (sp.y <= 1) return;
  const int rbi = R / p.unit_rows, Ru = R - rbi * p.unit_rows;
  const int64_t x0 = (int64_t)sp.x + ((int64_t)kvh * p.row_blocks + rbi) * sp.y;
  if (x0 < 0 || x0 + sp.y > p.ctas) {
    if (lane == 0) report_error(p.err, kErrBounds);
    return;
  }
  float M = -INFINITY;
  for (int s = 0; s < sp.y; ++s) M = fmaxf(M, __ldcg(&p.part_ml[(x0 + s) * p.unit_rows + Ru]).x);
  float lsum = 0.0f, acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
  for (int s = 0; s < sp.y; ++s) {
    const int64_t slot_row = (x0 + s) * p.unit_rows + Ru;
    const float2 ml = __ldcg(&p.part_ml[slot_row]);
    if (!(ml.y > 0.0f)) continue;  // no key of this row in the piece
    const float w = ex2(ml.x - M);
    lsum += w * ml.y;
    const float4 v = __ldcg(reinterpret_cast<const float4*>(p.part_o + slot_row * kAttD) + lane);
    acc[0] += w * v.x;
    acc[1] += w * v.y;
    acc[2] += w * v.z;
    acc[3] += w * v.w;
  }
  const float inv = lsum > 0.0f ? 1.0f / lsum : 0.0f;
  __nv_bfloat16* dst = p.out + (((int64_t)b * p.n + j) * p.H + kvh * p.G + g) * kAttD + 4 * lane;
  *reinterpret_cast<__nv_bfloat162*>(dst) = __floats2bfloat162_rn(acc[0] * inv, acc[1] * inv);
  *reinterpret_cast<__nv_bfloat162*>(dst + 2) = __floats2bfloat162_rn(acc[2] * inv, acc[3] * inv);
}

// --------------------------------------------------------- KV compaction
// Grid (B, layers). The accepted root path, root first, is path[0 .. depth);
// path[d] >= d, so a move only reads positions at or past the ones earlier
// moves have written: the moves go in chunks of depths, each chunk read
// whole into registers before any of it is written.
constexpr int kCompactThreads = 256;
constexpr int kCompactPerThread = 16;  // 16-byte words a thread holds per chunk

__global__ void __launch_bounds__(kCompactThreads) kv_compact_kernel(uint4* kc, uint4* vc, const int32_t* lens,
                                                                     const int32_t* parents, const int32_t* node,
                                                                     int B, int n, int Hkv, int row_words, int Lcap,
                                                                     int32_t* new_lens, unsigned* err) {
  grid_launch_dependents();
  grid_dependency_wait();
  __shared__ int path[kAttMaxNodes + 1];
  __shared__ int s_depth, s_len;
  const int b = blockIdx.x, layer = blockIdx.y, tid = threadIdx.x;
  if (tid == 0) {
    int len = lens[b];
    if (len < 0 || len > Lcap - n) {
      report_error(err, kErrInput);
      len = len < 0 ? 0 : Lcap - n;
    }
    int j = node[b];
    bool bad = j < 0 || j >= n;
    if (bad) j = 0;
    int depth = 0;
    int tmp[kAttMaxNodes + 1];
    while (j >= 0 && depth <= n) {
      tmp[depth++] = j;
      const int par = parents ? parents[(int64_t)b * n + j] : j - 1;
      if (j == 0 ? par != -1 : (par < 0 || par >= j)) {
        bad = true;
        break;
      }
      j = par;
    }
    if (bad) {  // the root alone
      depth = 1;
      tmp[0] = 0;
      report_error(err, kErrInput);
    }
    for (int d = 0; d < depth; ++d) path[d] = tmp[depth - 1 - d];
    s_depth = depth;
    s_len = len;
    if (layer == 0) new_lens[b] = len + depth;
  }
  __syncthreads();
  const int depth = s_depth, len = s_len;
  const int per_depth = 2 * Hkv * row_words;  // keys and values of every head
  const int chunk = max(1, kCompactThreads * kCompactPerThread / per_depth);
  const int64_t head_words = (int64_t)Lcap * row_words;
  const int64_t bh0 = ((int64_t)layer * B + b) * Hkv;
  for (int d0 = 1; d0 < depth; d0 += chunk) {
    const int d1 = min(depth, d0 + chunk);
    const int total = (d1 - d0) * per_depth;
    uint4 v[kCompactPerThread];
#pragma unroll
    for (int k = 0; k < kCompactPerThread; ++k) {
      const int idx = tid + k * kCompactThreads;
      if (idx < total) {
        const int d = d0 + idx / per_depth, rem = idx % per_depth;
        const int c = rem / (Hkv * row_words), h = (rem / row_words) % Hkv, w = rem % row_words;
        const uint4* src = (c ? vc : kc) + (bh0 + h) * head_words + (int64_t)(len + path[d]) * row_words + w;
        if (in_bounds(err, (int64_t)(len + path[d]) * row_words + w, head_words)) v[k] = *src;
      }
    }
    __syncthreads();
#pragma unroll
    for (int k = 0; k < kCompactPerThread; ++k) {
      const int idx = tid + k * kCompactThreads;
      if (idx < total) {
        const int d = d0 + idx / per_depth, rem = idx % per_depth;
        if (path[d] == d) continue;  // already in place
        const int c = rem / (Hkv * row_words), h = (rem / row_words) % Hkv, w = rem % row_words;
        uint4* dst = (c ? vc : kc) + (bh0 + h) * head_words + (int64_t)(len + d) * row_words + w;
        if (in_bounds(err, (int64_t)(len + d) * row_words + w, head_words)) *dst = v[k];
      }
    }
    __syncthreads();
  }
}

// ------------------------------------------------------------------ host

// warps per CTA: 1, 2, 4 or 8 (measured on the 5-position chain with 64
// heads on 8: four warps with two stages beat three with three stages)

AttnPlan attn_plan(int B, int n, int H, int Hkv, int max_len, int num_sms) {
  AttnPlan pl;
  const int G = H / Hkv;
  pl.rows = n * G;
  // the tcgen05 kernel: two 128-row tiles per CTA above 128 query rows per
  // KV head, one up to 128
  pl.tiles = pl.rows > kTaRows ? 2 : 1;
  const int per_cta = pl.tiles * kTaRows;
  pl.row_blocks = (pl.rows + per_cta - 1) / per_cta;
  // one wave of CTAs: up to 64 sequences are cut into pieces on the device
  // (from the committed lengths) when their units leave at least half the
  // CTAs free (with fewer free, only the longest few would be cut and the
  // combine costs more than it saves: K = 4 sequence draft at B = 16, 128
  // units on 152 SMs, 63.3 us uncut against 67.8 us cut)
  const int64_t units = (int64_t)B * Hkv * pl.row_blocks;
  pl.ctas = num_sms > 0 ? num_sms : 1;
  pl.cut = B <= 64 && 2 * units <= pl.ctas ? 1 : 0;
  pl.pieces_max = (int)(units > pl.ctas ? units : pl.ctas);
  pl.ws_bytes = pl.cut ? (size_t)pl.ctas * per_cta * (kAttD * 4 + 8) + (size_t)B * 8 : 0;
  return pl;
}


template <int TILES>
static cudaError_t launch_attn_tc_t(const CUtensorMap& km, const CUtensorMap& vm, const AttnParams& p, dim3 grid,
                                    cudaStream_t stream) {
  constexpr int smem = TaLayout<TILES>::kTotal;
  cudaError_t e =
      cudaFuncSetAttribute(tree_attention_tc_kernel<TILES>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  return launch_pdl(tree_attention_tc_kernel<TILES>, grid, dim3(TaConfig<TILES>::kThreads), (size_t)smem, stream,
                    km, vm, p);
}

cudaError_t launch_tree_attention(const void* q, const void* k_cache, const void* v_cache, const int32_t* lens,
                                  const int32_t* parents, int B, int n, int H, int Hkv, int Lcap, int max_len,
                                  float scale, void* out, void* workspace, const AttnPlan& pl, unsigned* err,
                                  cudaStream_t stream) {
  auto encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(tensor_map_encode_fn());
  if (!encode) return cudaErrorNotSupported;
  CUtensorMap km, vm;
  const cuuint64_t dims[2] = {(cuuint64_t)kAttD, (cuuint64_t)B * Hkv * Lcap};
  const cuuint64_t strides[1] = {(cuuint64_t)kAttD * 2};
  const cuuint32_t box[2] = {64u, (cuuint32_t)kAttKeys};
  const cuuint32_t es[2] = {1u, 1u};
  for (int c = 0; c < 2; ++c)
    if (encode(c ? &vm : &km, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(c ? v_cache : k_cache), dims,
               strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  AttnParams p;
  p.q = static_cast<const __nv_bfloat16*>(q);
  p.lens = lens;
  p.parents = parents;
  p.out = static_cast<__nv_bfloat16*>(out);
  p.part_o = static_cast<float*>(workspace);
  const size_t slot_rows = (size_t)pl.ctas * pl.tiles * kTaRows;
  p.part_ml = reinterpret_cast<float2*>(static_cast<uint8_t*>(workspace) + slot_rows * kAttD * 4);
  p.seq_pieces = reinterpret_cast<int2*>(static_cast<uint8_t*>(workspace) + slot_rows * (kAttD * 4 + 8));
  p.err = err;
  p.B = B;
  p.n = n;
  p.H = H;
  p.Hkv = Hkv;
  p.G = H / Hkv;
  p.Lcap = Lcap;
  p.max_len = max_len;
  p.rows = pl.rows;
  p.unit_rows = pl.tiles * kTaRows;
  p.row_blocks = pl.row_blocks;
  p.ctas = pl.ctas;
  p.pieces_max = pl.pieces_max;
  p.cut = pl.cut;
  p.scale_log2 = scale * 1.4426950408889634f;
  const dim3 grid((unsigned)pl.pieces_max);
  cudaError_t e;
  if (pl.tiles == 2)
    e = launch_attn_tc_t<2>(km, vm, p, grid, stream);
  else
    e = launch_attn_tc_t<1>(km, vm, p, grid, stream);
  if (e != cudaSuccess || !pl.cut) return e;
  const int64_t rows = (int64_t)B * Hkv * pl.rows;
  return launch_pdl(tree_attention_combine_kernel, dim3((unsigned)((rows + 7) / 8)), dim3(256), 0, stream, p);
}

cudaError_t launch_kv_compact(void* k_cache, void* v_cache, const int32_t* lens, const int32_t* parents,
                              const int32_t* node, int B, int n, int Hkv, int D, int Lcap, int layers,
                              int32_t* new_lens, unsigned* err, cudaStream_t stream) {
  return launch_pdl(kv_compact_kernel, dim3((unsigned)B, (unsigned)layers), dim3(kCompactThreads), 0, stream,
                    static_cast<uint4*>(k_cache), static_cast<uint4*>(v_cache), lens, parents, node, B, n, Hkv,
                    D / 8, Lcap, new_lens, err);
}

}  // namespace w4a16
