// W4A16 verify linear, tensor-core fragment path (mma.sync m16n8k16 bf16),
// for the sequence-draft token counts (M = 1..8).
//
// out[M][N] = bf16(x[M][K] . W^T) with W = code * scale (int4, group 128).
// Work split: the (row-tile, group) units of the packed weight stream are cut
// into items of contiguous units (sched.cuh); CTA c takes items c, c + C, ...
// (C = grid size) and streams their units through a ring of shared-memory
// stages filled by 1-D bulk copies (TMA engine), so every weight byte is read
// from HBM exactly once.
//
// One CTA per SM: 6 consumer groups of 4 warps (a warp owns one 32-row
// slice of the 128-row unit) and one producer warp. A ring stage holds one
// unit per group, consecutive units of one tile segment, and group j takes
// unit j, so all the consumer warps of the SM move through the weight stream
// together (four independent CTAs per SM let the hardware's oldest-first
// scheduling starve the youngest, which then finished far behind). The
// groups' sums of a segment meet in shared memory, group 0 stores the tile.
// A consumer dequantises 16 packed words per unit into
// exact bf16 codes (offset-binary nibble OR'ed into the mantissa of 128.0,
// then 136 subtracted: a bit trick in the spirit of Kim et al. 2022, "Who
// Says Elephants Can't Run", arXiv:2211.10017), multiplies them with the
// token fragments on the tensor cores (swap-AB: weight rows are the MMA's M
// dimension, tokens its N = 8), accumulates the group in fp32 and applies
// the fp16 group scale once in fp32.
//
// A tile covered by one item is stored directly; a tile whose K range is
// split between items is finished by its last contributor, which adds the
// fp32 partials of all contributors in item order: the result does not
// depend on timing. Counters reset themselves for the next call.
#include "common.cuh"
#include "format.cuh"
#include "internal.h"
#include "sched.cuh"

namespace w4a16 {

constexpr int kSkConsumerWarps = 4;  // warps of a group: one 32-row slice each

#if W4A16_TEST_HOOKS
// Debug builds only: the producer of CTA 0 leaves out the ring stage with
// this index (no copies, no arrival), so that the consumers' bounded wait on
// it runs out and the kernel reports a timeout. -1: off.
__device__ int g_test_skip_stage = -1;
__device__ __forceinline__ bool test_skip_stage(int n_stage) {
  return blockIdx.x == 0 && n_stage == *(volatile int*)&g_test_skip_stage;
}
#else
__device__ __forceinline__ bool test_skip_stage(int) { return false; }
#endif


// Stage metadata written by the producer: {item, tile, first group, flags | n << 8}
constexpr int kStItemFirst = 1;  // the stage holds the item's first unit
constexpr int kStSegFirst = 2;   // the stage starts a tile segment of the item
constexpr int kStSegLast = 4;    // the stage ends it

template <int MT8>
struct SkinnyLayout {
  // consumer groups (units per stage) and ring depth: six groups of four
  // warps when the token tile is one MMA wide (25 warps x 80 registers fill
  // the register file; more warps hide more latency), four when it is two
  // wide (shared memory)
  static constexpr int kGroups = MT8 == 1 ? 6 : 4;
  static constexpr int kStages = 3;
  static constexpr int kConsumers = kGroups * kSkConsumerWarps;  // warps 0 .. kConsumers - 1
  static constexpr int kProducerWarp = kConsumers;               // the last warp
  static constexpr int kThreads = 32 * (kConsumers + 1);
  // bytes per token row of a stage's token tile: the units' 128-wide K
  // slices side by side + padding, so rows fall 32 bytes apart mod 128
  static constexpr int kXRowStride = kGroups * 256 + 32;
  static constexpr int kW = kGroups * kUnitBytes;       // codes of the stage's units
  static constexpr int kS = kGroups * kUnitScaleBytes;  // their scales
  static constexpr int kX = MT8 * 8 * kXRowStride;      // token rows
  static constexpr int kStage = kW + kS + kX;
  // group sums of a segment end: [kRedBufs][group 1..kGroups-1][slice][2*MT8 float4][32 lanes]
  // (one buffer: segment ends are many stages apart, so the groups never
  // wait for group 0 to have read the previous segment's sums)
  static constexpr int kRedBufs = 1;
  static constexpr int kRedSlot = 2 * MT8 * 32 * 16;
  static constexpr int kRedOff = kStages * kStage;
  static constexpr int kMetaOff = kRedOff + kRedBufs * (kGroups - 1) * kSkConsumerWarps * kRedSlot;
  static constexpr int kBarOff = kMetaOff + kStages * 16;
  // full[stages], empty[stages], red_full[2], red_empty[2]
  static constexpr int kTotal = kBarOff + (2 * kStages + 4) * 8;
  static_assert(kStage % 128 == 0 && kW % 16 == 0 && (kW + kS) % 16 == 0 && kXRowStride % 128 == 32,
                "stage alignment");
  static_assert(kTotal <= 227 * 1024, "shared memory");
};

struct SkinnyParams {
  const __nv_bfloat16* x;
  const uint8_t* qw;
  const uint8_t* sc;
  __nv_bfloat16* out;
  float4* partials;  // split-tile partial slots
  int* counters;     // split-tile counters
  unsigned* err;
  int64_t K, N, G;
  int M;
  int items;  // R * C
  ItemSched sched;
  int64_t partial_cap;  // float4 slots in partials (bounds-checked builds)
};

__device__ __forceinline__ void mma_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t lop3_and_or(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(a), "r"(b), "r"(c));  // (a & b) | c
  return d;
}

__device__ __forceinline__ uint32_t fma_bf16x2(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;
  asm("fma.rn.bf16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}

// 8 offset-binary nibbles -> four bf16x2 registers of exact signed codes:
// (nibble | 0x4300) is the bf16 value 128 + c, and (128 + c) * 1 - 136 = c - 8.
__device__ __forceinline__ void dequant8(uint32_t w, uint32_t (&a)[4]) {
  const uint32_t mask = 0x000F000Fu, magic = 0x43004300u;
  const uint32_t one = 0x3F803F80u, neg136 = 0xC308C308u;
  a[0] = fma_bf16x2(lop3_and_or(w, mask, magic), one, neg136);
  a[1] = fma_bf16x2(lop3_and_or(w >> 4, mask, magic), one, neg136);
  a[2] = fma_bf16x2(lop3_and_or(w >> 8, mask, magic), one, neg136);
  a[3] = fma_bf16x2(lop3_and_or(w >> 12, mask, magic), one, neg136);
}

template <int MT8>
__device__ __forceinline__ void store_tile(const SkinnyParams& p, int64_t t, int warp, int lane,
                                           const float (&acc)[2][MT8][4]) {
  const int gid = lane >> 2, cq = lane & 3;
#pragma unroll
  for (int rt = 0; rt < 2; ++rt) {
    const int64_t n_lo = t * kUnitRows + warp * 32 + rt * 16 + gid;
#pragma unroll
    for (int nt = 0; nt < MT8; ++nt) {
      const int m0 = nt * 8 + 2 * cq;
      const int64_t mn = (int64_t)p.M * p.N;
      if (m0 < p.M && in_bounds(p.err, (int64_t)m0 * p.N + n_lo + 8, mn)) {
        p.out[(int64_t)m0 * p.N + n_lo] = __float2bfloat16_rn(acc[rt][nt][0]);
        p.out[(int64_t)m0 * p.N + n_lo + 8] = __float2bfloat16_rn(acc[rt][nt][2]);
      }
      if (m0 + 1 < p.M && in_bounds(p.err, (int64_t)(m0 + 1) * p.N + n_lo + 8, mn)) {
        p.out[(int64_t)(m0 + 1) * p.N + n_lo] = __float2bfloat16_rn(acc[rt][nt][1]);
        p.out[(int64_t)(m0 + 1) * p.N + n_lo + 8] = __float2bfloat16_rn(acc[rt][nt][3]);
      }
    }
  }
}

// Split tiles. Each item that covers part of a tile's K range writes its
// fp32 sums to its own slot (item, segment, warp) and counts itself in with
// an atomic per (tile, warp); whichever contributor arrives last adds all
// slots in item order and stores the tile: the result does not depend on
// timing. Counters reset themselves for the next call.
template <int MT8>
__device__ __forceinline__ float4* partial_slot(const SkinnyParams& p, int item, int seg, int warp) {
  return p.partials + (((int64_t)item * 2 + seg) * kSkConsumerWarps + warp) * (int64_t)(2 * MT8 * 32);
}

template <int MT8>
__device__ void finish_split_tile(const SkinnyParams& p, int item, int seg, int64_t t, int warp, int lane,
                                  const float (&acc)[2][MT8][4]) {
  float4* slot = partial_slot<MT8>(p, item, seg, warp);
  const bool slot_ok = in_bounds(p.err, (slot - p.partials) + 2 * MT8 * 32 - 1, p.partial_cap);
#pragma unroll
  for (int rt = 0; rt < 2; ++rt)
#pragma unroll
    for (int nt = 0; nt < MT8; ++nt)
      if (slot_ok)
        __stcg(&slot[(rt * MT8 + nt) * 32 + lane],
               make_float4(acc[rt][nt][0], acc[rt][nt][1], acc[rt][nt][2], acc[rt][nt][3]));
  __syncwarp();
  const int64_t ci = kTileCounterBase + t * kSkConsumerWarps + warp;
  if (!in_bounds(p.err, ci, kMaxCounters)) return;
  int* counter = &p.counters[ci];
  int old = 0;
  if (lane == 0) old = atomic_add_acq_rel(counter, 1);
  old = __shfl_sync(0xffffffffu, old, 0);
  const int64_t t_begin = t * p.G;
  const int cf = item_owner(p.sched, t_begin);
  const int cl = item_owner(p.sched, t_begin + p.G - 1);
  if (old != cl - cf) return;  // not the last contributor
  __syncwarp();
  // only the first contributor can have started in an earlier tile (its
  // partial for this tile is then its segment 1)
  const int seg_cf = item_begin(p.sched, cf) >= t_begin ? 0 : 1;
  float sum[2][MT8][4];
#pragma unroll
  for (int rt = 0; rt < 2; ++rt)
#pragma unroll
    for (int nt = 0; nt < MT8; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) sum[rt][nt][e] = 0.0f;
  constexpr int RB = MT8 == 1 ? 4 : 2;  // contributors loaded together (one L2 round trip)
  for (int c0 = cf; c0 <= cl; c0 += RB) {
    float4 v[RB][2][MT8];
#pragma unroll
    for (int j = 0; j < RB; ++j) {
      const int cc = c0 + j;
      const float4* sl = partial_slot<MT8>(p, cc, cc == cf ? seg_cf : 0, warp);
      const bool ok = cc <= cl && in_bounds(p.err, (sl - p.partials) + 2 * MT8 * 32 - 1, p.partial_cap);
#pragma unroll
      for (int rt = 0; rt < 2; ++rt)
#pragma unroll
        for (int nt = 0; nt < MT8; ++nt)
          v[j][rt][nt] = ok ? __ldcg(&sl[(rt * MT8 + nt) * 32 + lane]) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int j = 0; j < RB; ++j)
#pragma unroll
      for (int rt = 0; rt < 2; ++rt)
#pragma unroll
        for (int nt = 0; nt < MT8; ++nt) {
          sum[rt][nt][0] += v[j][rt][nt].x;
          sum[rt][nt][1] += v[j][rt][nt].y;
          sum[rt][nt][2] += v[j][rt][nt].z;
          sum[rt][nt][3] += v[j][rt][nt].w;
        }
  }
  store_tile<MT8>(p, t, warp, lane, sum);
  if (lane == 0) *counter = 0;
}

template <int MT8>
__global__ void __launch_bounds__(SkinnyLayout<MT8>::kThreads, 1) w4a16_skinny_kernel(const SkinnyParams p) {
  using L = SkinnyLayout<MT8>;
  constexpr int S = L::kStages;
  constexpr int kSkGroups = L::kGroups;
  constexpr int kSkConsumers = L::kConsumers;
  constexpr int kSkProducerWarp = L::kProducerWarp;
  constexpr int kXRowStride = L::kXRowStride;
  extern __shared__ __align__(128) uint8_t smem[];
  int4* meta = reinterpret_cast<int4*>(smem + L::kMetaOff);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L::kBarOff);
  uint64_t* empty = full + S;
  uint64_t* red_full = empty + S;   // [kRedBufs used]: groups 1.. have written their sums
  uint64_t* red_empty = red_full + 2;  // [2]: group 0 has read them
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  grid_launch_dependents();
  if (threadIdx.x == 0) {
    for (int st = 0; st < S; ++st) {
      mbar_init(&full[st], 1);
      mbar_init(&empty[st], kSkConsumers);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&red_full[b], (kSkGroups - 1) * kSkConsumerWarps);
      mbar_init(&red_empty[b], kSkConsumerWarps);
    }
    fence_mbarrier_init();
  }
  // token rows M .. 8*MT8-1 of every stage are never copied: zero them once
  {
    constexpr int kChunks = kXRowStride / 16;
    const int zrows = MT8 * 8 - p.M;
    for (int idx = threadIdx.x; idx < S * zrows * kChunks; idx += blockDim.x) {
      const int st = idx / (zrows * kChunks), r = (idx / kChunks) % zrows, c16 = idx % kChunks;
      *reinterpret_cast<uint4*>(smem + st * L::kStage + L::kW + L::kS + (p.M + r) * kXRowStride + c16 * 16) =
          make_uint4(0u, 0u, 0u, 0u);
    }
  }
  __syncthreads();

  if (warp == kSkProducerWarp) {
    // ---------------------------------------------------------- producer
    // A stage takes up to kSkGroups consecutive units of one tile segment of
    // the item: codes, scales and each token row's K range are contiguous in
    // global memory, so a stage is 2 + M bulk copies.
    // CTA c takes items c, c + C, ... (C = grid size). The packed weights are
    // never written by the kernel this one may overlap, so the first ring
    // stages' codes and scales go out at once, before the grid dependency
    // resolves; their token rows (x may come from that kernel) follow after
    // it, on the same stage barrier. Measured in a CUDA graph of back-to-back
    // verify linears, this beat both waiting first and an L2 prefetch of the
    // first units (which delayed the first stage's own copies).
    if (lane != 0) return;
    const uint64_t pol = policy_evict_first();
    int n_stage = 0;  // stages filled so far
    bool ok = true;
    int item = blockIdx.x;
    int64_t ub = 0, ue = 0, u = 0;
    if (item < p.items) {
      ub = item_begin(p.sched, item);
      ue = item_begin(p.sched, item + 1);
      u = ub;
    }
    // the stage's units and token columns lie inside the packed weights and x
    auto stage_in_bounds = [&](int64_t u0, int64_t g0, int64_t n) {
      return in_bounds(p.err, u0 + n - 1, (p.N / kUnitRows) * p.G) &&
             in_bounds(p.err, (int64_t)(p.M - 1) * p.K + (g0 + n) * kGroup - 1, (int64_t)p.M * p.K);
    };
    // one stage: up to kSkGroups units of the current tile segment; returns the units taken
    auto stage_codes = [&](int st, int64_t& g0_out, bool skip) -> int64_t {
      const int64_t t = u / p.G, g0 = u - t * p.G;
      int64_t n = ue - u;
      if (n > kSkGroups) n = kSkGroups;
      if (n > p.G - g0) n = p.G - g0;
      const int flags = (u == ub ? kStItemFirst : 0) | ((u == ub || g0 == 0) ? kStSegFirst : 0) |
                        ((u + n == ue || g0 + n == p.G) ? kStSegLast : 0) | ((int)n << 8);
      meta[st] = make_int4(item, (int)t, (int)g0, flags);
      g0_out = g0;
      if (skip) return n;
      uint8_t* sb = smem + st * L::kStage;
      const uint32_t nb = (uint32_t)n;
      if (!stage_in_bounds(u, g0, n)) {  // bounds-checked builds: complete the stage without copies
        mbar_arrive(&full[st]);
        return n;
      }
      mbar_arrive_expect_tx(&full[st], nb * (uint32_t)(kUnitBytes + kUnitScaleBytes + p.M * 256));
      bulk_g2s_hint(sb, p.qw + u * kUnitBytes, nb * kUnitBytes, &full[st], pol);
      bulk_g2s(sb + L::kW, p.sc + u * kUnitScaleBytes, nb * kUnitScaleBytes, &full[st]);
      return n;
    };
    auto stage_tokens = [&](int st, int64_t u0, int64_t g0, int64_t n) {
      if (!stage_in_bounds(u0, g0, n)) return;  // the stage went without copies
      uint8_t* sb = smem + st * L::kStage;
      for (int m = 0; m < p.M; ++m)
        bulk_g2s(sb + L::kW + L::kS + m * kXRowStride, p.x + (int64_t)m * p.K + g0 * kGroup, (uint32_t)n * 256u,
                 &full[st]);
    };
    int64_t early_g0[S], early_n[S], early_u[S];
    int n_early = 0;
    while (n_early < S && item < p.items && u < ue) {
      early_u[n_early] = u;
      early_n[n_early] = stage_codes(n_early, early_g0[n_early], false);
      u += early_n[n_early];
      ++n_early;
      ++n_stage;
    }
    grid_dependency_wait();
    for (int i = 0; i < n_early; ++i) stage_tokens(i, early_u[i], early_g0[i], early_n[i]);
    while (ok && item < p.items) {
      if (u >= ue) {  // next item of this CTA
        item += gridDim.x;
        if (item >= p.items) break;
        ub = item_begin(p.sched, item);
        ue = item_begin(p.sched, item + 1);
        u = ub;
        continue;
      }
      const int st = n_stage % S;
      if (n_stage >= S && !mbar_wait(&empty[st], ((uint32_t)(n_stage / S) & 1u) ^ 1u, p.err)) {
        ok = false;
        break;
      }
      int64_t g0;
      const bool skip = test_skip_stage(n_stage);
      const int64_t n = stage_codes(st, g0, skip);
      if (!skip) stage_tokens(st, u, g0, n);
      u += n;
      ++n_stage;
    }
    if (ok) {  // stop marker for the consumers
      const int st = n_stage % S;
      if (n_stage < S || mbar_wait(&empty[st], ((uint32_t)(n_stage / S) & 1u) ^ 1u, p.err)) {
        meta[st] = make_int4(-1, 0, 0, 0);
        mbar_arrive(&full[st]);
      }
    } else {  // let copies already in flight land before the CTA exits
      for (int i = (n_stage > S ? n_stage - S : 0); i < n_stage; ++i)
        mbar_wait(&full[i % S], (uint32_t)(i / S) & 1u, p.err);
    }
    return;
  }

  // ------------------------------------------------------------ consumers
  grid_dependency_wait();  // out, partials and counters may still be in use by the preceding grid
  const int grp = warp >> 2, q = warp & 3;  // group (unit of the stage), 32-row slice
  const int gid = lane >> 2, cq = lane & 3;
  float acc[2][MT8][4];
#pragma unroll
  for (int rt = 0; rt < 2; ++rt)
#pragma unroll
    for (int nt = 0; nt < MT8; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) acc[rt][nt][e] = 0.0f;
  int item = 0, item_t0 = 0, seg_g0 = 0, n_seg = 0;

  for (int i = 0;; ++i) {
    const int st = i % S;
    if (!mbar_wait(&full[st], (uint32_t)(i / S) & 1u, p.err)) return;
    const uint32_t sb = smem_u32(smem + st * L::kStage);
    const uint4 mu = lds128(smem_u32(&meta[st]));
    const int4 mt = make_int4((int)mu.x, (int)mu.y, (int)mu.z, (int)mu.w);
    if (mt.x < 0) break;
    const int flags = mt.w & 0xff, n = mt.w >> 8;
    if (flags & kStItemFirst) {
      item = mt.x;
      item_t0 = mt.y;
    }
    if (flags & kStSegFirst) seg_g0 = mt.z;
    if (grp < n) {
      const uint32_t wb = sb + grp * kUnitBytes + q * 2048 + lane * 16;
      uint4 wq[2][2];
#pragma unroll
      for (int rt = 0; rt < 2; ++rt)
#pragma unroll
        for (int h = 0; h < 2; ++h) wq[rt][h] = lds128(wb + (rt * 2 + h) * 512);
      const uint2 sc2 = lds64(sb + L::kW + grp * kUnitScaleBytes + (q * 8 + gid) * 8);

      float part[2][MT8][4];
#pragma unroll
      for (int rt = 0; rt < 2; ++rt)
#pragma unroll
        for (int nt = 0; nt < MT8; ++nt)
#pragma unroll
          for (int e = 0; e < 4; ++e) part[rt][nt][e] = 0.0f;

      const uint32_t xb = sb + L::kW + L::kS + gid * kXRowStride + grp * 256 + cq * 8;
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        uint2 b[MT8];
#pragma unroll
        for (int nt = 0; nt < MT8; ++nt) b[nt] = lds64(xb + nt * 8 * kXRowStride + kk * 32);
#pragma unroll
        for (int rt = 0; rt < 2; ++rt) {
          const uint4 q4 = wq[rt][kk >> 2];
          const uint32_t word = (kk & 3) == 0 ? q4.x : (kk & 3) == 1 ? q4.y : (kk & 3) == 2 ? q4.z : q4.w;
          uint32_t a[4];
          dequant8(word, a);
#pragma unroll
          for (int nt = 0; nt < MT8; ++nt) mma_16816(part[rt][nt], a, b[nt].x, b[nt].y);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[st]);

      const __half2 s_rt0 = *reinterpret_cast<const __half2*>(&sc2.x);
      const __half2 s_rt1 = *reinterpret_cast<const __half2*>(&sc2.y);
      const float sc[2][2] = {{__low2float(s_rt0), __high2float(s_rt0)}, {__low2float(s_rt1), __high2float(s_rt1)}};
#pragma unroll
      for (int rt = 0; rt < 2; ++rt)
#pragma unroll
        for (int nt = 0; nt < MT8; ++nt) {
          ffma2(acc[rt][nt][0], acc[rt][nt][1], sc[rt][0], sc[rt][0], part[rt][nt][0], part[rt][nt][1]);
          ffma2(acc[rt][nt][2], acc[rt][nt][3], sc[rt][1], sc[rt][1], part[rt][nt][2], part[rt][nt][3]);
        }
    } else {
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[st]);  // no unit for this group in the stage
    }

    if (flags & kStSegLast) {  // end of this item's segment of tile mt.y: add the groups' sums
      const int rb = n_seg % L::kRedBufs;
      const uint32_t par = (uint32_t)(n_seg / L::kRedBufs) & 1u;
      if (grp > 0) {
        if (n_seg >= L::kRedBufs && !mbar_wait(&red_empty[rb], par ^ 1u, p.err)) return;
        float4* slot = reinterpret_cast<float4*>(
            smem + L::kRedOff + ((rb * (kSkGroups - 1) + grp - 1) * kSkConsumerWarps + q) * L::kRedSlot);
#pragma unroll
        for (int rt = 0; rt < 2; ++rt)
#pragma unroll
          for (int nt = 0; nt < MT8; ++nt)
            slot[(rt * MT8 + nt) * 32 + lane] = make_float4(acc[rt][nt][0], acc[rt][nt][1], acc[rt][nt][2], acc[rt][nt][3]);
        __syncwarp();
        if (lane == 0) mbar_arrive(&red_full[rb]);
      } else {
        if (!mbar_wait(&red_full[rb], par, p.err)) return;
#pragma unroll
        for (int g = 1; g < kSkGroups; ++g) {  // groups in order: the sum does not depend on timing
          const float4* slot = reinterpret_cast<const float4*>(
              smem + L::kRedOff + ((rb * (kSkGroups - 1) + g - 1) * kSkConsumerWarps + q) * L::kRedSlot);
#pragma unroll
          for (int rt = 0; rt < 2; ++rt)
#pragma unroll
            for (int nt = 0; nt < MT8; ++nt) {
              const float4 v = slot[(rt * MT8 + nt) * 32 + lane];
              acc[rt][nt][0] += v.x;
              acc[rt][nt][1] += v.y;
              acc[rt][nt][2] += v.z;
              acc[rt][nt][3] += v.w;
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&red_empty[rb]);
        if (seg_g0 == 0 && mt.z + n - 1 == p.G - 1)
          store_tile<MT8>(p, mt.y, q, lane, acc);
        else
          finish_split_tile<MT8>(p, item, mt.y == item_t0 ? 0 : 1, mt.y, q, lane, acc);
      }
#pragma unroll
      for (int rt = 0; rt < 2; ++rt)
#pragma unroll
        for (int nt = 0; nt < MT8; ++nt)
#pragma unroll
          for (int e = 0; e < 4; ++e) acc[rt][nt][e] = 0.0f;
      ++n_seg;
    }
  }
}

// ------------------------------------------------------------------ host

template <int MT8>
static cudaError_t skinny_occupancy(int* blocks_per_sm) {
  using L = SkinnyLayout<MT8>;
  cudaError_t e =
      cudaFuncSetAttribute(w4a16_skinny_kernel<MT8>, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kTotal);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(w4a16_skinny_kernel<MT8>, cudaFuncAttributePreferredSharedMemoryCarveout,
                           cudaSharedmemCarveoutMaxShared);
  if (e != cudaSuccess) return e;
  return cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks_per_sm, w4a16_skinny_kernel<MT8>, L::kThreads,
                                                      L::kTotal);
}

// token tiles of 8: the fragment path serves M = 1..8 (one tile); the
// tcgen05 path takes M >= 9
static int skinny_smem(int) { return SkinnyLayout<1>::kTotal; }

static cudaError_t skinny_occupancy_dispatch(int mt8, int* nb) {
  return mt8 == 1 ? skinny_occupancy<1>(nb) : cudaErrorInvalidValue;
}

cudaError_t skinny_plan(int M, int64_t N, int64_t K, const DeviceInfo& dev, size_t max_partial_bytes,
                        SkinnyPlan* plan) {
  static int cached_nb[64][3];  // [device][mt8] blocks per SM (0 = unknown)
  if (M < 1 || M >= kTcMinM) return cudaErrorInvalidValue;  // M >= 9 runs on the tcgen05 path
  plan->mt8 = (M + 7) / 8;
  plan->units = (N / kUnitRows) * (K / kGroup);
  int nb = 0;
  if (dev.device >= 0 && dev.device < 64) nb = cached_nb[dev.device][plan->mt8];
  if (nb == 0) {
    cudaError_t e = skinny_occupancy_dispatch(plan->mt8, &nb);
    if (e != cudaSuccess) return e;
    if (nb < 1) nb = 1;
    if (nb > 1) nb = 1;  // one CTA per SM: its 4 consumer groups share the SM's stream
    if (dev.device >= 0 && dev.device < 64) cached_nb[dev.device][plan->mt8] = nb;
  }
  int64_t ctas = (int64_t)dev.num_sms * nb;
  if (ctas > plan->units) ctas = plan->units;
  plan->ctas = ctas;
  // partial slots: 2 segments x 4 slices x (32 rows x 8*MT8 tokens) fp32 per
  // item. Every split tile costs its contributors a partial store and an
  // atomic round trip, so this path keeps one round: every CTA one contiguous
  // run of units, at most two split tiles per CTA.
  (void)max_partial_bytes;
  const size_t per_item = (size_t)2 * kSkConsumerWarps * 2 * plan->mt8 * 32 * sizeof(float4);
  plan->sched = make_item_sched(plan->units, (int)ctas, 1, 1);
  plan->counter_bytes = kCounterRegionBytes;
  plan->partial_bytes = (size_t)plan->sched.R * ctas * per_item;
  plan->smem_bytes = (size_t)skinny_smem(plan->mt8);
  return cudaSuccess;
}

size_t skinny_workspace_bytes(const SkinnyPlan& plan) { return plan.counter_bytes + plan.partial_bytes; }

template <int MT8>
static cudaError_t launch_skinny_t(const SkinnyParams& p, const SkinnyPlan& plan, cudaStream_t stream) {
  using L = SkinnyLayout<MT8>;
  return launch_pdl(w4a16_skinny_kernel<MT8>, dim3((unsigned)plan.ctas), dim3(L::kThreads), (size_t)L::kTotal, stream,
                    p);
}

cudaError_t launch_skinny(const void* x, int M, int64_t K, const void* qw_packed, const void* sc_packed, int64_t N,
                          void* out, void* workspace, const SkinnyPlan& plan, const DeviceInfo& dev,
                          cudaStream_t stream) {
  SkinnyParams p;
  p.x = static_cast<const __nv_bfloat16*>(x);
  p.qw = static_cast<const uint8_t*>(qw_packed);
  p.sc = static_cast<const uint8_t*>(sc_packed);
  p.out = static_cast<__nv_bfloat16*>(out);
  p.counters = static_cast<int*>(workspace);
  p.partials = reinterpret_cast<float4*>(static_cast<uint8_t*>(workspace) + plan.counter_bytes);
  p.partial_cap = (int64_t)(plan.partial_bytes / sizeof(float4));
  p.err = dev.err;
  p.K = K;
  p.N = N;
  p.G = K / kGroup;
  p.M = M;
  p.items = plan.sched.R * plan.sched.C;
  p.sched = plan.sched;
  switch (plan.mt8) {
    case 1: return launch_skinny_t<1>(p, plan, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace w4a16

#if W4A16_TEST_HOOKS
// Debug builds only (not part of the C ABI header): see g_test_skip_stage.
extern "C" int w4a16_test_set_skip_stage(int n_stage) {
  return (int)cudaMemcpyToSymbol(w4a16::g_test_skip_stage, &n_stage, sizeof(int));
}
#endif
