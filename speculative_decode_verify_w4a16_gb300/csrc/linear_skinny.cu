// W4A16 verify linear, tensor-core fragment path (mma.sync m16n8k16 f16),
// for the sequence-draft token counts (M = 1..15).
//
// out[M][N] = bf16(x[M][K] . W^T) with W = code * scale (int4, group 128).
// Work split: the (row-tile, group) units of the packed weight stream are cut
// into items of contiguous units (sched.cuh); CTA c takes items c, c + C, ...
// (C = grid size) and streams their units through a ring of shared-memory
// stages filled by 1-D bulk copies (TMA engine), so every weight byte is read
// from HBM exactly once.
//
// One CTA per SM: 4 or 5 consumer groups of 4 warps (a warp owns one 32-row
// slice of the 128-row unit) and one producer warp. A ring stage holds one
// unit per group, consecutive units of one tile segment, and group j takes
// unit j, so all the consumer warps of the SM move through the weight stream
// together (four independent CTAs per SM let the hardware's oldest-first
// scheduling starve the youngest, which then finished far behind). The
// groups' sums of a segment meet in shared memory, group 0 stores the tile.
//
// Dequantisation is one AND per pair of codes: the offset-binary code
// o = c + 8 of a nibble at bits 0-3 (16-19) of a 16-bit half is the fp16
// subnormal o * 2^-24, and one at bits 4-7 (20-23) is 16 * o * 2^-24, so a
// packed word gives its four A-fragment registers with one shift and four
// masks (the packed layout puts rows r and r + 8 of a 16-row MMA tile in the
// low and high nibble of each byte; the tensor cores take fp16 subnormal
// operands exactly). The tokens are the fp16 copy x * 2^-e_m made by the
// pre-pass (xprep.cu). The MMA (swap-AB: weight rows are the MMA's M
// dimension, tokens its N = 8) accumulates each 128-wide group in fp32; the
// epilogue removes the offset (2^-24 h * 8 * sum x, h = 1 or 16 by row half,
// from the pre-pass) and applies the fp16 group scale once, in fp32; the
// store multiplies by 2^(24 + e_m) / h.
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


// Stage metadata written by the producer: {item, tile, first group, flags | n << 8}
constexpr int kStItemFirst = 1;  // the stage holds the item's first unit
constexpr int kStSegFirst = 2;   // the stage starts a tile segment of the item
constexpr int kStSegLast = 4;    // the stage ends it

template <int MT8>
struct SkinnyLayout {
  // consumer groups (units per stage) and ring depth: five groups of four
  // warps when the token tile is one MMA wide (more warps hide more latency),
  // four when it is two wide (shared memory)
  static constexpr int kGroups = MT8 == 1 ? 5 : 4;
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
  // the units' offset records: per group, kSkTokenStride fp32 token sums
  static constexpr int kXsBytes = kGroups * kSkTokenStride * 4;
  static constexpr int kXs = (kXsBytes + 127) / 128 * 128;
  static constexpr int kStage = kW + kS + kX + kXs;
  // group sums of a segment end, double-buffered: [2][group 1..3][slice][2*MT8 float4][32 lanes]
  static constexpr int kRedSlot = 2 * MT8 * 32 * 16;
  static constexpr int kRedOff = kStages * kStage;
  static constexpr int kMetaOff = kRedOff + 2 * (kGroups - 1) * kSkConsumerWarps * kRedSlot;
  static constexpr int kBarOff = kMetaOff + kStages * 16;
  // full[stages], empty[stages], red_full[2], red_empty[2]
  static constexpr int kTotal = kBarOff + (2 * kStages + 4) * 8;
  static_assert(kStage % 128 == 0 && kW % 16 == 0 && (kW + kS) % 16 == 0 && kXRowStride % 128 == 32 &&
                    (kW + kS + kX) % 16 == 0,
                "stage alignment");
  static_assert(kTotal <= 227 * 1024, "shared memory");
};

struct SkinnyParams {
  const __half* xh;  // fp16 tokens x * 2^-e_m [M][K] (pre-pass)
  const float* xs;   // offset records [G][kSkTokenStride] (pre-pass)
  const int* xe;     // row exponents e_m [kSkTokenStride] (pre-pass)
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
};

__device__ __forceinline__ void mma_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// One packed word (8 offset-binary nibbles) -> the four fp16x2 A-fragment
// registers: a[0] (row gid, k 4c..4c+1) and a[2] (row gid, k 4c+2..4c+3) hold
// o * 2^-24; a[1] and a[3] (row gid + 8, same k) hold 16 * o * 2^-24.
__device__ __forceinline__ void dequant8(uint32_t w, uint32_t (&a)[4]) {
  const uint32_t w8 = w >> 8;
  a[0] = w & 0x000F000Fu;
  a[1] = w & 0x00F000F0u;
  a[2] = w8 & 0x000F000Fu;
  a[3] = w8 & 0x00F000F0u;
}

// acc (rows gid: 2^-24 * sum c x' * s; rows gid + 8: 16 times that) -> bf16
// outputs x . W^T, i.e. times 2^(24 + e_m) and 2^(20 + e_m).
template <int MT8>
__device__ __forceinline__ void store_tile(const SkinnyParams& p, int64_t t, int warp, int lane,
                                           const float (&acc)[2][MT8][4]) {
  const int gid = lane >> 2, cq = lane & 3;
#pragma unroll
  for (int nt = 0; nt < MT8; ++nt) {
    const int m0 = nt * 8 + 2 * cq;  // < kSkTokenStride: the exponent table is padded
    const int e0 = __ldcg(&p.xe[m0]), e1 = __ldcg(&p.xe[m0 + 1]);
#pragma unroll
    for (int rt = 0; rt < 2; ++rt) {
      const int64_t n_lo = t * kUnitRows + warp * 32 + rt * 16 + gid;
      if (m0 < p.M) {
        p.out[(int64_t)m0 * p.N + n_lo] = __float2bfloat16_rn(ldexpf(acc[rt][nt][0], 24 + e0));
        p.out[(int64_t)m0 * p.N + n_lo + 8] = __float2bfloat16_rn(ldexpf(acc[rt][nt][2], 20 + e0));
      }
      if (m0 + 1 < p.M) {
        p.out[(int64_t)(m0 + 1) * p.N + n_lo] = __float2bfloat16_rn(ldexpf(acc[rt][nt][1], 24 + e1));
        p.out[(int64_t)(m0 + 1) * p.N + n_lo + 8] = __float2bfloat16_rn(ldexpf(acc[rt][nt][3], 20 + e1));
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
#pragma unroll
  for (int rt = 0; rt < 2; ++rt)
#pragma unroll
    for (int nt = 0; nt < MT8; ++nt)
      __stcg(&slot[(rt * MT8 + nt) * 32 + lane],
             make_float4(acc[rt][nt][0], acc[rt][nt][1], acc[rt][nt][2], acc[rt][nt][3]));
  __syncwarp();
  int* counter = &p.counters[kTileCounterBase + t * kSkConsumerWarps + warp];
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
#pragma unroll
      for (int rt = 0; rt < 2; ++rt)
#pragma unroll
        for (int nt = 0; nt < MT8; ++nt)
          v[j][rt][nt] = cc <= cl ? __ldcg(&sl[(rt * MT8 + nt) * 32 + lane]) : make_float4(0.f, 0.f, 0.f, 0.f);
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
  uint64_t* red_full = empty + S;   // [2]: groups 1..3 have written their sums
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
  } else if (threadIdx.x == 32 * kSkProducerWarp && (int)blockIdx.x < p.items) {
    // The packed weights are not written by the kernel this one may overlap:
    // pull the first units of this CTA's first item into L2.
    const int64_t u0 = item_begin(p.sched, blockIdx.x);
    int64_t n = item_begin(p.sched, blockIdx.x + 1) - u0;
    if (n > 2 * S * kSkGroups) n = 2 * S * kSkGroups;
    prefetch_l2(p.qw + u0 * kUnitBytes, (uint32_t)(n * kUnitBytes));
    prefetch_l2(p.sc + u0 * kUnitScaleBytes, (uint32_t)(n * kUnitScaleBytes));
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
    // CTA c takes items c, c + C, ... (C = grid size). The stage copies wait
    // for the preceding grid (x may come from it; issuing the codes earlier
    // and the token rows after would queue a stage's token rows behind
    // several stages of codes, and the L2 prefetch above already moves the
    // first units' codes during that grid's tail).
    if (lane != 0) return;
    grid_dependency_wait();
    const uint64_t pol = policy_evict_first();
    int n_stage = 0;  // stages filled so far
    bool ok = true;
    for (int item = blockIdx.x; ok && item < p.items; item += gridDim.x) {
      const int64_t ub = item_begin(p.sched, item);
      const int64_t ue = item_begin(p.sched, item + 1);
      for (int64_t u = ub; u < ue; ++n_stage) {
        const int64_t t = u / p.G, g0 = u - t * p.G;
        int64_t n = ue - u;
        if (n > kSkGroups) n = kSkGroups;
        if (n > p.G - g0) n = p.G - g0;
        const int st = n_stage % S;
        if (n_stage >= S && !mbar_wait(&empty[st], ((uint32_t)(n_stage / S) & 1u) ^ 1u, p.err)) {
          ok = false;
          break;
        }
        const int flags = (u == ub ? kStItemFirst : 0) | ((u == ub || g0 == 0) ? kStSegFirst : 0) |
                          ((u + n == ue || g0 + n == p.G) ? kStSegLast : 0) | ((int)n << 8);
        meta[st] = make_int4(item, (int)t, (int)g0, flags);
        uint8_t* sb = smem + st * L::kStage;
        const uint32_t nb = (uint32_t)n;
        mbar_arrive_expect_tx(&full[st],
                              nb * (uint32_t)(kUnitBytes + kUnitScaleBytes + p.M * 256 + kSkTokenStride * 4));
        bulk_g2s_hint(sb, p.qw + u * kUnitBytes, nb * kUnitBytes, &full[st], pol);
        bulk_g2s(sb + L::kW, p.sc + u * kUnitScaleBytes, nb * kUnitScaleBytes, &full[st]);
        for (int m = 0; m < p.M; ++m)
          bulk_g2s(sb + L::kW + L::kS + m * kXRowStride, p.xh + (int64_t)m * p.K + g0 * kGroup, nb * 256u, &full[st]);
        bulk_g2s(sb + L::kW + L::kS + L::kX, p.xs + g0 * kSkTokenStride, nb * (uint32_t)(kSkTokenStride * 4),
                 &full[st]);
        u += n;
      }
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
      uint2 xsv[MT8];  // offset sums of this unit's group for tokens m0, m0 + 1 of each token tile
#pragma unroll
      for (int nt = 0; nt < MT8; ++nt)
        xsv[nt] = lds64(sb + L::kW + L::kS + L::kX + grp * (kSkTokenStride * 4) + (nt * 8 + 2 * cq) * 4);

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
          // remove the code offset (h * 2^-24 * 8 * sum x'), then scale: acc += s * (part - h * xs)
          const float xs0 = __uint_as_float(xsv[nt].x), xs1 = __uint_as_float(xsv[nt].y);
          ffma2(part[rt][nt][0], part[rt][nt][1], -1.0f, -1.0f, xs0, xs1);
          ffma2(part[rt][nt][2], part[rt][nt][3], -16.0f, -16.0f, xs0, xs1);
          ffma2(acc[rt][nt][0], acc[rt][nt][1], sc[rt][0], sc[rt][0], part[rt][nt][0], part[rt][nt][1]);
          ffma2(acc[rt][nt][2], acc[rt][nt][3], sc[rt][1], sc[rt][1], part[rt][nt][2], part[rt][nt][3]);
        }
    } else {
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[st]);  // no unit for this group in the stage
    }

    if (flags & kStSegLast) {  // end of this item's segment of tile mt.y: add the groups' sums
      const int rb = n_seg & 1;
      const uint32_t par = (uint32_t)(n_seg >> 1) & 1u;
      if (grp > 0) {
        if (n_seg >= 2 && !mbar_wait(&red_empty[rb], par ^ 1u, p.err)) return;
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

static int skinny_smem(int mt8) { return mt8 == 1 ? SkinnyLayout<1>::kTotal : SkinnyLayout<2>::kTotal; }

static cudaError_t skinny_occupancy_dispatch(int mt8, int* nb) {
  return mt8 == 1 ? skinny_occupancy<1>(nb) : skinny_occupancy<2>(nb);
}

cudaError_t skinny_plan(int M, int64_t N, int64_t K, const DeviceInfo& dev, size_t max_partial_bytes,
                        SkinnyPlan* plan) {
  static int cached_nb[64][3];  // [device][mt8] blocks per SM (0 = unknown)
  if (M < 1 || M >= kTcMinM) return cudaErrorInvalidValue;  // M >= 16 runs on the tcgen05 path
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
  auto up256 = [](size_t v) { return (v + 255) / 256 * 256; };
  plan->xh_off = up256(plan->counter_bytes + plan->partial_bytes);
  plan->xs_off = plan->xh_off + up256((size_t)M * K * 2);
  plan->xe_off = plan->xs_off + up256((size_t)(K / kGroup) * kSkTokenStride * 4);
  plan->total_bytes = plan->xe_off + 256;
  plan->smem_bytes = (size_t)skinny_smem(plan->mt8);
  return cudaSuccess;
}

size_t skinny_workspace_bytes(const SkinnyPlan& plan) { return plan.total_bytes; }

template <int MT8>
static cudaError_t launch_skinny_t(const SkinnyParams& p, const SkinnyPlan& plan, cudaStream_t stream) {
  using L = SkinnyLayout<MT8>;
  return launch_pdl(w4a16_skinny_kernel<MT8>, dim3((unsigned)plan.ctas), dim3(L::kThreads), (size_t)L::kTotal, stream,
                    p);
}

cudaError_t launch_skinny(const void* x, int M, int64_t K, const void* qw_packed, const void* sc_packed, int64_t N,
                          void* out, void* workspace, const SkinnyPlan& plan, const DeviceInfo& dev,
                          cudaStream_t stream) {
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  cudaError_t e = launch_xprep(x, M, K, kSkTokenStride, ws + plan.xh_off, reinterpret_cast<float*>(ws + plan.xs_off),
                               reinterpret_cast<int*>(ws + plan.xe_off), stream);
  if (e != cudaSuccess) return e;
  SkinnyParams p;
  p.xh = reinterpret_cast<const __half*>(ws + plan.xh_off);
  p.xs = reinterpret_cast<const float*>(ws + plan.xs_off);
  p.xe = reinterpret_cast<const int*>(ws + plan.xe_off);
  p.qw = static_cast<const uint8_t*>(qw_packed);
  p.sc = static_cast<const uint8_t*>(sc_packed);
  p.out = static_cast<__nv_bfloat16*>(out);
  p.counters = static_cast<int*>(workspace);
  p.partials = reinterpret_cast<float4*>(static_cast<uint8_t*>(workspace) + plan.counter_bytes);
  p.err = dev.err;
  p.K = K;
  p.N = N;
  p.G = K / kGroup;
  p.M = M;
  p.items = plan.sched.R * plan.sched.C;
  p.sched = plan.sched;
  switch (plan.mt8) {
    case 1: return launch_skinny_t<1>(p, plan, stream);
    case 2: return launch_skinny_t<2>(p, plan, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace w4a16
