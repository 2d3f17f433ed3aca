// W4A16 verify linear on the 5th-generation tensor cores (tcgen05 + TMEM).
//
// Same item schedule of the packed (row-tile, group) units as the fragment
// path (sched.cuh); one CTA per SM owns the SM's whole tensor memory.
// Warp roles, per unit (128 weight rows x 128 K):
//   producer warp     the CTA's items; 1-D bulk copies of the packed codes
//                     and scales into a deep ring
//   token-tile warp   2-D TMA of the token tile x[0:NT, 128g : 128g+128]
//                     (128-byte swizzle; token rows past M read as zero) into
//                     a ring of kR stages (L2 hits), following the codes ring
//   2 dequant groups  of 4 warps (one per TMEM lane quadrant) take the units
//                     in turn: dequantise the unit to exact bf16 codes and
//                     store them into TMEM, the UMMA A operand; hand the
//                     unit's scales and metadata on to the epilogue
//   2 MMA warps       one per dequant group (its units only): 8 x
//                     tcgen05.mma kind::f16 (M = 128 weight rows, N = NT
//                     tokens, K = 16) per unit into a TMEM accumulator and
//                     one commit. Two issuers keep the tensor pipe fed while
//                     each waits on its barriers.
//   4 epilogue warps  (one per TMEM lane quadrant, all NT tokens) read each
//                     unit's fp32 product from TMEM and fold it into
//                     registers with the row's fp16 group scale; at the end
//                     of a tile segment a 2-D TMA store (or the split-tile
//                     fix-up)
// TMEM holds a ring of kR dequantised units (64 columns each) and kR
// accumulators (NT columns each); consecutive units are dequantised by
// different groups, so the dequantisation of several units, the MMAs of
// another and the epilogues of earlier ones all overlap.
// A tile split between items is finished by its last contributor, which
// adds the fp32 partials of all contributors in item order.
#include <cudaTypedefs.h>
#include <float.h>

#include <mutex>
#include <string.h>

#include "common.cuh"
#include "format.cuh"
#include "internal.h"
#include "sched.cuh"
#include "tcgen05.cuh"

namespace w4a16 {

constexpr int kTcDqGroups = 2;                  // dequant groups of 4 warps, one MMA warp each
constexpr int kTcDqWarps = 4 * kTcDqGroups;     // warps 0 .. 7
constexpr int kTcEpWarps = 4;                   // warps 8 .. 11, one per TMEM lane quadrant
constexpr int kTcProducerWarp = kTcDqWarps + kTcEpWarps;  // warp 12: items, codes + scales
constexpr int kTcMmaWarp0 = kTcProducerWarp + 1;          // warps 13, 14
constexpr int kTcXWarp = kTcMmaWarp0 + kTcDqGroups;       // warp 15: token tiles
constexpr int kTcThreads = 32 * (kTcXWarp + 1);
constexpr uint32_t kTcTmemCols = 512;  // the whole tensor memory of the SM
constexpr int kTcRing = 16;            // scale / metadata hand-off ring (units)

template <int NT, bool FUSED = false>
struct TcLayout {
  // TMEM ring depths: kA dequantised units (64 columns each) at column 0,
  // kD accumulators (NT columns each) after them
  //
  // Every ring below has a multiple of kTcDqGroups slots, so that a slot is
  // always used by units of one dequant group and one MMA warp, in order:
  // each waiter is then at most one phase ahead of the slot's barrier, which
  // a parity wait requires (units are dealt round-robin to the groups).
  //
  // One event releases a unit's A buffer and token tile and hands its
  // accumulator to the epilogue: the completion of the unit's MMAs, one
  // commit per unit to done[i % kR] (each tcgen05.commit costs the tensor
  // pipe about as much as an MMA). kR, the depth of the completion barriers
  // and of the token-tile ring, is a multiple of both TMEM ring depths, so a
  // waiter on done[] for unit i finds the barrier at most one phase ahead
  // (unit i + kR needs slots that unit i's consumers release first).
  // At 80 tokens four accumulators do not fit beside four A buffers; two
  // accumulators are then taken one unit at a time.
  static constexpr int kA = NT <= 16 ? 6 : 4;
  static constexpr int kD = NT <= 16 ? 6 : (NT <= 64 ? 4 : 2);
  static constexpr int kR = kA > kD ? kA : kD;
  static_assert(kR % kA == 0 && kR % kD == 0, "completion barriers shared by the TMEM rings");
  static_assert(kA * 64 + kD * NT <= (int)kTcTmemCols, "TMEM budget");
  static_assert(kA % kTcDqGroups == 0 && kD % kTcDqGroups == 0, "ring slots per group");
  static constexpr bool kPairs = kD >= 4;  // the epilogue takes units in pairs
  // a unit's hand-off entry is rewritten kTcRing units later, by the group
  // that then has finished its previous unit (kTcDqGroups back): that one
  // waited for the MMAs kA units before it, which waited for the epilogue
  // kD units before those
  static_assert(kTcDqGroups + kA + kD <= kTcRing, "hand-off ring depth");
  // Two shared-memory rings: token tiles (read by the MMAs, a few units
  // ahead; they come from L2) and packed codes + scales (read by the dequant
  // groups and released as soon as they are in registers; deep, so that
  // enough HBM reads are in flight).
  static constexpr int kX = NT * 128;             // one 64-wide K half of the token tile
  static constexpr int kXStage = 2 * kX;          // 1024-aligned (swizzled UMMA operand)
  static constexpr int kXStages = kR;
  static constexpr int kWStage = kUnitBytes + kUnitScaleBytes;  // codes, then scales
  static constexpr int kXOff = 0;
  // output staging, one slice per epilogue warp: [NT tokens][32 rows] bf16
  // written to global memory by a 2-D TMA store; in the fused-statistics
  // variant fp32 in the 128-byte swizzle (1024-byte aligned)
  static constexpr int kOutSlice = FUSED ? NT * 32 * 4 : NT * 32 * 2;
  static constexpr int kOutOff = kXOff + kXStages * kXStage;
  static constexpr int kWOff = kOutOff + kTcEpWarps * kOutSlice;
  static constexpr int kWStages = (200 * 1024 - kWOff) / kWStage / kTcDqGroups * kTcDqGroups;
  static constexpr int kScRingOff = kWOff + kWStages * kWStage;       // kTcRing x 256 B scales
  static constexpr int kMetaRingOff = kScRingOff + kTcRing * kUnitScaleBytes;  // kTcRing x int4
  static constexpr int kMetaOff = kMetaRingOff + kTcRing * 16;        // kWStages x int4 (per stage)
  static constexpr int kBarOff = kMetaOff + kWStages * 16;
  // wfull[SW], wempty[SW], xfull[kR], a_full[kR], done[kR], d_free[kR], mma_fin[groups], tmem base
  static constexpr int kTotal = kBarOff + (2 * kWStages + 4 * kR + kTcDqGroups) * 8 + 16 + 1024;  // +1024: alignment
  static_assert(kX % 1024 == 0, "token tile halves must stay 1024-byte aligned");
  static_assert(kOutSlice % 128 == 0, "TMA store source alignment");
  static_assert(!FUSED || (kOutSlice % 1024 == 0 && kOutOff % 1024 == 0), "128-byte swizzle atoms");
  static_assert(kWStage % 16 == 0, "bulk copy alignment");
  static_assert(kWStages >= 2 * kTcDqGroups, "ring depth");
  static_assert(kWStages % kTcDqGroups == 0 && kXStages % kTcDqGroups == 0, "ring slots per group");
};

struct TcParams {
  float* logits;   // fused-statistics variant: fp32 outputs [M][N]
  float2* stats;   // and (max, sum exp(l - max)) per (token, 32-row slice) [M][N/32]
  const uint8_t* qw;
  int tma_store;  // output tiles through the 2-D TMA store (out 16-byte aligned)
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

// Stage metadata written by the producer: the unit's item, tile and group.
constexpr int kTcUnitFirst = 1;  // first unit of its item
constexpr int kTcUnitLast = 2;   // last unit of its item

__device__ __forceinline__ uint32_t tc_lop3(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}
__device__ __forceinline__ uint32_t tc_fma_bf16x2(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;
  asm("fma.rn.bf16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}

// One packed word -> the four 16x256b TMEM registers of one 16-wide K step:
// (row g, k 4c..4c+1), (row g, k 4c+2..4c+3), (row g+8, k 4c..), (row g+8, k 4c+2..).
// (nibble | 0x4300) is the bf16 value 128 + c, and (128 + c) * 1 - 136 = c - 8.
__device__ __forceinline__ void tc_dequant(uint32_t w, uint32_t* r) {
  const uint32_t mask = 0x000F000Fu, magic = 0x43004300u, one = 0x3F803F80u, neg136 = 0xC308C308u;
  r[0] = tc_fma_bf16x2(tc_lop3(w, mask, magic), one, neg136);                     // bits 0/16
  r[2] = tc_fma_bf16x2(tc_lop3(w >> 4, mask, magic), one, neg136);     // bits 4/20
  r[1] = tc_fma_bf16x2(tc_lop3(w >> 8, mask, magic), one, neg136);     // bits 8/24
  r[3] = tc_fma_bf16x2(tc_lop3(w >> 12, mask, magic), one, neg136);    // bits 12/28
}

// Epilogue slice of a warp: rows 32q + lane, tokens 0 .. NT - 1. With the
// TMA store the slice goes through the warp's [NT][32] staging area (token
// rows past M are not written: the tensor map ends at M); otherwise one
// 2-byte store per token. The fused-statistics variant stages fp32 outputs
// the same way (or stores each token's 32 rows as one 128-byte store) and
// reads the staged rows back for the maximum and sum of exp(l - max) of the
// 32 rows per token.
template <int NT, bool FUSED>
__device__ __forceinline__ void tc_store(const TcParams& p, const CUtensorMap* omap, uint8_t* stage, int64_t t, int q,
                                         int lane, const float (&acc)[NT]) {
  const int64_t n = t * kUnitRows + 32 * q + lane;
  if constexpr (FUSED) {
    // staging [NT tokens][32 rows] fp32: 128-byte token rows in the 128-byte
    // swizzle of the TMA store (16-byte chunk c of row m sits at chunk
    // c ^ (m % 8)), so that both the per-token row writes here and the
    // 16-byte reads of whole token rows below are free of bank conflicts
    float* sv = reinterpret_cast<float*>(stage);
    if (p.tma_store && lane == 0) bulk_wait_group_read0();  // the previous store of this area has read it
    __syncwarp();
#pragma unroll
    for (int m = 0; m < NT; ++m) sv[m * 32 + ((((lane >> 2) ^ m) & 7) << 2) + (lane & 3)] = acc[m];
    if (p.tma_store) {
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        tma_store_2d(omap, (int32_t)(t * kUnitRows + 32 * q), 0, stage);
        bulk_commit_group();
      }
    } else {
#pragma unroll
      for (int m = 0; m < NT; ++m)
        if (m < p.M && in_bounds(p.err, (int64_t)m * p.N + n, (int64_t)p.M * p.N)) p.logits[(int64_t)m * p.N + n] = acc[m];
      __syncwarp();
    }
    // lane j: tokens j, j + 32, ... (all rounds interleaved, four independent
    // chains each, so that the latencies overlap); ex2.approx-based
    // exponential, as the accept step's own statistics pass uses for its
    // normalisers (about 1e-7 of the sum)
    constexpr int RN = (NT + 31) / 32;
    const float* row[RN];
    int sw[RN];
    float mx[RN][4], z[RN][4];
#pragma unroll
    for (int j = 0; j < RN; ++j) {
      const int m = min(lane + 32 * j, NT - 1);  // rows past NT: any staged row, not stored
      row[j] = sv + m * 32;
      sw[j] = m & 7;
#pragma unroll
      for (int c = 0; c < 4; ++c) mx[j][c] = -FLT_MAX;
    }
#pragma unroll
    for (int c = 0; c < 8; ++c)
#pragma unroll
      for (int j = 0; j < RN; ++j) {
        const float4 v = *reinterpret_cast<const float4*>(row[j] + ((c ^ sw[j]) << 2));
        mx[j][0] = fmaxf(mx[j][0], v.x);
        mx[j][1] = fmaxf(mx[j][1], v.y);
        mx[j][2] = fmaxf(mx[j][2], v.z);
        mx[j][3] = fmaxf(mx[j][3], v.w);
      }
#pragma unroll
    for (int j = 0; j < RN; ++j) {
      mx[j][0] = fmaxf(fmaxf(mx[j][0], mx[j][1]), fmaxf(mx[j][2], mx[j][3]));
#pragma unroll
      for (int c = 0; c < 4; ++c) z[j][c] = 0.0f;
    }
#pragma unroll
    for (int c = 0; c < 8; ++c)
#pragma unroll
      for (int j = 0; j < RN; ++j) {
        const float4 v = *reinterpret_cast<const float4*>(row[j] + ((c ^ sw[j]) << 2));
        z[j][0] += __expf(v.x - mx[j][0]);
        z[j][1] += __expf(v.y - mx[j][0]);
        z[j][2] += __expf(v.z - mx[j][0]);
        z[j][3] += __expf(v.w - mx[j][0]);
      }
    const int64_t slice = t * 4 + q;
#pragma unroll
    for (int j = 0; j < RN; ++j) {
      const int m = lane + 32 * j;
      if (m < p.M && in_bounds(p.err, (int64_t)m * (p.N / 32) + slice, (int64_t)p.M * (p.N / 32)))
        p.stats[(int64_t)m * (p.N / 32) + slice] = make_float2(mx[j][0], (z[j][0] + z[j][1]) + (z[j][2] + z[j][3]));
    }
    __syncwarp();  // every lane has read the staging area before it is rewritten
    return;
  }
  if (p.tma_store) {
    if (lane == 0) bulk_wait_group_read0();  // the previous store of this area has read it
    __syncwarp();
    __nv_bfloat16* sv = reinterpret_cast<__nv_bfloat16*>(stage);
#pragma unroll
    for (int m = 0; m < NT; ++m) sv[m * 32 + lane] = __float2bfloat16_rn(acc[m]);
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) {
      tma_store_2d(omap, (int32_t)(t * kUnitRows + 32 * q), 0, stage);
      bulk_commit_group();
    }
    return;
  }
#pragma unroll
  for (int m = 0; m < NT; ++m)
    if (m < p.M && in_bounds(p.err, (int64_t)m * p.N + n, (int64_t)p.M * p.N))
      p.out[(int64_t)m * p.N + n] = __float2bfloat16_rn(acc[m]);
}

// Split tiles. Each item that covers part of a tile's K range writes the
// fp32 sums of each epilogue warp's slice (32 rows x NT tokens) to its own
// slot (item, segment, warp) and counts itself in with an atomic per (tile,
// warp); whichever contributor arrives last adds all slots in item order and
// stores the tile: the result does not depend on timing. Counters reset
// themselves for the next call.
template <int NT>
__device__ __forceinline__ float4* tc_slot(const TcParams& p, int item, int seg, int epw) {
  return p.partials + (((int64_t)item * 2 + seg) * kTcEpWarps + epw) * (int64_t)(NT / 4 * 32);
}

template <int NT, bool FUSED>
__device__ void tc_finish_split(const TcParams& p, const CUtensorMap* omap, uint8_t* stage, int item, int seg,
                                int64_t t, int q, int lane, float (&acc)[NT], bool ends_item) {
  const int epw = q;
  constexpr int JB = NT / 4 < 8 ? NT / 4 : 8;  // float4 of a slot per pass (register budget)
  {
    // Fast path: every other contributor has already counted in, so this one
    // is the last. It publishes nothing and adds the others' slots to its own
    // sums in registers. The sum must still run in item order, c_f + c_f+1 +
    // ...: with this contributor first or second that is the same as adding
    // the others, in order, to its own sums (a single fp32 addition is
    // commutative), which saves the slot stores, the releasing atomic and the
    // reload of its own slot. Only a segment that ends its item inside the
    // tile is tested (the item after it began the tile's rest at its start,
    // so this contributor is almost always the last).
    const int64_t ci = kTileCounterBase + t * kTcEpWarps + epw;
    const int64_t t_begin = t * p.G;
    const int cf = item_owner(p.sched, t_begin);
    const int cl = item_owner(p.sched, t_begin + p.G - 1);
    if (ends_item && item - cf <= 1 && in_bounds(p.err, ci, kMaxCounters)) {
      int seen = 0;
      if (lane == 0) seen = ld_acquire_gpu(&p.counters[ci]);
      seen = __shfl_sync(0xffffffffu, seen, 0);
      __syncwarp();
      if (seen == cl - cf) {
        const int seg_cf = item_begin(p.sched, cf) >= t_begin ? 0 : 1;
        for (int cc = cf; cc <= cl; ++cc) {
          if (cc == item) continue;
          const float4* sl = tc_slot<NT>(p, cc, cc == cf ? seg_cf : 0, epw);
          const bool ok = in_bounds(p.err, (sl - p.partials) + NT / 4 * 32 - 1, p.partial_cap);
#pragma unroll
          for (int j0 = 0; j0 < NT / 4; j0 += JB) {
            float4 v[JB];
#pragma unroll
            for (int j = 0; j < JB; ++j) v[j] = ok ? __ldcg(&sl[(j0 + j) * 32 + lane]) : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int j = 0; j < JB; ++j) {
              acc[4 * (j0 + j)] += v[j].x;
              acc[4 * (j0 + j) + 1] += v[j].y;
              acc[4 * (j0 + j) + 2] += v[j].z;
              acc[4 * (j0 + j) + 3] += v[j].w;
            }
          }
        }
        tc_store<NT, FUSED>(p, omap, stage, t, q, lane, acc);
        if (lane == 0) p.counters[ci] = 0;
        return;
      }
    }
  }
  float4* slot = tc_slot<NT>(p, item, seg, epw);
  const bool slot_ok = in_bounds(p.err, (slot - p.partials) + NT / 4 * 32 - 1, p.partial_cap);
#pragma unroll
  for (int j = 0; j < NT / 4; ++j)
    if (slot_ok)
      __stcg(&slot[j * 32 + lane], make_float4(acc[4 * j], acc[4 * j + 1], acc[4 * j + 2], acc[4 * j + 3]));
  __syncwarp();
  const int64_t ci = kTileCounterBase + t * kTcEpWarps + epw;
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
  float sum[NT];
#pragma unroll
  for (int j = 0; j < NT; ++j) sum[j] = 0.0f;
  constexpr int RB = NT <= 16 ? 4 : (NT <= 32 ? 2 : 1);  // contributors loaded together
  for (int c0 = cf; c0 <= cl; c0 += RB) {
#pragma unroll
    for (int j0 = 0; j0 < NT / 4; j0 += JB) {
      float4 v[RB][JB];
#pragma unroll
      for (int r = 0; r < RB; ++r) {
        const int cc = c0 + r;
        const float4* sl = tc_slot<NT>(p, cc, cc == cf ? seg_cf : 0, epw);
        const bool ok = cc <= cl && in_bounds(p.err, (sl - p.partials) + NT / 4 * 32 - 1, p.partial_cap);
#pragma unroll
        for (int j = 0; j < JB; ++j)
          v[r][j] = ok ? __ldcg(&sl[(j0 + j) * 32 + lane]) : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int r = 0; r < RB; ++r)
#pragma unroll
        for (int j = 0; j < JB; ++j) {
          sum[4 * (j0 + j)] += v[r][j].x;
          sum[4 * (j0 + j) + 1] += v[r][j].y;
          sum[4 * (j0 + j) + 2] += v[r][j].z;
          sum[4 * (j0 + j) + 3] += v[r][j].w;
        }
    }
  }
  tc_store<NT, FUSED>(p, omap, stage, t, q, lane, sum);
  if (lane == 0) *counter = 0;
}

// acc[j] += sc * D[lane][col + j], j < W (TMEM columns of this warp's slice;
// W a multiple of 16), up to 32 columns per round trip: a round trip of
// tcgen05.ld + wait::ld costs about 160 cycles however many columns it
// carries (measured on GB300), and the other warps' TMEM traffic does not
// slow the MMAs, so the epilogue of a unit takes as few rounds as the
// registers allow. The accumulator goes back to the MMAs (arrival on
// `release`) as soon as its last columns are in registers: the ring of
// accumulators is the loop that paces the kernel (MMA, completion, epilogue,
// release), and the last multiply-adds need not be inside it.
template <int W>
__device__ __forceinline__ void tc_epilogue_fma(uint32_t dt, float sc, float (&acc)[W], uint64_t* release, int lane) {
#pragma unroll
  for (int c0 = 0; c0 < W; c0 += 32) {
    const int cw = W - c0 < 32 ? W - c0 : 32;
    uint32_t v[32];
#pragma unroll
    for (int j = 0; j < 32; j += 8)
      if (j < cw) tmem_ld_32x32b_x8(dt + c0 + j, *reinterpret_cast<uint32_t(*)[8]>(&v[j]));
    tmem_wait_ld();
    if (c0 + 32 >= W) {
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(release);
    }
#pragma unroll
    for (int c = 0; c < 32; c += 2)
      if (c < cw) ffma2(acc[c0 + c], acc[c0 + c + 1], sc, sc, __uint_as_float(v[c]), __uint_as_float(v[c + 1]));
  }
}

template <int NT, bool FUSED>
__global__ void __launch_bounds__(kTcThreads, 1) w4a16_tc_kernel(const __grid_constant__ CUtensorMap xmap,
                                                                const __grid_constant__ CUtensorMap omap,
                                                                const TcParams p) {
  using L = TcLayout<NT, FUSED>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* wfull = reinterpret_cast<uint64_t*>(smem + L::kBarOff);
  uint64_t* wempty = wfull + L::kWStages;
  uint64_t* xfull = wempty + L::kWStages;
  uint64_t* a_full = xfull + L::kR;
  uint64_t* done = a_full + L::kR;  // unit i's MMAs complete: frees A, x and hands D to the epilogue
  uint64_t* d_free = done + L::kR;
  uint64_t* mma_fin = d_free + L::kR;  // per MMA warp: all its MMAs complete (teardown)
  uint64_t* const xempty = done;
  uint64_t* const a_free = done;
  uint64_t* const mma_done = done;
  uint32_t* tmem_base_s = reinterpret_cast<uint32_t*>(mma_fin + kTcDqGroups);
  int4* meta = reinterpret_cast<int4*>(smem + L::kMetaOff);
  int4* meta_ring = reinterpret_cast<int4*>(smem + L::kMetaRingOff);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  grid_launch_dependents();
  if (threadIdx.x == 0) {
    for (int s = 0; s < L::kWStages; ++s) {
      mbar_init(&wfull[s], 1);
      mbar_init(&wempty[s], 5);  // the dequant group's 4 warps (codes used) + the token-tile warp (g read)
    }
    for (int b = 0; b < L::kR; ++b) {
      mbar_init(&xfull[b], 1);
      mbar_init(&a_full[b], 4);  // the 4 warps of the dequant group
      mbar_init(&done[b], 2);    // commit of the unit's MMAs + the MMA thread's release of the hand-off
      mbar_init(&d_free[b], kTcEpWarps);
    }
    for (int j = 0; j < kTcDqGroups; ++j) mbar_init(&mma_fin[j], 1);
    fence_mbarrier_init();
  }
  if (warp == kTcMmaWarp0) {
    tmem_alloc(tmem_base_s, kTcTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // Programmatic dependent launch: the packed weights and scales are never
  // written by another kernel, so the producer, the dequant groups and the
  // MMA warps start while the preceding grid is still finishing; only the
  // token-tile warp (reads x) and the epilogue (writes out, partials and
  // counters) wait for it.
  const uint32_t tmem = *tmem_base_s;
  auto a_col = [](int buf) { return (uint32_t)(buf * 64); };
  auto d_col = [](int buf) { return (uint32_t)(L::kA * 64 + buf * NT); };
  int mma_issued = 0;  // units whose MMAs were committed (MMA warp only)

  if (warp == kTcProducerWarp) {
    // ---------------------------------------------------------- producer
    // Codes + scales run up to kWStages units ahead of the dequant groups.
    // CTA c takes items c, c + C, ... (C = grid size): fixed before the
    // preceding grid completes, so no claim counter is read here.
    if (lane == 0) {
      const uint64_t pol = policy_evict_first();
      uint32_t n_w = 0;  // units whose codes have been issued
      bool ok = true;
      for (int item = blockIdx.x; ok && item < p.items; item += gridDim.x) {
        const int64_t ub = item_begin(p.sched, item);
        const int64_t ue = item_begin(p.sched, item + 1);
        int64_t t = ub / p.G;
        int64_t g = ub - t * p.G;
        for (int64_t u = ub; u < ue; ++u, ++n_w) {
          const uint32_t s = n_w % L::kWStages;
          if (n_w >= (uint32_t)L::kWStages && !mbar_wait(&wempty[s], ((n_w / L::kWStages) & 1u) ^ 1u, p.err)) {
            ok = false;
            break;
          }
          meta[s] = make_int4(item, (int)t, (int)g, (u == ub ? kTcUnitFirst : 0) | (u == ue - 1 ? kTcUnitLast : 0));
          uint8_t* ws = smem + L::kWOff + s * L::kWStage;
          if (in_bounds(p.err, u, (p.N / kUnitRows) * p.G)) {
            mbar_arrive_expect_tx(&wfull[s], (uint32_t)L::kWStage);
            bulk_g2s_hint(ws, p.qw + u * kUnitBytes, kUnitBytes, &wfull[s], pol);
            bulk_g2s(ws + kUnitBytes, p.sc + u * kUnitScaleBytes, kUnitScaleBytes, &wfull[s]);
          } else {
            mbar_arrive(&wfull[s]);  // bounds-checked builds: the stage without copies
          }
          if (++g == p.G) {
            g = 0;
            ++t;
          }
        }
      }
      // one stop marker per dequant group (each reads every kTcDqGroups-th
      // stage): -1 at the first index past the last unit, where the MMA warp
      // and the epilogue stop too; -2 at the other groups' next indices
      for (int k = 0; ok && k < kTcDqGroups; ++k, ++n_w) {
        const uint32_t s = n_w % L::kWStages;
        if (n_w >= (uint32_t)L::kWStages && !mbar_wait(&wempty[s], ((n_w / L::kWStages) & 1u) ^ 1u, p.err)) {
          ok = false;
          break;
        }
        meta[s] = make_int4(k == 0 ? -1 : -2, 0, 0, 0);
        mbar_arrive(&wfull[s]);
      }
      if (!ok) {  // let copies already in flight land before the CTA exits
        for (uint32_t i = (n_w > (uint32_t)L::kWStages ? n_w - L::kWStages : 0u); i < n_w; ++i)
          mbar_wait(&wfull[i % L::kWStages], (i / L::kWStages) & 1u, p.err);
      }
    }
  } else if (warp == kTcXWarp) {
    // ------------------------------------------------------- token tiles
    // Follows the codes ring: once unit i's codes have landed its group g is
    // known (stage metadata); the token tile goes to the x ring as soon as the
    // MMAs free a slot. Counting in on wempty keeps the stage (and its
    // metadata) from being recycled before it was read here.
    grid_dependency_wait();  // x may be written by the preceding grid
    if (lane == 0) {
      uint32_t n_x = 0;
      for (;; ++n_x) {
        const uint32_t s = n_x % L::kWStages, sx = n_x % L::kXStages;
        const uint32_t pw = (n_x / L::kWStages) & 1u, pe = ((n_x / L::kXStages) & 1u) ^ 1u;
        // both barriers tested at once (one latency); wait in order only if one is still open
        const bool tw = mbar_test(&wfull[s], pw);
        const bool te = mbar_test(&xempty[sx], pe) | (n_x < (uint32_t)L::kXStages);
        if (!tw && !mbar_wait(&wfull[s], pw, p.err)) break;
        const int4 m = meta[s];
        if (m.x < 0) break;  // stop marker
        mbar_arrive(&wempty[s]);
        if (!te && !mbar_wait(&xempty[sx], pe, p.err)) break;
        uint8_t* xs = smem + L::kXOff + sx * L::kXStage;
        mbar_arrive_expect_tx(&xfull[sx], (uint32_t)L::kXStage);
        tma_load_2d(xs, &xmap, m.z * kGroup, 0, &xfull[sx]);
        tma_load_2d(xs + L::kX, &xmap, m.z * kGroup + 64, 0, &xfull[sx]);
      }
      // let token tiles in flight land before the CTA exits (normally the MMAs
      // have consumed them all already)
      for (uint32_t i = (n_x > (uint32_t)L::kXStages ? n_x - L::kXStages : 0u); i < n_x; ++i)
        mbar_wait(&xfull[i % L::kXStages], (i / L::kXStages) & 1u, p.err);
    }
  } else if (warp >= kTcMmaWarp0) {
    // ------------------------------------------------------------- MMA
    // MMA warp j issues the units of dequant group j (i = j, j + 2, ...).
    // The group waited for the unit's stage before it arrived on a_full, so
    // the token tile is in shared memory once a_full completes.
    const uint32_t idesc = umma_idesc_bf16(NT);
    for (uint32_t i = warp - kTcMmaWarp0;; i += kTcDqGroups) {
      const uint32_t sx = i % L::kXStages, b = i % L::kA, db = i % L::kD, cb = i % L::kR;
      const uint32_t pa = (i / L::kA) & 1u, pd = ((i / L::kD) & 1u) ^ 1u, px = (i / L::kXStages) & 1u;
      int st = 1;  // 1: go on, 0: a wait ran out, 2: stop marker
      if (lane == 0) {
        // the three barriers tested at once (one latency); waits in order only
        // for those still open (the token tile after the stop check)
        const bool ta = mbar_test(&a_full[b], pa);
        const bool td = mbar_test(&d_free[db], pd) | (i < (uint32_t)L::kD);
        const bool tx = mbar_test(&xfull[sx], px);
        if ((!ta && !mbar_wait(&a_full[b], pa, p.err)) || (!td && !mbar_wait(&d_free[db], pd, p.err))) {
          st = 0;
        } else {
          const int mk = meta_ring[i % kTcRing].x;  // written by the group before a_full
          if (mk < 0) {  // stop marker
            if (mk == -1) {  // the epilogue's last index: complete its phase without MMAs
              mbar_arrive(&mma_done[cb]);
              mbar_arrive(&mma_done[cb]);
            }
            st = 2;
          } else if (!tx && !mbar_wait(&xfull[sx], px, p.err)) {
            st = 0;
          }
        }
      }
      st = __shfl_sync(0xffffffffu, st, 0);
      __syncwarp();
      if (st != 1) break;
      tc_fence_after();
      const uint64_t bd0 = umma_desc_sw128_kmajor(smem_u32(smem + L::kXOff + sx * L::kXStage));
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        // start-address field (bits 0..13, 16-byte units) of the K step's rows
        const uint64_t bd = bd0 + (uint64_t)(((kk < 4 ? 0 : L::kX) + 32 * (kk & 3)) >> 4);
        umma_bf16_ts_warp(tmem + d_col(db), tmem + a_col(b) + 8 * kk, bd, idesc, kk > 0 ? 1u : 0u);
      }
      umma_commit_warp(&done[cb]);  // frees A[b] and the token tile (cb == sx), hands D[db] to the epilogue
      // release (to the epilogue) of the hand-off entry lane 0 acquired through a_full
      if (lane == 0) mbar_arrive(&done[cb]);
      mma_issued = (int)i + 1;
    }
    if (mma_issued > 0) umma_commit_warp(&mma_fin[warp - kTcMmaWarp0]);  // tracks all of this warp's MMAs
  } else if (warp < kTcDqWarps) {
    // ------------------------------------------------------ dequant groups
    const int grp = warp >> 2, q = warp & 3;
    for (uint32_t i = grp;; i += kTcDqGroups) {
      const uint32_t s = i % L::kWStages, b = i % L::kA;
      // A[b] is free once the MMAs of unit i - kA have completed
      const uint32_t ia = i - (uint32_t)L::kA, fb = ia % L::kR;
      const uint32_t pw = (i / L::kWStages) & 1u, pa = (ia / L::kR) & 1u;
      // both barriers tested at once, waits only for one still open
      const bool tw = mbar_test(&wfull[s], pw);
      const bool ta = i < (uint32_t)L::kA || mbar_test(&a_free[fb], pa);
      if (!tw && !mbar_wait(&wfull[s], pw, p.err)) break;
      const uint4 mu = lds128(smem_u32(&meta[s]));
      const bool stop = (int)mu.x < 0;
      if (stop) {
        if (!ta && !mbar_wait(&a_free[fb], pa, p.err)) break;
        // forward the marker to this group's MMA warp (and through it to the
        // epilogue, which stops at the first one)
        if (q == 0 && lane == 0) meta_ring[i % kTcRing] = make_int4((int)mu.x, 0, 0, 0);
        __syncwarp();
        if (lane == 0) mbar_arrive(&a_full[b]);
        break;
      }
      const uint32_t st = smem_u32(smem + L::kWOff + s * L::kWStage);
      if (q == 0) {  // hand the unit's scales and metadata on to the epilogue
        if (lane < kUnitScaleBytes / 16) {
          const uint4 v = lds128(st + kUnitBytes + lane * 16);
          *reinterpret_cast<uint4*>(smem + L::kScRingOff + (i % kTcRing) * kUnitScaleBytes + lane * 16) = v;
        }
        if (lane == 0) meta_ring[i % kTcRing] = make_int4((int)mu.x, (int)mu.y, (int)mu.z, (int)mu.w);
      }
      uint4 w[2][2];  // this warp's 32 rows
#pragma unroll
      for (int rt = 0; rt < 2; ++rt)
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) w[rt][hh] = lds128(st + (((q * 2 + rt) * 2 + hh) * 32 + lane) * 16);
      // the whole unit is dequantised into registers before A[b] is needed,
      // so the arithmetic overlaps the MMAs that still read A[b]
      uint32_t r[2][2][16];  // 16 rows x 64 K -> 16 lanes x 32 TMEM columns, per (rt, hh)
#pragma unroll
      for (int rt = 0; rt < 2; ++rt)
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          tc_dequant(w[rt][hh].x, &r[rt][hh][0]);
          tc_dequant(w[rt][hh].y, &r[rt][hh][4]);
          tc_dequant(w[rt][hh].z, &r[rt][hh][8]);
          tc_dequant(w[rt][hh].w, &r[rt][hh][12]);
        }
      // every code and scale of the stage has been used, so its loads have
      // completed: release it to the producer
      __syncwarp();
      if (lane == 0) mbar_arrive(&wempty[s]);
      if (!ta && !mbar_wait(&a_free[fb], pa, p.err)) break;
#pragma unroll
      for (int rt = 0; rt < 2; ++rt)
#pragma unroll
        for (int hh = 0; hh < 2; ++hh)
          tmem_st_16x256b_x4(tmem + ((uint32_t)(32 * q + 16 * rt) << 16) + a_col(b) + 32 * hh, r[rt][hh]);
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&a_full[b]);
    }
  } else if (warp < kTcDqWarps + kTcEpWarps) {
    // ------------------------------------------------------------ epilogue
    grid_dependency_wait();  // out, partials and counters may still be in use by the preceding grid
    const int q = warp & 3;  // TMEM lane quadrant
    const int sc_half = ((q * 8 + (lane & 7)) * 2 + (lane >> 4)) * 2 + ((lane >> 3) & 1);  // row 32q + lane
    float acc[NT];
#pragma unroll
    for (int c = 0; c < NT; ++c) acc[c] = 0.0f;
    int item = 0, item_t0 = 0, seg_g0 = 0;
    auto scale_of = [&](uint32_t u) {
      return __half2float(__ushort_as_half(*reinterpret_cast<const unsigned short*>(
          smem + L::kScRingOff + (u % kTcRing) * kUnitScaleBytes + 2 * sc_half)));
    };
    auto meta_of = [&](uint32_t u) {
      const uint4 mu = lds128(smem_u32(&meta_ring[u % kTcRing]));
      return make_int4((int)mu.x, (int)mu.y, (int)mu.z, (int)mu.w);
    };
    // Units are taken two at a time (one barrier round trip for both) unless
    // the first one ends a tile segment or the second is the stop marker;
    // one at a time with two accumulators, which a pair would both hold.
    for (uint32_t e = 0;;) {
      const uint32_t db = e % L::kD, db1 = (e + 1) % L::kD;
      const uint32_t cb = e % L::kR, cb1 = (e + 1) % L::kR;
      const uint32_t p0 = (e / L::kR) & 1u, p1 = ((e + 1) / L::kR) & 1u;
      // both accumulators tested at once; waits only for one still open
      const bool t0 = mbar_test(&mma_done[cb], p0);
      const bool t1 = L::kPairs && mbar_test(&mma_done[cb1], p1);
      if (!t0 && !mbar_wait(&mma_done[cb], p0, p.err)) break;
      const int4 me = meta_of(e);
      if (me.x < 0) break;  // stop marker
      if (me.w & kTcUnitFirst) {
        item = me.x;
        item_t0 = me.y;
        seg_g0 = me.z;
      }
      const bool seg_end = me.z == p.G - 1 || (me.w & kTcUnitLast);
      bool pair = false;
      int4 me1 = me;
      if (L::kPairs && !seg_end) {
        if (!t1 && !mbar_wait(&mma_done[cb1], p1, p.err)) break;
        me1 = meta_of(e + 1);
        pair = me1.x >= 0;
      }
      tc_fence_after();
      const uint32_t dt = tmem + ((uint32_t)(32 * q) << 16);
      tc_epilogue_fma<NT>(dt + d_col(db), scale_of(e), acc, &d_free[db], lane);  // unit e first, then e + 1
      if (pair) tc_epilogue_fma<NT>(dt + d_col(db1), scale_of(e + 1), acc, &d_free[db1], lane);
      const int4 ml = pair ? me1 : me;  // last unit taken
      if (ml.z == p.G - 1 || (ml.w & kTcUnitLast)) {  // end of this item's segment of tile ml.y
        if (seg_g0 == 0 && ml.z == p.G - 1)
          tc_store<NT, FUSED>(p, &omap, smem + L::kOutOff + q * L::kOutSlice, ml.y, q, lane, acc);
        else
          tc_finish_split<NT, FUSED>(p, &omap, smem + L::kOutOff + q * L::kOutSlice, item, ml.y == item_t0 ? 0 : 1,
                                     ml.y, q, lane, acc, ml.z != p.G - 1);
#pragma unroll
        for (int c = 0; c < NT; ++c) acc[c] = 0.0f;
        seg_g0 = 0;
      }
      if (L::kPairs && !pair && !seg_end) break;  // the second unit was the stop marker
      e += pair ? 2u : 1u;
    }
  }

  // ---------------------------------------------------------- teardown
  if (warp >= kTcDqWarps && warp < kTcDqWarps + kTcEpWarps && lane == 0 && p.tma_store)
    bulk_wait_group0();  // this warp's output tiles are written
  tc_fence_before();
  __syncthreads();
  if (warp >= kTcMmaWarp0 && warp < kTcMmaWarp0 + kTcDqGroups && lane == 0 && mma_issued > 0)
    mbar_wait(&mma_fin[warp - kTcMmaWarp0], 0u, p.err);  // no MMA in flight when TMEM is freed
  tc_fence_before();
  __syncthreads();
  if (warp == kTcMmaWarp0) {
    tc_fence_after();
    tmem_dealloc(tmem, kTcTmemCols);
  }
}

// ------------------------------------------------------------------ host

static PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  });
  return fn;
}

void* tensor_map_encode_fn() { return reinterpret_cast<void*>(tensor_map_encoder()); }

static int tc_nt(int M) { return (M + 15) / 16 * 16; }

// CTAs per SM, from the shared-memory, register and TMEM budgets (the
// occupancy query under-reports for this kernel, so the limits are applied
// directly); also sets the kernel's shared-memory attributes.
template <int NT, bool FUSED>
static cudaError_t tc_prepare(int device, int* nb) {
  using L = TcLayout<NT, FUSED>;
  cudaError_t e =
      cudaFuncSetAttribute(w4a16_tc_kernel<NT, FUSED>, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kTotal);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(w4a16_tc_kernel<NT, FUSED>, cudaFuncAttributePreferredSharedMemoryCarveout,
                           cudaSharedmemCarveoutMaxShared);
  if (e != cudaSuccess) return e;
  cudaFuncAttributes fa;
  e = cudaFuncGetAttributes(&fa, w4a16_tc_kernel<NT, FUSED>);
  if (e != cudaSuccess) return e;
  int smem_sm = 0, smem_reserved = 0, regs_sm = 0;
  if ((e = cudaDeviceGetAttribute(&smem_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, device)) != cudaSuccess)
    return e;
  if ((e = cudaDeviceGetAttribute(&smem_reserved, cudaDevAttrReservedSharedMemoryPerBlock, device)) != cudaSuccess)
    return e;
  if ((e = cudaDeviceGetAttribute(&regs_sm, cudaDevAttrMaxRegistersPerMultiprocessor, device)) != cudaSuccess)
    return e;
  const int by_smem = smem_sm / (L::kTotal + (int)fa.sharedSizeBytes + smem_reserved);
  const int regs_cta = ((fa.numRegs * 32 + 255) / 256 * 256) * (kTcThreads / 32);
  const int by_regs = regs_sm / (regs_cta > 0 ? regs_cta : 1);
  const int by_tmem = 512 / (int)kTcTmemCols;  // 1: the kernel takes the whole tensor memory
  int n = by_smem < by_regs ? by_smem : by_regs;
  n = n < by_tmem ? n : by_tmem;
  *nb = n;
  return cudaSuccess;
}

template <bool FUSED>
static cudaError_t tc_prepare_dispatch(int nt, int device, int* nb, int* smem) {
  switch (nt) {
    case 16: *smem = TcLayout<16, FUSED>::kTotal; return tc_prepare<16, FUSED>(device, nb);
    case 32: *smem = TcLayout<32, FUSED>::kTotal; return tc_prepare<32, FUSED>(device, nb);
    case 48: *smem = TcLayout<48, FUSED>::kTotal; return tc_prepare<48, FUSED>(device, nb);
    case 64: *smem = TcLayout<64, FUSED>::kTotal; return tc_prepare<64, FUSED>(device, nb);
    case 80: *smem = TcLayout<80, FUSED>::kTotal; return tc_prepare<80, FUSED>(device, nb);
    default: return cudaErrorInvalidValue;
  }
}

static cudaError_t tc_plan_impl(int M, int64_t N, int64_t K, const DeviceInfo& dev, bool fused, TcPlan* plan) {
  static int cached[64][2][6];  // [device][fused][nt / 16]: CTAs per SM (0 = unknown)
  static int cached_smem[2][6];
  plan->nt = tc_nt(M);
  if (plan->nt > kTcMaxM) return cudaErrorInvalidValue;
  plan->units = (N / kUnitRows) * (K / kGroup);
  const int slot = plan->nt / 16;
  int nb = (dev.device >= 0 && dev.device < 64) ? cached[dev.device][fused][slot] : 0;
  int smem = cached_smem[fused][slot];
  if (nb == 0) {
    cudaError_t e = fused ? tc_prepare_dispatch<true>(plan->nt, dev.device, &nb, &smem)
                          : tc_prepare_dispatch<false>(plan->nt, dev.device, &nb, &smem);
    if (e != cudaSuccess) return e;
    if (nb < 1) nb = 1;
    if (nb > 1) nb = 1;  // one CTA owns the SM's 512 TMEM columns
    if (dev.device >= 0 && dev.device < 64) cached[dev.device][fused][slot] = nb;
    cached_smem[fused][slot] = smem;
  }
  int64_t ctas = (int64_t)dev.num_sms * nb;
  if (ctas > plan->units) ctas = plan->units;
  plan->ctas = ctas;
  // partial slots: 2 segments x 128 rows x NT fp32 per item. A split costs
  // 4*NT*128 bytes of partials written and read again (at M = 64, four units'
  // worth of weight bytes), so this path keeps one round: every CTA one
  // contiguous run of units, at most two split tiles per CTA.
  const size_t per_item = (size_t)2 * plan->nt * kUnitRows * sizeof(float);
  plan->sched = make_item_sched(plan->units, (int)ctas, 1, 1);
  plan->counter_bytes = kCounterRegionBytes;
  plan->partial_bytes = (size_t)plan->sched.R * ctas * per_item;
  plan->smem_bytes = (size_t)smem;
  return cudaSuccess;
}

cudaError_t tc_plan(int M, int64_t N, int64_t K, const DeviceInfo& dev, size_t max_partial_bytes, TcPlan* plan) {
  (void)max_partial_bytes;
  return tc_plan_impl(M, N, K, dev, false, plan);
}

cudaError_t tc_plan_fused(int M, int64_t N, int64_t K, const DeviceInfo& dev, TcPlan* plan) {
  return tc_plan_impl(M, N, K, dev, true, plan);
}

size_t tc_workspace_bytes(const TcPlan& plan) { return plan.counter_bytes + plan.partial_bytes; }

template <int NT, bool FUSED>
static cudaError_t launch_tc_t(const CUtensorMap& map, const CUtensorMap& omap, const TcParams& p, const TcPlan& plan,
                               cudaStream_t stream) {
  return launch_pdl(w4a16_tc_kernel<NT, FUSED>, dim3((unsigned)plan.ctas), dim3(kTcThreads),
                    (size_t)TcLayout<NT, FUSED>::kTotal, stream, map, omap, p);
}

template <bool FUSED>
static cudaError_t launch_tc_dispatch(const CUtensorMap& map, const CUtensorMap& omap, const TcParams& p,
                                      const TcPlan& plan, cudaStream_t stream) {
  switch (plan.nt) {
    case 16: return launch_tc_t<16, FUSED>(map, omap, p, plan, stream);
    case 32: return launch_tc_t<32, FUSED>(map, omap, p, plan, stream);
    case 48: return launch_tc_t<48, FUSED>(map, omap, p, plan, stream);
    case 64: return launch_tc_t<64, FUSED>(map, omap, p, plan, stream);
    case 80: return launch_tc_t<80, FUSED>(map, omap, p, plan, stream);
    default: return cudaErrorInvalidValue;
  }
}

// Shared part of both launches: the token tensor map and the kernel parameters.
static cudaError_t tc_setup(const void* x, int M, int64_t K, const void* qw_packed, const void* sc_packed, int64_t N,
                            void* workspace, const TcPlan& plan, const DeviceInfo& dev, CUtensorMap* map, TcParams* p) {
  PFN_cuTensorMapEncodeTiled_v12000 encode = tensor_map_encoder();
  if (!encode) return cudaErrorNotSupported;
  const cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)M};
  const cuuint64_t strides[1] = {(cuuint64_t)K * 2};
  const cuuint32_t box[2] = {64u, (cuuint32_t)plan.nt};
  const cuuint32_t es[2] = {1u, 1u};
  if (encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(x), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;
  memset(p, 0, sizeof(*p));
  p->qw = static_cast<const uint8_t*>(qw_packed);
  p->sc = static_cast<const uint8_t*>(sc_packed);
  p->counters = static_cast<int*>(workspace);
  p->partials = reinterpret_cast<float4*>(static_cast<uint8_t*>(workspace) + plan.counter_bytes);
  p->err = dev.err;
  p->K = K;
  p->N = N;
  p->G = K / kGroup;
  p->M = M;
  p->items = plan.sched.R * plan.sched.C;
  p->sched = plan.sched;
  p->partial_cap = (int64_t)(plan.partial_bytes / sizeof(float4));
  return cudaSuccess;
}

cudaError_t launch_tc(const void* x, int M, int64_t K, const void* qw_packed, const void* sc_packed, int64_t N,
                      void* out, void* workspace, const TcPlan& plan, const DeviceInfo& dev, cudaStream_t stream) {
  CUtensorMap map;
  TcParams p;
  cudaError_t e = tc_setup(x, M, K, qw_packed, sc_packed, N, workspace, plan, dev, &map, &p);
  if (e != cudaSuccess) return e;
  // output tiles: [M][N] bf16, boxes of 32 rows (n) x NT tokens (m); the TMA
  // store wants a 16-byte aligned base, else the kernel stores per element
  CUtensorMap omap;
  memset(&omap, 0, sizeof(omap));
  if ((reinterpret_cast<uintptr_t>(out) & 15) == 0) {
    const cuuint64_t odims[2] = {(cuuint64_t)N, (cuuint64_t)M};
    const cuuint64_t ostrides[1] = {(cuuint64_t)N * 2};
    const cuuint32_t obox[2] = {32u, (cuuint32_t)plan.nt};
    const cuuint32_t es[2] = {1u, 1u};
    if (tensor_map_encoder()(&omap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, out, odims, ostrides, obox, es,
                             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS)
      p.tma_store = 1;
  }
  p.out = static_cast<__nv_bfloat16*>(out);
  return launch_tc_dispatch<false>(map, omap, p, plan, stream);
}

cudaError_t launch_tc_fused(const void* x, int M, int64_t K, const void* qw_packed, const void* sc_packed, int64_t N,
                            float* logits, float2* stats, void* workspace, const TcPlan& plan, const DeviceInfo& dev,
                            cudaStream_t stream) {
  CUtensorMap map;
  TcParams p;
  cudaError_t e = tc_setup(x, M, K, qw_packed, sc_packed, N, workspace, plan, dev, &map, &p);
  if (e != cudaSuccess) return e;
  // fp32 output tiles: [M][N], boxes of 32 rows (n, 128 bytes) x NT tokens,
  // 128-byte swizzle; per element when the base is not 16-byte aligned
  CUtensorMap omap;
  memset(&omap, 0, sizeof(omap));
  if ((reinterpret_cast<uintptr_t>(logits) & 15) == 0) {
    const cuuint64_t odims[2] = {(cuuint64_t)N, (cuuint64_t)M};
    const cuuint64_t ostrides[1] = {(cuuint64_t)N * 4};
    const cuuint32_t obox[2] = {32u, (cuuint32_t)plan.nt};
    const cuuint32_t es[2] = {1u, 1u};
    if (tensor_map_encoder()(&omap, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, logits, odims, ostrides, obox, es,
                             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS)
      p.tma_store = 1;
  }
  p.logits = logits;
  p.stats = stats;
  return launch_tc_dispatch<true>(map, omap, p, plan, stream);
}

}  // namespace w4a16
