// W4A16 verify linear on the 5th-generation tensor cores (tcgen05 + TMEM),
// for the larger verify token counts of a tree draft (M = 16..64).
//
// Same stream-K split of the packed (row-tile, group) units as the
// fragment path. Per unit (128 weight rows x 128 K):
//   producer warp   1-D bulk copies of the packed codes and scales, 2-D TMA
//                   of the token tile x[0:NT, 128g : 128g+128] (128-byte
//                   swizzle; token rows past M read as zero)
//   8 consumer warps  dequantise their 16 rows x 128 K to exact bf16 codes
//                   and store them into TMEM (the UMMA A operand), then, one
//                   unit behind, read the fp32 group product from TMEM and
//                   fold it into registers with the row's fp16 scale
//   MMA warp        8 x tcgen05.mma kind::f16 (M=128 weight rows, N=NT
//                   tokens, K=16) per unit into a TMEM accumulator, commit
// A and D are double-buffered in TMEM so dequantisation of unit i overlaps
// the MMAs of unit i and the scale epilogue of unit i-1.
// A tile split between CTAs is finished by its last contributor, summing the
// fp32 partials in CTA order (deterministic); counters reset themselves.
#include <cudaTypedefs.h>

#include <mutex>

#include "common.cuh"
#include "format.cuh"
#include "internal.h"
#include "tcgen05.cuh"

namespace w4a16 {

constexpr int kTcConsumerWarps = 8;
constexpr int kTcProducerWarp = 8;
constexpr int kTcMmaWarp = 9;
constexpr int kTcThreads = 32 * 10;
constexpr uint32_t kTcTmemCols = 256;  // A: 2 x 64 columns at 0 / 64; D: 2 x NT columns from 128

template <int NT>
struct TcLayout {
  // ring depth: as many stages as two CTAs per SM can hold
  static constexpr int kStages = NT <= 16 ? 8 : (NT <= 32 ? 6 : (NT <= 48 ? 5 : 4));
  // TMEM: 2 A buffers of 64 columns, kDBuf accumulators of NT columns; the
  // epilogue of a unit runs kDBuf - 1 units after its dequantisation so the
  // MMAs have that long to complete before anyone waits for them
  static constexpr int kDBuf = NT <= 32 ? 3 : 2;
  static constexpr int kLag = kDBuf - 1;
  static constexpr int kX = NT * 128;                 // one 64-wide K half of the token tile
  static constexpr int kXOff0 = 0;
  static constexpr int kXOff1 = kX;
  static constexpr int kWOff = 2 * kX;
  static constexpr int kSOff = kWOff + kUnitBytes;
  static constexpr int kStageRaw = kSOff + kUnitScaleBytes;
  static constexpr int kStage = (kStageRaw + 1023) / 1024 * 1024;
  static constexpr int kBarOff = kStages * kStage;
  // full[S], empty[S], a_full[2], mma_done[kDBuf], d_free[kDBuf], tmem base
  static constexpr int kTotal = kBarOff + (2 * kStages + 2 + 2 * kDBuf) * 8 + 16 + 1024;  // +1024: alignment slack
  static_assert(kX % 1024 == 0, "token tile halves must stay 1024-byte aligned");
};

struct DequantConstsTc {
  uint32_t m4, m8, m12;  // 2^28, 2^24, 2^20: multiply-high by these shifts right by 4, 8, 12
};

struct TcParams {
  const uint8_t* qw;
  const uint8_t* sc;
  __nv_bfloat16* out;
  float4* partials;
  int* counters;
  unsigned* err;
  int64_t K, N, U, G, C;
  int M;
  DequantConstsTc dq;
};

__device__ __forceinline__ uint32_t tc_lop3(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}
__device__ __forceinline__ uint32_t tc_mulhi(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("mul.hi.u32 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
__device__ __forceinline__ uint32_t tc_fma_bf16x2(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;
  asm("fma.rn.bf16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}

// One packed word -> the four 16x256b TMEM registers of one 16-wide K step:
// (row g, k 4c..4c+1), (row g, k 4c+2..4c+3), (row g+8, k 4c..), (row g+8, k 4c+2..).
__device__ __forceinline__ void tc_dequant(uint32_t w, const DequantConstsTc& k, uint32_t* r) {
  const uint32_t mask = 0x000F000Fu, magic = 0x43004300u, one = 0x3F803F80u, neg136 = 0xC308C308u;
  r[0] = tc_fma_bf16x2(tc_lop3(w, mask, magic), one, neg136);                     // bits 0/16
  r[2] = tc_fma_bf16x2(tc_lop3(tc_mulhi(w, k.m4), mask, magic), one, neg136);     // bits 4/20
  r[1] = tc_fma_bf16x2(tc_lop3(tc_mulhi(w, k.m8), mask, magic), one, neg136);     // bits 8/24
  r[3] = tc_fma_bf16x2(tc_lop3(tc_mulhi(w, k.m12), mask, magic), one, neg136);    // bits 12/28
}

// Partial-sum slot of one consumer warp: 32 rows x NT/2 fp32, float4-interleaved by lane.
template <int NT>
__device__ __forceinline__ float4* tc_slot(const TcParams& p, int64_t cta, int seg, int warp) {
  return p.partials + ((cta * 2 + seg) * kTcConsumerWarps + warp) * (int64_t)(NT / 8 * 32);
}

template <int NT>
__device__ __forceinline__ void tc_store(const TcParams& p, int64_t t, int q, int h, int lane,
                                         const float (&acc)[NT / 2]) {
  const int64_t n = t * kUnitRows + 32 * q + lane;
#pragma unroll
  for (int j = 0; j < NT / 2; ++j) {
    const int m = h * (NT / 2) + j;
    if (m < p.M) p.out[(int64_t)m * p.N + n] = __float2bfloat16_rn(acc[j]);
  }
}

template <int NT>
__device__ void tc_finish_split(const TcParams& p, int64_t cta, int64_t t, int warp, int lane,
                                const float (&acc)[NT / 2]) {
  const int q = warp & 3, h = warp >> 2;
  const int64_t tile_first = streamk_begin(p.U, p.C, cta) / p.G;
  float4* slot = tc_slot<NT>(p, cta, t == tile_first ? 0 : 1, warp);
#pragma unroll
  for (int j = 0; j < NT / 8; ++j)
    __stcg(&slot[j * 32 + lane], make_float4(acc[4 * j], acc[4 * j + 1], acc[4 * j + 2], acc[4 * j + 3]));
  __threadfence();
  __syncwarp();
  int old = 0;
  if (lane == 0) old = atomicAdd(&p.counters[t * kTcConsumerWarps + warp], 1);
  old = __shfl_sync(0xffffffffu, old, 0);
  const int64_t cf = streamk_owner(p.U, p.C, t * p.G);
  const int64_t cl = streamk_owner(p.U, p.C, t * p.G + p.G - 1);
  if (old != (int)(cl - cf)) return;
  __threadfence();
  float sum[NT / 2];
#pragma unroll
  for (int j = 0; j < NT / 2; ++j) sum[j] = 0.0f;
  constexpr int RB = NT <= 16 ? 4 : (NT <= 32 ? 2 : 1);
  for (int64_t c0 = cf; c0 <= cl; c0 += RB) {
    float4 v[RB][NT / 8];
#pragma unroll
    for (int i = 0; i < RB; ++i) {
      const int64_t cc = c0 + i;
      if (cc <= cl) {
        const int64_t tf = streamk_begin(p.U, p.C, cc) / p.G;
        const float4* sl = tc_slot<NT>(p, cc, t == tf ? 0 : 1, warp);
#pragma unroll
        for (int j = 0; j < NT / 8; ++j) v[i][j] = __ldcg(&sl[j * 32 + lane]);
      }
    }
#pragma unroll
    for (int i = 0; i < RB; ++i)
      if (c0 + i <= cl) {
#pragma unroll
        for (int j = 0; j < NT / 8; ++j) {
          sum[4 * j] += v[i][j].x;
          sum[4 * j + 1] += v[i][j].y;
          sum[4 * j + 2] += v[i][j].z;
          sum[4 * j + 3] += v[i][j].w;
        }
      }
  }
  tc_store<NT>(p, t, q, h, lane, sum);
  if (lane == 0) p.counters[t * kTcConsumerWarps + warp] = 0;
}

template <int NT>
__global__ void __launch_bounds__(kTcThreads, 2) w4a16_tc_kernel(const __grid_constant__ CUtensorMap xmap,
                                                                const TcParams p) {
  using L = TcLayout<NT>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L::kBarOff);
  uint64_t* empty = full + L::kStages;
  uint64_t* a_full = empty + L::kStages;
  uint64_t* mma_done = a_full + 2;
  uint64_t* d_free = mma_done + L::kDBuf;
  uint32_t* tmem_base_s = reinterpret_cast<uint32_t*>(d_free + L::kDBuf);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t cta = blockIdx.x;
  const int64_t u0 = streamk_begin(p.U, p.C, cta);
  const int n_units = (int)(streamk_begin(p.U, p.C, cta + 1) - u0);

  if (threadIdx.x == 0) {
    for (int s = 0; s < L::kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);  // released by the commit of the unit's MMAs
    }
    for (int b = 0; b < 2; ++b) mbar_init(&a_full[b], kTcConsumerWarps);
    for (int b = 0; b < L::kDBuf; ++b) {
      mbar_init(&mma_done[b], 1);
      mbar_init(&d_free[b], kTcConsumerWarps);
    }
    fence_mbarrier_init();
  }
  if (warp == kTcMmaWarp) {
    tmem_alloc(tmem_base_s, kTcTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_base_s;
  const uint32_t a_col[2] = {0u, 64u};
  auto d_col = [](int buf) { return 128u + (uint32_t)(buf * NT); };
  int mma_issued = 0;  // units whose MMAs were committed (MMA warp only)

  if (warp == kTcProducerWarp) {
    // ---------------------------------------------------------- producer
    if (lane == 0) {
      const uint64_t pol = policy_evict_first();
      const uint32_t tx = (uint32_t)(2 * L::kX + kUnitBytes + kUnitScaleBytes);
      int issued = 0;
      bool ok = true;
      int64_t g = u0 % p.G;
      for (int i = 0; i < n_units; ++i, g = (g + 1 == p.G) ? 0 : g + 1) {
        const int s = i % L::kStages;
        if (i >= L::kStages && !mbar_wait(&empty[s], ((uint32_t)(i / L::kStages) & 1u) ^ 1u, p.err)) {
          ok = false;
          break;
        }
        const int64_t u = u0 + i;
        uint8_t* st = smem + s * L::kStage;
        mbar_arrive_expect_tx(&full[s], tx);
        tma_load_2d(st + L::kXOff0, &xmap, (int32_t)(g * kGroup), 0, &full[s]);
        tma_load_2d(st + L::kXOff1, &xmap, (int32_t)(g * kGroup + 64), 0, &full[s]);
        bulk_g2s_hint(st + L::kWOff, p.qw + u * kUnitBytes, kUnitBytes, &full[s], pol);
        bulk_g2s(st + L::kSOff, p.sc + u * kUnitScaleBytes, kUnitScaleBytes, &full[s]);
        issued = i + 1;
      }
      if (!ok)
        for (int i = (issued > L::kStages ? issued - L::kStages : 0); i < issued; ++i)
          mbar_wait(&full[i % L::kStages], (uint32_t)(i / L::kStages) & 1u, p.err);
    }
  } else if (warp == kTcMmaWarp) {
    // ------------------------------------------------------------- MMA
    if (lane == 0) {
      const uint32_t idesc = umma_idesc_bf16(NT);
      for (int i = 0; i < n_units; ++i) {
        const int s = i % L::kStages, b = i & 1, db = i % L::kDBuf;
        if (!mbar_wait(&full[s], (uint32_t)(i / L::kStages) & 1u, p.err)) break;
        if (!mbar_wait(&a_full[b], (uint32_t)(i >> 1) & 1u, p.err)) break;
        if (i >= L::kDBuf && !mbar_wait(&d_free[db], ((uint32_t)(i / L::kDBuf) & 1u) ^ 1u, p.err)) break;
        tc_fence_after();
        const uint32_t xs = smem_u32(smem + s * L::kStage);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint64_t bd = umma_desc_sw128_kmajor(xs + (kk < 4 ? L::kXOff0 : L::kXOff1) + 32 * (kk & 3));
          umma_bf16_ts(tmem + d_col(db), tmem + a_col[b] + 8 * kk, bd, idesc, kk > 0 ? 1u : 0u);
        }
        umma_commit(&mma_done[db]);
        umma_commit(&empty[s]);  // codes were read before a_full, the token tile by these MMAs
        mma_issued = i + 1;
      }
    }
  } else {
    // ------------------------------------------------------- consumers
    const int q = warp & 3, h = warp >> 2;  // TMEM lane quadrant, row-tile / column half
    const int j = lane;                      // row inside the 32-row slice (epilogue)
    const int sc_half = ((q * 8 + (j & 7)) * 2 + (j >> 4)) * 2 + ((j >> 3) & 1);
    float acc[NT / 2];
#pragma unroll
    for (int c = 0; c < NT / 2; ++c) acc[c] = 0.0f;
    float sc_q[L::kLag + 1];  // scales of units i, i-1, .., i-kLag
#pragma unroll
    for (int k = 0; k <= L::kLag; ++k) sc_q[k] = 0.0f;
    int64_t te = u0 / p.G, ge = u0 - te * p.G;  // (tile, group) of the unit in the epilogue
    int64_t seg_g0 = ge;
    for (int i = 0; i < n_units + L::kLag; ++i) {
#pragma unroll
      for (int k = L::kLag; k > 0; --k) sc_q[k] = sc_q[k - 1];
      sc_q[0] = 0.0f;
      if (i < n_units) {
        const int s = i % L::kStages, b = i & 1;
        if (!mbar_wait(&full[s], (uint32_t)(i / L::kStages) & 1u, p.err)) break;
        if (i >= 2) {  // A[b] is free once the MMAs of unit i-2 have completed
          const int e2 = i - 2;
          if (!mbar_wait(&mma_done[e2 % L::kDBuf], (uint32_t)(e2 / L::kDBuf) & 1u, p.err)) break;
          tc_fence_after();
        }
        const uint32_t st = smem_u32(smem + s * L::kStage);
        const uint32_t wb = st + L::kWOff + ((q * 2 + h) * 2) * 512 + lane * 16;
        sc_q[0] = __half2float(__ushort_as_half(
            *reinterpret_cast<const unsigned short*>(smem + s * L::kStage + L::kSOff + 2 * sc_half)));
        const uint32_t ta = tmem + ((uint32_t)(32 * q + 16 * h) << 16) + a_col[b];
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {  // K half: 4 words -> 4 K steps -> 32 TMEM columns
          const uint4 w = lds128(wb + hh * 512);
          uint32_t r[16];
          tc_dequant(w.x, p.dq, &r[0]);
          tc_dequant(w.y, p.dq, &r[4]);
          tc_dequant(w.z, p.dq, &r[8]);
          tc_dequant(w.w, p.dq, &r[12]);
          tmem_st_16x256b_x4(ta + 32 * hh, r);
        }
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&a_full[b]);
      }
      if (i >= L::kLag) {
        // epilogue of unit e = i - kLag
        const int e = i - L::kLag, db = e % L::kDBuf;
        if (!mbar_wait(&mma_done[db], (uint32_t)(e / L::kDBuf) & 1u, p.err)) break;
        tc_fence_after();
        const float sc_e = sc_q[L::kLag];
        const uint32_t dt = tmem + ((uint32_t)(32 * q) << 16) + d_col(db) + h * (NT / 2);
        if constexpr (NT / 2 >= 16) {
#pragma unroll
          for (int c0 = 0; c0 + 16 <= NT / 2; c0 += 16) {
            uint32_t v[16];
            tmem_ld16_sync(dt + c0, v);
#pragma unroll
            for (int c = 0; c < 16; ++c) acc[c0 + c] = fmaf(sc_e, __uint_as_float(v[c]), acc[c0 + c]);
          }
        }
        if constexpr ((NT / 2) % 16 != 0) {
          constexpr int c0 = (NT / 2) / 16 * 16;
          uint32_t v[8];
          tmem_ld8_sync(dt + c0, v);
#pragma unroll
          for (int c = 0; c < 8; ++c) acc[c0 + c] = fmaf(sc_e, __uint_as_float(v[c]), acc[c0 + c]);
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&d_free[db]);
        if (ge == p.G - 1 || e == n_units - 1) {
          if (seg_g0 == 0 && ge == p.G - 1)
            tc_store<NT>(p, te, q, h, lane, acc);
          else
            tc_finish_split<NT>(p, cta, te, warp, lane, acc);
#pragma unroll
          for (int c = 0; c < NT / 2; ++c) acc[c] = 0.0f;
          seg_g0 = 0;
        }
        if (++ge == p.G) {
          ge = 0;
          ++te;
        }
      }
    }
  }

  // ---------------------------------------------------------- teardown
  tc_fence_before();
  __syncthreads();
  if (warp == kTcMmaWarp) {
    if (lane == 0 && mma_issued > 0) {  // normally already observed by the consumers
      const int e = mma_issued - 1;
      mbar_wait(&mma_done[e % L::kDBuf], (uint32_t)(e / L::kDBuf) & 1u, p.err);
    }
    __syncwarp();
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

static int tc_nt(int M) { return (M + 15) / 16 * 16; }

template <int NT>
static int tc_smem() {
  return TcLayout<NT>::kTotal;
}

static int tc_smem_dispatch(int nt) {
  switch (nt) {
    case 16: return tc_smem<16>();
    case 32: return tc_smem<32>();
    case 48: return tc_smem<48>();
    default: return tc_smem<64>();
  }
}

// CTAs per SM, from the shared-memory, register and TMEM budgets (the
// occupancy query under-reports for this kernel, so the limits are applied
// directly).
template <int NT>
static cudaError_t tc_prepare(int device, int* nb) {
  cudaError_t e = cudaFuncSetAttribute(w4a16_tc_kernel<NT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       TcLayout<NT>::kTotal);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(w4a16_tc_kernel<NT>, cudaFuncAttributePreferredSharedMemoryCarveout,
                           cudaSharedmemCarveoutMaxShared);
  if (e != cudaSuccess) return e;
  cudaFuncAttributes fa;
  e = cudaFuncGetAttributes(&fa, w4a16_tc_kernel<NT>);
  if (e != cudaSuccess) return e;
  int smem_sm = 0, smem_reserved = 0, regs_sm = 0;
  if ((e = cudaDeviceGetAttribute(&smem_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, device)) != cudaSuccess)
    return e;
  if ((e = cudaDeviceGetAttribute(&smem_reserved, cudaDevAttrReservedSharedMemoryPerBlock, device)) != cudaSuccess)
    return e;
  if ((e = cudaDeviceGetAttribute(&regs_sm, cudaDevAttrMaxRegistersPerMultiprocessor, device)) != cudaSuccess)
    return e;
  const int by_smem = smem_sm / (TcLayout<NT>::kTotal + (int)fa.sharedSizeBytes + smem_reserved);
  const int regs_cta = ((fa.numRegs * 32 + 255) / 256 * 256) * (kTcThreads / 32);
  const int by_regs = regs_sm / (regs_cta > 0 ? regs_cta : 1);
  const int by_tmem = 512 / (int)kTcTmemCols;
  int n = by_smem < by_regs ? by_smem : by_regs;
  n = n < by_tmem ? n : by_tmem;
  *nb = n;
  return cudaSuccess;
}

cudaError_t tc_plan(int M, int64_t N, int64_t K, const DeviceInfo& dev, TcPlan* plan) {
  static int cached[64][5];
  plan->nt = tc_nt(M);
  plan->units = (N / kUnitRows) * (K / kGroup);
  const int slot = plan->nt / 16;
  int nb = (dev.device >= 0 && dev.device < 64) ? cached[dev.device][slot] : 0;
  if (nb == 0) {
    cudaError_t e;
    switch (plan->nt) {
      case 16: e = tc_prepare<16>(dev.device, &nb); break;
      case 32: e = tc_prepare<32>(dev.device, &nb); break;
      case 48: e = tc_prepare<48>(dev.device, &nb); break;
      default: e = tc_prepare<64>(dev.device, &nb); break;
    }
    if (e != cudaSuccess) return e;
    if (nb < 1) nb = 1;
    if (nb > 2) nb = 2;  // two CTAs x 256 TMEM columns fill the SM's 512
    if (dev.device >= 0 && dev.device < 64) cached[dev.device][slot] = nb;
  }
  int64_t ctas = (int64_t)dev.num_sms * nb;
  if (ctas > plan->units) ctas = plan->units;
  plan->ctas = ctas;
  plan->counter_bytes = kCounterRegionBytes;
  plan->partial_bytes = (size_t)ctas * 2 * kTcConsumerWarps * (plan->nt / 2) * 32 * sizeof(float);
  plan->smem_bytes = (size_t)tc_smem_dispatch(plan->nt);
  return cudaSuccess;
}

size_t tc_workspace_bytes(const TcPlan& plan) { return plan.counter_bytes + plan.partial_bytes; }

template <int NT>
static cudaError_t launch_tc_t(const CUtensorMap& map, const TcParams& p, const TcPlan& plan, cudaStream_t stream) {
  w4a16_tc_kernel<NT><<<(unsigned)plan.ctas, kTcThreads, TcLayout<NT>::kTotal, stream>>>(map, p);
  return cudaGetLastError();
}

cudaError_t launch_tc(const void* x, int M, int64_t K, const void* qw_packed, const void* sc_packed, int64_t N,
                      void* out, void* workspace, const TcPlan& plan, const DeviceInfo& dev, cudaStream_t stream) {
  PFN_cuTensorMapEncodeTiled_v12000 encode = tensor_map_encoder();
  if (!encode) return cudaErrorNotSupported;
  CUtensorMap map;
  const cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)M};
  const cuuint64_t strides[1] = {(cuuint64_t)K * 2};
  const cuuint32_t box[2] = {64u, (cuuint32_t)plan.nt};
  const cuuint32_t es[2] = {1u, 1u};
  if (encode(&map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(x), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;
  TcParams p;
  p.qw = static_cast<const uint8_t*>(qw_packed);
  p.sc = static_cast<const uint8_t*>(sc_packed);
  p.out = static_cast<__nv_bfloat16*>(out);
  p.counters = static_cast<int*>(workspace);
  p.partials = reinterpret_cast<float4*>(static_cast<uint8_t*>(workspace) + plan.counter_bytes);
  p.err = dev.err;
  p.K = K;
  p.N = N;
  p.U = plan.units;
  p.G = K / kGroup;
  p.C = plan.ctas;
  p.M = M;
  p.dq.m4 = 1u << 28;
  p.dq.m8 = 1u << 24;
  p.dq.m12 = 1u << 20;
  switch (plan.nt) {
    case 16: return launch_tc_t<16>(map, p, plan, stream);
    case 32: return launch_tc_t<32>(map, p, plan, stream);
    case 48: return launch_tc_t<48>(map, p, plan, stream);
    case 64: return launch_tc_t<64>(map, p, plan, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace w4a16
