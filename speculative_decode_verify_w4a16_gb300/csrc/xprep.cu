// Token pre-pass of the fragment-path linear: x (bf16) -> the fp16 operand the
// tensor cores multiply with the 4-bit codes, plus what the epilogue needs to
// undo the code offset and the scaling.
//
// The fragment path feeds the offset-binary codes o = c + 8 to the MMA as fp16
// subnormals (o * 2^-24 is the bit pattern o itself), so one AND per pair of
// codes replaces the whole dequantisation. The activations must then be fp16
// as well (both MMA operands have one type). Per token row m:
//   e_m   = the power of two that puts max_k |x[m,k]| in [2^14, 2^15)
//   xh    = fp16_rn(x * 2^-e_m): exact for every value within 2^28 of the row
//           maximum (bf16 has 8 significant bits, fp16 11); smaller values
//           round to fp16 subnormals (absolute error <= 2^(e_m - 25))
//   xs    = 2^-21 * sum_{k in group g} xh[m,k] (fp32, a fixed pairwise order):
//           the MMA sums 2^-24 * (c + 8) * xh, so subtracting xs (in the same
//           units) leaves 2^-24 * sum c * xh.
// Rows M .. MP-1 of the group records are written as zeros.
#include "common.cuh"
#include "internal.h"

namespace w4a16 {

constexpr int kXpThreads = 256;
constexpr int kXpGroupsPerBlock = kXpThreads / 32;  // one warp per (row, group)

// Grid (ceil(G / 8), MP): block (b, m) converts groups 8b .. 8b + 7 of row m.
// Every block first takes the maximum of the whole row itself (16-byte loads,
// eight per thread in flight at once; a row of the verify shapes is at most
// 56 KB and comes from L2), so no block waits for another.
__global__ void __launch_bounds__(kXpThreads) xprep_kernel(const __nv_bfloat16* __restrict__ x, int M, int64_t K,
                                                          int MP, __half* __restrict__ xh, float* __restrict__ xs,
                                                          int* __restrict__ xe) {
  grid_launch_dependents();
  grid_dependency_wait();  // x may come from the preceding grid, and its readers of xh / xs must be done
  const int m = blockIdx.y;
  const int64_t G = K / 128;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t g = (int64_t)blockIdx.x * kXpGroupsPerBlock + warp;
  if (m >= M) {  // padding token: zero records
    if (g < G && lane == 0) xs[g * MP + m] = 0.0f;
    if (blockIdx.x == 0 && threadIdx.x == 0) xe[m] = 0;
    return;
  }
  const __nv_bfloat16* row = x + (int64_t)m * K;
  // row maximum of |x|: K / 8 chunks of 16 bytes, up to 8 per thread issued together
  constexpr int kU = 8;
  float amax = 0.0f;
  for (int64_t c0 = 0; c0 < K / 8; c0 += (int64_t)kXpThreads * kU) {
    uint4 v[kU];
#pragma unroll
    for (int j = 0; j < kU; ++j) {
      const int64_t c = c0 + (int64_t)j * kXpThreads + threadIdx.x;
      v[j] = c < K / 8 ? __ldcg(reinterpret_cast<const uint4*>(row) + c) : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int j = 0; j < kU; ++j) {
      const uint32_t w[4] = {v[j].x, v[j].y, v[j].z, v[j].w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        amax = fmaxf(amax, fabsf(__uint_as_float(w[i] << 16)));
        amax = fmaxf(amax, fabsf(__uint_as_float(w[i] & 0xFFFF0000u)));
      }
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  __shared__ float wmax[kXpThreads / 32];
  if (lane == 0) wmax[warp] = amax;
  __syncthreads();
  amax = wmax[0];
#pragma unroll
  for (int i = 1; i < kXpThreads / 32; ++i) amax = fmaxf(amax, wmax[i]);
  int e = 0;
  if (amax > 0.0f && amax <= 3.4028235e38f) {
    int E;
    (void)frexpf(amax, &E);  // amax = f * 2^E, f in [0.5, 1)
    e = E - 15;              // amax * 2^-e in [2^14, 2^15)
  }
  if (blockIdx.x == 0 && threadIdx.x == 0) xe[m] = e;
  if (g >= G) return;
  // lane l converts k = 128g + 4l .. 4l + 3; the warp sums the group
  const uint2 v = __ldcg(reinterpret_cast<const uint2*>(row + g * 128 + lane * 4));
  const float f0 = ldexpf(__uint_as_float(v.x << 16), -e);
  const float f1 = ldexpf(__uint_as_float(v.x & 0xFFFF0000u), -e);
  const float f2 = ldexpf(__uint_as_float(v.y << 16), -e);
  const float f3 = ldexpf(__uint_as_float(v.y & 0xFFFF0000u), -e);
  const __half2 h01 = __floats2half2_rn(f0, f1);
  const __half2 h23 = __floats2half2_rn(f2, f3);
  uint2 o;
  o.x = *reinterpret_cast<const uint32_t*>(&h01);
  o.y = *reinterpret_cast<const uint32_t*>(&h23);
  *reinterpret_cast<uint2*>(xh + (int64_t)m * K + g * 128 + lane * 4) = o;
  float s = (__low2float(h01) + __high2float(h01)) + (__low2float(h23) + __high2float(h23));
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
  if (lane == 0) xs[g * MP + m] = s * 4.76837158203125e-07f;  // 2^-21
}

cudaError_t launch_xprep(const void* x, int M, int64_t K, int MP, void* xh, float* xs, int* xe,
                         cudaStream_t stream) {
  const int64_t G = K / 128;
  const dim3 grid((unsigned)((G + kXpGroupsPerBlock - 1) / kXpGroupsPerBlock), (unsigned)MP);
  return launch_pdl(xprep_kernel, grid, dim3(kXpThreads), 0, stream, static_cast<const __nv_bfloat16*>(x), M, K, MP,
                    static_cast<__half*>(xh), xs, xe);
}

}  // namespace w4a16
