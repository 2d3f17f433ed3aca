// int4 g128 format kernels: group quantiser (canonical layout) and the
// one-time prepack into the streaming layout described in format.cuh.
#include "common.cuh"
#include "format.cuh"
#include "internal.h"

namespace w4a16 {

// One warp per (row, group): s = fp16(max|w| / 7), code = clamp(rne(w / s), -8, 7).
// Lane l holds k = 4l .. 4l+3 of the group; lanes 2i and 2i+1 share one
// canonical word (8 codes), written by the even lane.
__global__ void quantize_kernel(const float* __restrict__ w, int64_t N, int64_t K, uint32_t* __restrict__ qweight,
                                __half* __restrict__ scales) {
  const int lane = threadIdx.x & 31;
  const int64_t G = K / kGroup;
  const int64_t item = (int64_t)blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5);
  if (item >= N * G) return;
  const int64_t n = item / G, g = item % G;
  const float4 v = *reinterpret_cast<const float4*>(w + n * K + g * kGroup + lane * 4);
  float a = fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w)));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
  const __half s16 = __float2half_rn(a / 7.0f);
  const float s = __half2float(s16);
  const float vals[4] = {v.x, v.y, v.z, v.w};
  uint32_t nib = 0;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    int q = 0;
    if (s != 0.0f) {
      const float r = rintf(vals[j] / s);
      q = r > 7.0f ? 7 : (r < -8.0f ? -8 : (int)r);
    }
    nib |= ((uint32_t)q & 0xFu) << (4 * j);
  }
  const uint32_t other = __shfl_xor_sync(0xffffffffu, nib, 1);
  if ((lane & 1) == 0) qweight[n * (K / 8) + g * 16 + lane / 2] = nib | (other << 16);
  if (lane == 0) scales[n * G + g] = s16;
}

// One thread per packed word.
__global__ void prepack_weights_kernel(const uint32_t* __restrict__ qw, int64_t N, int64_t K,
                                       uint32_t* __restrict__ out) {
  const int64_t total = N * K / 8;
  const int64_t G = K / kGroup;
  for (int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; idx < total;
       idx += (int64_t)gridDim.x * blockDim.x) {
    const int64_t u = idx / kUnitWords;
    const int o = (int)(idx % kUnitWords);
    const int j = o & 3, lane = (o >> 2) & 31, h = (o >> 7) & 1, rt = (o >> 8) & 1, w4 = (o >> 9) & 3;
    const int64_t t = u / G, g = u % G;
    const int gid = lane >> 2, c = lane & 3;
    const int64_t r_lo = t * kUnitRows + 32 * w4 + 16 * rt + gid;
    const int64_t r_hi = r_lo + 8;
    const int64_t kb = g * kGroup + 16 * (4 * h + j) + 4 * c;  // 4 consecutive k in one canonical word
    const int sh = 4 * (int)(kb % 8);
    const uint32_t wl = qw[r_lo * (K / 8) + kb / 8] >> sh;  // nibbles of k = kb..kb+3, row r_lo
    const uint32_t wh = qw[r_hi * (K / 8) + kb / 8] >> sh;
    auto nib = [](uint32_t wv, int i) { return ((wv >> (4 * i)) & 0xFu) ^ 0x8u; };  // offset-binary
    uint32_t r = 0;
    r |= nib(wl, 0) << 0;
    r |= nib(wl, 1) << 16;
    r |= nib(wh, 0) << 4;
    r |= nib(wh, 1) << 20;
    r |= nib(wl, 2) << 8;
    r |= nib(wl, 3) << 24;
    r |= nib(wh, 2) << 12;
    r |= nib(wh, 3) << 28;
    out[idx] = r;
  }
}

__global__ void prepack_scales_kernel(const uint16_t* __restrict__ sc, int64_t N, int64_t K,
                                      uint16_t* __restrict__ out) {
  const int64_t G = K / kGroup;
  const int64_t total = N * G;
  for (int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; idx < total;
       idx += (int64_t)gridDim.x * blockDim.x) {
    const int64_t u = idx / 128;
    const int o = (int)(idx % 128);
    const int hi = o & 1, rt = (o >> 1) & 1, gid = (o >> 2) & 7, w4 = (o >> 5) & 3;
    const int64_t t = u / G, g = u % G;
    const int64_t row = t * kUnitRows + 32 * w4 + 16 * rt + gid + 8 * hi;
    out[idx] = sc[row * G + g];
  }
}

cudaError_t launch_quantize(const float* w, int64_t N, int64_t K, uint32_t* qweight, uint16_t* scales,
                            cudaStream_t stream) {
  const int64_t items = N * (K / kGroup);
  const int warps_per_block = 8;
  const int64_t blocks = (items + warps_per_block - 1) / warps_per_block;
  if (blocks > 0x7fffffffLL) return cudaErrorInvalidValue;
  quantize_kernel<<<(unsigned)blocks, 32 * warps_per_block, 0, stream>>>(w, N, K, qweight,
                                                                         reinterpret_cast<__half*>(scales));
  return cudaGetLastError();
}

cudaError_t launch_prepack(const uint32_t* qweight, const uint16_t* scales, int64_t N, int64_t K,
                           uint32_t* qw_packed, uint16_t* sc_packed, cudaStream_t stream) {
  const int64_t words = N * K / 8;
  int64_t blocks = (words + 255) / 256;
  if (blocks > 65536) blocks = 65536;
  prepack_weights_kernel<<<(unsigned)blocks, 256, 0, stream>>>(qweight, N, K, qw_packed);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const int64_t halves = N * (K / kGroup);
  int64_t b2 = (halves + 255) / 256;
  if (b2 > 65536) b2 = 65536;
  prepack_scales_kernel<<<(unsigned)b2, 256, 0, stream>>>(scales, N, K, sc_packed);
  return cudaGetLastError();
}

}  // namespace w4a16
