// w4a16_linear_noalloc: the W4A16 verify linear for callers that cannot
// allocate device memory themselves (a plugin slot that hands over only its
// inputs and outputs, an embedding runtime that owns every allocation, code
// that must not call cudaMalloc on its hot path). Its scratch (the split-tile
// partial sums and completion counters of the stream-K linear) lives in one
// file-scope device array that every process loading this library holds for
// its lifetime on each GPU it uses.
#include <mutex>

#include "../../include/w4a16sv.h"
#include "common.cuh"
#include "format.cuh"
#include "internal.h"

namespace w4a16 {

constexpr size_t kNoAllocScratchBytes = 24u << 20;  // 24 MiB

// Shared by every call on a device; keeps the last call's contents.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

namespace {
std::mutex g_na_mu;
void* g_na_ptr[64];  // device address of g_noalloc_scratch, per device
}  // namespace

// Once per device, with that device current: look up the array's device
// address (host code must never use the symbol itself as a pointer).
static cudaError_t noalloc_scratch(int dev, void** out) {
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;  // g_na_ptr has one slot per device id < 64
  std::lock_guard<std::mutex> lk(g_na_mu);
  if (!g_na_ptr[dev]) {
    void* p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    g_na_ptr[dev] = p;
  }
  *out = g_na_ptr[dev];
  return cudaSuccess;
}

}  // namespace w4a16

using namespace w4a16;

extern "C" size_t w4a16_linear_noalloc_scratch_bytes(void) { return kNoAllocScratchBytes; }

extern "C" w4a16_status w4a16_linear_noalloc(const void* x, int M, int64_t K, const void* qweight_packed,
                                             const void* scales_packed, int64_t N, void* out, void* stream) {
  if (!x || !qweight_packed || !scales_packed || !out) return W4A16_ERR_INVALID_ARG;
  if (M < 1 || N <= 0 || K <= 0 || N % kUnitRows != 0 || K % kGroup != 0 || N > (int64_t(1) << 20) ||
      K > (int64_t(1) << 24))
    return W4A16_ERR_INVALID_ARG;
  if (M > kTcMaxM || K < 1024) return W4A16_ERR_UNSUPPORTED;
  if ((reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(qweight_packed) |
       reinterpret_cast<uintptr_t>(scales_packed)) % 16 != 0 ||
      reinterpret_cast<uintptr_t>(out) % 4 != 0)
    return W4A16_ERR_INVALID_ARG;
  DeviceInfo dev;
  if (device_info(&dev) != cudaSuccess) return W4A16_ERR_CUDA;
  LinearPlan plan;
  if (linear_plan(M, N, K, dev, &plan, kNoAllocScratchBytes - kCounterRegionBytes) != cudaSuccess)
    return W4A16_ERR_CUDA;
  if (plan.workspace_bytes > kNoAllocScratchBytes) return W4A16_ERR_WORKSPACE;
  void* scratch = nullptr;
  if (noalloc_scratch(dev.device, &scratch) != cudaSuccess) return W4A16_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // The kernels leave their completion counters at zero, but a call that
  // timed out may not have: clear the ones this call uses (one per (row tile,
  // epilogue warp) after the reserved ints).
  const size_t counter_bytes = (kTileCounterBase + (size_t)(N / kUnitRows) * 4) * sizeof(int);
  if (cudaMemsetAsync(scratch, 0, counter_bytes, s) != cudaSuccess) return W4A16_ERR_CUDA;
  return launch_linear(x, M, K, qweight_packed, scales_packed, N, out, scratch, plan, dev, s) == cudaSuccess
             ? W4A16_OK
             : W4A16_ERR_CUDA;
}
