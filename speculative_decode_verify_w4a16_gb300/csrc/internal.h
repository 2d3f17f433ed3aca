// Internal host-side interface between the C-ABI layer and the kernel files.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "sched.cuh"

namespace w4a16 {

// Every workspace starts with this many bytes of zero-initialised counters
// (int32: from index 64 the linear's per (tile, warp) split-tile counters;
// the accept step's per-row counters), shared so that one
// workspace can serve any sequence of calls; each call leaves them zero.
constexpr size_t kCounterRegionBytes = 256 * 1024 + 256;
constexpr int64_t kMaxCounters = (int64_t)(kCounterRegionBytes / sizeof(int));

// Budget for the split-tile partial sums of one linear call.
constexpr size_t kDefaultPartialBytes = 128u << 20;

// Launch with programmatic stream serialisation (the kernel may begin while
// the previous kernel on the stream finishes; it waits on that grid with
// griddepcontrol.wait before touching shared global memory).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                       Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args&&>(args)...);
}

struct DeviceInfo {
  int device = -1;
  int num_sms = 0;
  unsigned* err = nullptr;  // device address of the error word
};

// Per-device state (error word address, SM count); initialised on first use
// with that device current.
cudaError_t device_info(DeviceInfo* out);

// ---- format
cudaError_t launch_quantize(const float* w, int64_t N, int64_t K, uint32_t* qweight, uint16_t* scales,
                            cudaStream_t stream);
cudaError_t launch_prepack(const uint32_t* qweight, const uint16_t* scales, int64_t N, int64_t K,
                           uint32_t* qw_packed, uint16_t* sc_packed, cudaStream_t stream);

// ---- linear (tensor-core fragments via mma.sync; M <= 8; items of contiguous units)
struct SkinnyPlan {
  int mt8 = 0;          // ceil(M / 8)
  int64_t units = 0;    // (N/128) * (K/128)
  int64_t ctas = 0;     // grid size
  ItemSched sched = {};
  size_t counter_bytes = 0;
  size_t partial_bytes = 0;
  size_t smem_bytes = 0;
};
cudaError_t skinny_plan(int M, int64_t N, int64_t K, const DeviceInfo& dev, size_t max_partial_bytes,
                        SkinnyPlan* plan);
size_t skinny_workspace_bytes(const SkinnyPlan& plan);
cudaError_t launch_skinny(const void* x, int M, int64_t K, const void* qw_packed, const void* sc_packed,
                          int64_t N, void* out, void* workspace, const SkinnyPlan& plan, const DeviceInfo& dev,
                          cudaStream_t stream);

// ---- linear on tcgen05 / TMEM (M >= kTcMinM)
constexpr int kTcMinM = 9;
constexpr int kTcMaxM = 80;  // largest token tile (ring depth 2 in tensor memory)
struct TcPlan {
  int nt = 0;           // MMA N: M rounded up to a multiple of 16
  int64_t units = 0;
  int64_t ctas = 0;
  ItemSched sched = {};
  size_t counter_bytes = 0;
  size_t partial_bytes = 0;
  size_t smem_bytes = 0;
};
cudaError_t tc_plan(int M, int64_t N, int64_t K, const DeviceInfo& dev, size_t max_partial_bytes, TcPlan* plan);
size_t tc_workspace_bytes(const TcPlan& plan);
cudaError_t launch_tc(const void* x, int M, int64_t K, const void* qw_packed, const void* sc_packed, int64_t N,
                      void* out, void* workspace, const TcPlan& plan, const DeviceInfo& dev, cudaStream_t stream);
// The fused-statistics variant (any M in 1..kTcMaxM): fp32 outputs [M][N] and
// (max, sum exp(l - max)) per (token, 32-row slice) [M][N/32].
cudaError_t tc_plan_fused(int M, int64_t N, int64_t K, const DeviceInfo& dev, TcPlan* plan);
cudaError_t launch_tc_fused(const void* x, int M, int64_t K, const void* qw_packed, const void* sc_packed, int64_t N,
                            float* logits, float2* stats, void* workspace, const TcPlan& plan, const DeviceInfo& dev,
                            cudaStream_t stream);

// ---- linear dispatch (by M)
struct LinearPlan {
  bool use_tc = false;
  SkinnyPlan sk;
  TcPlan tc;
  size_t workspace_bytes = 0;
};
cudaError_t linear_plan(int M, int64_t N, int64_t K, const DeviceInfo& dev, LinearPlan* plan,
                        size_t max_partial_bytes = kDefaultPartialBytes);
cudaError_t launch_linear(const void* x, int M, int64_t K, const void* qw_packed, const void* sc_packed, int64_t N,
                          void* out, void* workspace, const LinearPlan& plan, const DeviceInfo& dev,
                          cudaStream_t stream);

// The driver's cuTensorMapEncodeTiled (as void*; null if unavailable).
void* tensor_map_encode_fn();

// ---- tree-masked verify attention and KV compaction
struct AttnPlan {
  int rows = 0;        // query rows per KV head: n * (H / Hkv)
  int tiles = 0;       // 128-row tiles per CTA: 2 above 128 query rows per KV head, else 1
  int row_blocks = 0;  // row blocks (CTAs along the rows) per KV head
  int ctas = 0;        // CTAs of one wave: the pieces are cut for them
  int pieces_max = 0;  // grid: max(ctas, B * Hkv * row_blocks)
  int cut = 0;         // 1: sequences may be cut into pieces (up to 64 sequences, units < ctas)
  size_t ws_bytes = 0;  // cut: a partial slot per CTA + per sequence (first piece, pieces); else 0
};
AttnPlan attn_plan(int B, int n, int H, int Hkv, int max_len, int num_sms);
cudaError_t launch_tree_attention(const void* q, const void* k_cache, const void* v_cache, const int32_t* lens,
                                  const int32_t* parents, int B, int n, int H, int Hkv, int Lcap, int max_len,
                                  float scale, void* out, void* workspace, const AttnPlan& plan, unsigned* err,
                                  cudaStream_t stream);
cudaError_t launch_kv_compact(void* k_cache, void* v_cache, const int32_t* lens, const int32_t* parents,
                              const int32_t* node, int B, int n, int Hkv, int D, int Lcap, int layers,
                              int32_t* new_lens, unsigned* err, cudaStream_t stream);

// ---- accept
struct AcceptPlan {
  int rows = 0;       // logit rows read by the statistics pass (upper bound over modes)
  int rows_seq = 0;   // statistics rows in stochastic mode: B * (2n + 1)
  int ch = 0;         // chunks per row (statistics pass)
  int chunk = 0;      // elements per chunk (multiple of 4)
  int cha = 0;        // chunks per row (argmax pass)
  int chunka = 0;     // elements per chunk (multiple of 4)
  int ch2_lo = 0;     // fewest chunks per batch row in the residual pass
  int ch2 = 0;        // most chunks per batch row in the residual pass (workspace)
  int chunk2 = 0;     // elements per chunk at ch2
  size_t stats_off = 0, dec_off = 0, csum_off = 0, total = 0;  // counters at offset 0
};
AcceptPlan accept_plan(int B, int n, int V);
// p_stats: NULL, or the target rows' (max, sum exp(l - max)) per 32-logit
// slice [B * (n + 1)][V / 32] (the statistics pass then reads the draft rows only).
// node: NULL, or [B] for the accepted node (the deepest accepted tree node;
// accepted_len for a sequence draft)
cudaError_t launch_accept_seq(const float* p, const float* q, const int32_t* d, const float* u, int B, int n, int V,
                              int32_t* acc, int32_t* next, void* ws, const AcceptPlan& plan, int num_sms,
                              unsigned* err, cudaStream_t stream, const float2* p_stats = nullptr,
                              int32_t* node = nullptr);
// stochastic token tree (one 8-CTA cluster per batch row; V <= 131072)
constexpr int kAcceptTreeMaxV = 131072;
cudaError_t launch_accept_tree(const float* p, const float* q, const int32_t* d, const int32_t* parents,
                               const float* u, int B, int n, int V, int32_t* acc, int32_t* next, int32_t* node,
                               unsigned* err, cudaStream_t stream);
cudaError_t launch_accept_greedy(const float* p, const int32_t* d, const int32_t* parents, int B, int n, int V,
                                 int32_t* acc, int32_t* next, void* ws, const AcceptPlan& plan, unsigned* err,
                                 cudaStream_t stream, int32_t* node = nullptr);

}  // namespace w4a16
