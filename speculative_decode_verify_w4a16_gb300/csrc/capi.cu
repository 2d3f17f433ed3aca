// C-ABI layer of libw4a16sv: argument checks, dispatch, device state.
// Declarations and the contract of every entry point are in w4a16sv.h.
#include <math.h>

#include <mutex>

#include "../../include/w4a16sv.h"
#include "common.cuh"
#include "format.cuh"
#include <math.h>

#include "internal.h"

namespace w4a16 {

// Device error word (one per device that loads the library).
__device__ unsigned g_error_word;

namespace {
std::mutex g_mu;
DeviceInfo g_dev[64];
}  // namespace

cudaError_t device_info(DeviceInfo* out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_dev[dev].device != dev) {
    DeviceInfo d;
    d.device = dev;
    e = cudaDeviceGetAttribute(&d.num_sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_error_word);
    if (e != cudaSuccess) return e;
    d.err = static_cast<unsigned*>(p);
    g_dev[dev] = d;
  }
  *out = g_dev[dev];
  return cudaSuccess;
}

cudaError_t linear_plan(int M, int64_t N, int64_t K, const DeviceInfo& dev, LinearPlan* plan,
                        size_t max_partial_bytes) {
  plan->use_tc = M >= kTcMinM;
  cudaError_t e;
  if (plan->use_tc) {
    e = tc_plan(M, N, K, dev, max_partial_bytes, &plan->tc);
    plan->workspace_bytes = tc_workspace_bytes(plan->tc);
  } else {
    e = skinny_plan(M, N, K, dev, max_partial_bytes, &plan->sk);
    plan->workspace_bytes = skinny_workspace_bytes(plan->sk);
  }
  return e;
}

cudaError_t launch_linear(const void* x, int M, int64_t K, const void* qw_packed, const void* sc_packed, int64_t N,
                          void* out, void* workspace, const LinearPlan& plan, const DeviceInfo& dev,
                          cudaStream_t stream) {
  if (plan.use_tc) return launch_tc(x, M, K, qw_packed, sc_packed, N, out, workspace, plan.tc, dev, stream);
  return launch_skinny(x, M, K, qw_packed, sc_packed, N, out, workspace, plan.sk, dev, stream);
}

}  // namespace w4a16

using namespace w4a16;

static inline bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

static inline bool valid_nk(int64_t N, int64_t K) {
  return N > 0 && K > 0 && N % kUnitRows == 0 && K % kGroup == 0 && N <= (int64_t(1) << 20) &&
         K <= (int64_t(1) << 24);
}

extern "C" {

const char* w4a16_status_string(w4a16_status s) {
  switch (s) {
    case W4A16_OK: return "W4A16_OK";
    case W4A16_ERR_INVALID_ARG: return "W4A16_ERR_INVALID_ARG";
    case W4A16_ERR_UNSUPPORTED: return "W4A16_ERR_UNSUPPORTED";
    case W4A16_ERR_CUDA: return "W4A16_ERR_CUDA";
    case W4A16_ERR_DEVICE_TIMEOUT: return "W4A16_ERR_DEVICE_TIMEOUT";
    case W4A16_ERR_DEVICE_INPUT: return "W4A16_ERR_DEVICE_INPUT";
    case W4A16_ERR_WORKSPACE: return "W4A16_ERR_WORKSPACE";
    case W4A16_ERR_BOUNDS: return "W4A16_ERR_BOUNDS";
    default: return "W4A16_ERR_UNKNOWN";
  }
}

int w4a16_abi_version(void) { return 1; }

size_t w4a16_packed_weight_bytes(int64_t N, int64_t K) { return valid_nk(N, K) ? (size_t)(N * K / 2) : 0; }

size_t w4a16_packed_scale_bytes(int64_t N, int64_t K) { return valid_nk(N, K) ? (size_t)(N * K / 64) : 0; }

static bool item_args_ok(int64_t U, int C, int min_units) {
  return C >= 1 && U >= C && min_units >= 1 && U <= (int64_t(1) << 40);
}

int w4a16_item_rounds(int64_t U, int C, int min_units, int max_rounds, int64_t* rb) {
  if (!item_args_ok(U, C, min_units) || !rb) return 0;
  const ItemSched s = make_item_sched(U, C, min_units, max_rounds);
  for (int r = 0; r <= s.R; ++r) rb[r] = s.rb[r];
  return s.R;
}

int64_t w4a16_item_begin(int64_t U, int C, int min_units, int max_rounds, int i) {
  if (!item_args_ok(U, C, min_units)) return -1;
  const ItemSched s = make_item_sched(U, C, min_units, max_rounds);
  if (i < 0 || (int64_t)i > (int64_t)s.R * C) return -1;
  return item_begin(s, i);
}

int64_t w4a16_item_owner(int64_t U, int C, int min_units, int max_rounds, int64_t u) {
  if (!item_args_ok(U, C, min_units) || u < 0 || u >= U) return -1;
  return item_owner(make_item_sched(U, C, min_units, max_rounds), u);
}

w4a16_status w4a16_quantize(const float* w, int64_t N, int64_t K, uint32_t* qweight, uint16_t* scales,
                            void* stream) {
  if (!w || !qweight || !scales || !valid_nk(N, K)) return W4A16_ERR_INVALID_ARG;
  if (!aligned(w, 16) || !aligned(qweight, 4) || !aligned(scales, 2)) return W4A16_ERR_INVALID_ARG;
  return launch_quantize(w, N, K, qweight, scales, static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? W4A16_OK
             : W4A16_ERR_CUDA;
}

w4a16_status w4a16_prepack(const uint32_t* qweight, const uint16_t* scales, int64_t N, int64_t K,
                           void* qweight_packed, void* scales_packed, void* stream) {
  if (!qweight || !scales || !qweight_packed || !scales_packed || !valid_nk(N, K)) return W4A16_ERR_INVALID_ARG;
  if (!aligned(qweight_packed, 16) || !aligned(scales_packed, 16) || !aligned(qweight, 4) || !aligned(scales, 2))
    return W4A16_ERR_INVALID_ARG;
  return launch_prepack(qweight, scales, N, K, static_cast<uint32_t*>(qweight_packed),
                        static_cast<uint16_t*>(scales_packed), static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? W4A16_OK
             : W4A16_ERR_CUDA;
}

static bool linear_shape_ok(int M, int64_t N, int64_t K) {
  return M >= 1 && M <= kTcMaxM && valid_nk(N, K) && K >= 1024;
}

size_t w4a16_linear_workspace_bytes(int M, int64_t N, int64_t K) {
  if (!linear_shape_ok(M, N, K)) return 0;
  DeviceInfo dev;
  if (device_info(&dev) != cudaSuccess) return 0;
  LinearPlan plan;
  if (linear_plan(M, N, K, dev, &plan) != cudaSuccess) return 0;
  return plan.workspace_bytes;
}

w4a16_status w4a16_linear(const void* x, int M, int64_t K, const void* qweight_packed, const void* scales_packed,
                          int64_t N, void* out, void* workspace, size_t workspace_bytes, void* stream) {
  if (!x || !qweight_packed || !scales_packed || !out) return W4A16_ERR_INVALID_ARG;
  if (M < 1 || !valid_nk(N, K)) return W4A16_ERR_INVALID_ARG;
  if (M > kTcMaxM || K < 1024) return W4A16_ERR_UNSUPPORTED;
  if (!aligned(x, 16) || !aligned(qweight_packed, 16) || !aligned(scales_packed, 16) || !aligned(out, 4))
    return W4A16_ERR_INVALID_ARG;
  if (!workspace || !aligned(workspace, 256)) return W4A16_ERR_WORKSPACE;
  DeviceInfo dev;
  if (device_info(&dev) != cudaSuccess) return W4A16_ERR_CUDA;
  LinearPlan plan;
  if (linear_plan(M, N, K, dev, &plan) != cudaSuccess) return W4A16_ERR_CUDA;
  if (workspace_bytes < plan.workspace_bytes) return W4A16_ERR_WORKSPACE;
  return launch_linear(x, M, K, qweight_packed, scales_packed, N, out, workspace, plan, dev,
                       static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? W4A16_OK
             : W4A16_ERR_CUDA;
}

size_t w4a16_linear_logits_workspace_bytes(int M, int64_t N, int64_t K) {
  if (!linear_shape_ok(M, N, K)) return 0;
  DeviceInfo dev;
  if (device_info(&dev) != cudaSuccess) return 0;
  TcPlan plan;
  if (tc_plan_fused(M, N, K, dev, &plan) != cudaSuccess) return 0;
  return tc_workspace_bytes(plan);
}

w4a16_status w4a16_linear_logits(const void* x, int M, int64_t K, const void* qweight_packed,
                                 const void* scales_packed, int64_t N, float* logits, float* row_stats,
                                 void* workspace, size_t workspace_bytes, void* stream) {
  if (!x || !qweight_packed || !scales_packed || !logits || !row_stats) return W4A16_ERR_INVALID_ARG;
  if (M < 1 || !valid_nk(N, K)) return W4A16_ERR_INVALID_ARG;
  if (M > kTcMaxM || K < 1024) return W4A16_ERR_UNSUPPORTED;
  if (!aligned(x, 16) || !aligned(qweight_packed, 16) || !aligned(scales_packed, 16) || !aligned(logits, 4) ||
      !aligned(row_stats, 8))
    return W4A16_ERR_INVALID_ARG;
  if (!workspace || !aligned(workspace, 256)) return W4A16_ERR_WORKSPACE;
  DeviceInfo dev;
  if (device_info(&dev) != cudaSuccess) return W4A16_ERR_CUDA;
  TcPlan plan;
  if (tc_plan_fused(M, N, K, dev, &plan) != cudaSuccess) return W4A16_ERR_CUDA;
  if (workspace_bytes < tc_workspace_bytes(plan)) return W4A16_ERR_WORKSPACE;
  return launch_tc_fused(x, M, K, qweight_packed, scales_packed, N, logits, reinterpret_cast<float2*>(row_stats),
                         workspace, plan, dev, static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? W4A16_OK
             : W4A16_ERR_CUDA;
}

static bool accept_shape_ok(int B, int n, int V) {
  // grid rows: B * (2n + 1) statistics rows must fit one grid dimension
  return B >= 1 && B <= 32768 && n >= 1 && n <= 1024 && V >= 2 && V <= (1 << 20) &&
         (int64_t)B * (2 * n + 1) <= 65535;
}

size_t spec_accept_workspace_bytes(int B, int n, int V) {
  if (!accept_shape_ok(B, n, V)) return 0;
  return accept_plan(B, n, V).total;
}

static w4a16_status accept_impl(const float* p_logits, const float* q_logits, const int32_t* draft_ids,
                                const int32_t* tree_parents, const float* uniforms, int B, int n, int V,
                                int32_t* accepted_len, int32_t* next_token, int32_t* accepted_node, void* workspace,
                                size_t workspace_bytes, void* stream) {
  if (!p_logits || !draft_ids || !accepted_len || !next_token) return W4A16_ERR_INVALID_ARG;
  if (accepted_node && !aligned(accepted_node, 4)) return W4A16_ERR_INVALID_ARG;
  if (!accept_shape_ok(B, n, V)) return W4A16_ERR_INVALID_ARG;
  if (q_logits && !uniforms) return W4A16_ERR_INVALID_ARG;
  if (q_logits && tree_parents && V > kAcceptTreeMaxV) return W4A16_ERR_UNSUPPORTED;
  if (V % 4 == 0 && (!aligned(p_logits, 16) || (q_logits && !aligned(q_logits, 16)))) return W4A16_ERR_INVALID_ARG;
  if (!aligned(p_logits, 4) || !aligned(draft_ids, 4) || !aligned(accepted_len, 4) || !aligned(next_token, 4))
    return W4A16_ERR_INVALID_ARG;
  const AcceptPlan plan = accept_plan(B, n, V);
  if (!workspace || !aligned(workspace, 256) || workspace_bytes < plan.total) return W4A16_ERR_WORKSPACE;
  DeviceInfo dev;
  if (device_info(&dev) != cudaSuccess) return W4A16_ERR_CUDA;
  cudaError_t e;
  if (q_logits && tree_parents)
    e = launch_accept_tree(p_logits, q_logits, draft_ids, tree_parents, uniforms, B, n, V, accepted_len, next_token,
                           accepted_node, dev.err, static_cast<cudaStream_t>(stream));
  else if (q_logits)
    e = launch_accept_seq(p_logits, q_logits, draft_ids, uniforms, B, n, V, accepted_len, next_token, workspace, plan,
                          dev.num_sms, dev.err, static_cast<cudaStream_t>(stream), nullptr, accepted_node);
  else
    e = launch_accept_greedy(p_logits, draft_ids, tree_parents, B, n, V, accepted_len, next_token, workspace, plan,
                             dev.err, static_cast<cudaStream_t>(stream), accepted_node);
  return e == cudaSuccess ? W4A16_OK : W4A16_ERR_CUDA;
}

w4a16_status spec_accept(const float* p_logits, const float* q_logits, const int32_t* draft_ids,
                         const int32_t* tree_parents, const float* uniforms, int B, int n, int V,
                         int32_t* accepted_len, int32_t* next_token, void* workspace, size_t workspace_bytes,
                         void* stream) {
  return accept_impl(p_logits, q_logits, draft_ids, tree_parents, uniforms, B, n, V, accepted_len, next_token,
                     nullptr, workspace, workspace_bytes, stream);
}

w4a16_status spec_accept_node(const float* p_logits, const float* q_logits, const int32_t* draft_ids,
                              const int32_t* tree_parents, const float* uniforms, int B, int n, int V,
                              int32_t* accepted_len, int32_t* next_token, int32_t* accepted_node, void* workspace,
                              size_t workspace_bytes, void* stream) {
  if (!accepted_node) return W4A16_ERR_INVALID_ARG;
  return accept_impl(p_logits, q_logits, draft_ids, tree_parents, uniforms, B, n, V, accepted_len, next_token,
                     accepted_node, workspace, workspace_bytes, stream);
}

// ---------------------------------------------------- verify attention
static bool attn_shape_ok(int B, int n, int H, int Hkv, int Lcap, int max_len) {
  return B >= 1 && B <= 65535 && n >= 1 && H >= 1 && Hkv >= 1 && Hkv <= 65535 && H % Hkv == 0 && max_len >= 0 &&
         (int64_t)max_len + n <= Lcap && (int64_t)B * Hkv * Lcap <= INT32_MAX && (int64_t)n * H <= INT32_MAX;
}

size_t tree_attention_workspace_bytes(int B, int n, int H, int Hkv, int D, int Lcap, int max_len) {
  if (!attn_shape_ok(B, n, H, Hkv, Lcap, max_len) || D != 128 || n > 64) return 0;
  DeviceInfo dev;
  if (device_info(&dev) != cudaSuccess) return 0;
  return attn_plan(B, n, H, Hkv, max_len, dev.num_sms).ws_bytes;
}

w4a16_status tree_attention(const void* q, const void* k_cache, const void* v_cache, const int32_t* lens,
                            const int32_t* tree_parents, int B, int n, int H, int Hkv, int D, int Lcap, int max_len,
                            float scale, void* out, void* workspace, size_t workspace_bytes, void* stream) {
  if (!q || !k_cache || !v_cache || !lens || !out) return W4A16_ERR_INVALID_ARG;
  if (!attn_shape_ok(B, n, H, Hkv, Lcap, max_len) || !(scale > 0.0f) || !(scale < INFINITY))
    return W4A16_ERR_INVALID_ARG;
  if (D != 128 || n > 64) return W4A16_ERR_UNSUPPORTED;
  if (!aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(out, 16) || !aligned(lens, 4) ||
      (tree_parents && !aligned(tree_parents, 4)))
    return W4A16_ERR_INVALID_ARG;
  DeviceInfo dev;
  if (device_info(&dev) != cudaSuccess) return W4A16_ERR_CUDA;
  const AttnPlan plan = attn_plan(B, n, H, Hkv, max_len, dev.num_sms);
  if (plan.ws_bytes > 0 && (!workspace || !aligned(workspace, 256) || workspace_bytes < plan.ws_bytes))
    return W4A16_ERR_WORKSPACE;
  return launch_tree_attention(q, k_cache, v_cache, lens, tree_parents, B, n, H, Hkv, Lcap, max_len, scale, out,
                               workspace, plan, dev.err, static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? W4A16_OK
             : W4A16_ERR_CUDA;
}

w4a16_status kv_compact(void* k_cache, void* v_cache, const int32_t* lens, const int32_t* tree_parents,
                        const int32_t* accepted_node, int B, int n, int Hkv, int D, int Lcap, int n_layers,
                        int32_t* new_lens, void* stream) {
  if (!k_cache || !v_cache || !lens || !accepted_node || !new_lens) return W4A16_ERR_INVALID_ARG;
  if (B < 1 || n < 1 || Hkv < 1 || D < 8 || D % 8 != 0 || Lcap < n || n_layers < 1 || n_layers > 65535)
    return W4A16_ERR_INVALID_ARG;
  // one tree node's keys and values of every head: at most 4096 16-byte words
  if (n > 64 || (int64_t)2 * Hkv * (D / 8) > 4096) return W4A16_ERR_UNSUPPORTED;
  if (!aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(lens, 4) || !aligned(accepted_node, 4) ||
      !aligned(new_lens, 4) || (tree_parents && !aligned(tree_parents, 4)))
    return W4A16_ERR_INVALID_ARG;
  DeviceInfo dev;
  if (device_info(&dev) != cudaSuccess) return W4A16_ERR_CUDA;
  return launch_kv_compact(k_cache, v_cache, lens, tree_parents, accepted_node, B, n, Hkv, D, Lcap, n_layers,
                           new_lens, dev.err, static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? W4A16_OK
             : W4A16_ERR_CUDA;
}

w4a16_status spec_accept_prestat(const float* p_logits, const float* p_stats, const float* q_logits,
                                 const int32_t* draft_ids, const float* uniforms, int B, int n, int V,
                                 int32_t* accepted_len, int32_t* next_token, void* workspace,
                                 size_t workspace_bytes, void* stream) {
  if (!p_logits || !p_stats || !q_logits || !draft_ids || !uniforms || !accepted_len || !next_token)
    return W4A16_ERR_INVALID_ARG;
  if (!accept_shape_ok(B, n, V) || V % 32 != 0) return W4A16_ERR_INVALID_ARG;
  if (!aligned(p_logits, 16) || !aligned(q_logits, 16) || !aligned(p_stats, 8) || !aligned(draft_ids, 4) ||
      !aligned(uniforms, 4) || !aligned(accepted_len, 4) || !aligned(next_token, 4))
    return W4A16_ERR_INVALID_ARG;
  const AcceptPlan plan = accept_plan(B, n, V);
  if (!workspace || !aligned(workspace, 256) || workspace_bytes < plan.total) return W4A16_ERR_WORKSPACE;
  DeviceInfo dev;
  if (device_info(&dev) != cudaSuccess) return W4A16_ERR_CUDA;
  return launch_accept_seq(p_logits, q_logits, draft_ids, uniforms, B, n, V, accepted_len, next_token, workspace,
                           plan, dev.num_sms, dev.err, static_cast<cudaStream_t>(stream),
                           reinterpret_cast<const float2*>(p_stats)) == cudaSuccess
             ? W4A16_OK
             : W4A16_ERR_CUDA;
}

w4a16_status w4a16_check_device_status(void* stream) {
  DeviceInfo dev;
  if (device_info(&dev) != cudaSuccess) return W4A16_ERR_CUDA;
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return W4A16_ERR_CUDA;
  unsigned word = 0;
  if (cudaMemcpy(&word, dev.err, sizeof(word), cudaMemcpyDeviceToHost) != cudaSuccess) return W4A16_ERR_CUDA;
  if (word) {
    const unsigned zero = 0;
    if (cudaMemcpy(dev.err, &zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess) return W4A16_ERR_CUDA;
  }
  if (word & kErrTimeout) return W4A16_ERR_DEVICE_TIMEOUT;
  if (word & kErrBounds) return W4A16_ERR_BOUNDS;
  if (word & kErrInput) return W4A16_ERR_DEVICE_INPUT;
  return W4A16_OK;
}

}  // extern "C"
