/*
 * w4a16sv — W4A16 speculative-verify library for NVIDIA GB300 (sm_103a).
 *
 * C ABI: plain pointers and sizes. Every `void* stream` is a cudaStream_t
 * (NULL = the legacy default stream). Every buffer is caller-allocated; the
 * library never allocates or frees device memory. Every call that takes a
 * stream only enqueues work and returns after host-side argument checks; a
 * failure inside a kernel (a wait that ran out, an out-of-range id found on
 * the device) is recorded in a device error word and reported by
 * w4a16_check_device_status(). Errors are return codes: nothing here traps,
 * asserts or throws.
 *
 * What it computes follows the pages of "Speculative Decoding Meets
 * Quantization" (Zhang et al. 2025: verifying drafts on a 4-bit weight-only
 * quantised target, whose forward is bound by weight memory traffic) and the
 * tutorial "Speculative Decoding이란?" (section 3, Steps 2-4; sections 5-6:
 * the acceptance test, sequential acceptance, corrected distribution,
 * greedy equivalence). The 4-bit format is int4 symmetric, group size 128
 * along K, fp16 scales, 8 nibbles per uint32.
 */
#ifndef W4A16SV_H_
#define W4A16SV_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef int w4a16_status;
#define W4A16_OK 0
#define W4A16_ERR_INVALID_ARG 1     /* null pointer, bad size, misaligned buffer */
#define W4A16_ERR_UNSUPPORTED 2     /* valid request this build does not handle */
#define W4A16_ERR_CUDA 3            /* a CUDA runtime call failed */
#define W4A16_ERR_DEVICE_TIMEOUT 4  /* a kernel's bounded wait ran out (device error word) */
#define W4A16_ERR_DEVICE_INPUT 5    /* a kernel found an out-of-range id or a bad parent (device error word) */
#define W4A16_ERR_WORKSPACE 6       /* workspace pointer missing or smaller than required */
#define W4A16_ERR_BOUNDS 7          /* bounds-checked debug build only: a kernel's computed index left its
                                       buffer (recorded in the device error word, the access skipped) */

/* Human-readable name of a status code (static string, never NULL). */
const char* w4a16_status_string(w4a16_status status);

/* ABI version of this header (incremented on any signature change). */
int w4a16_abi_version(void);

/* ------------------------------------------------------------------------
 * 4-bit weight format
 *
 * Canonical layout (task specification; the pages fix no format):
 *   qweight[N][K/8] uint32: code of W[n][k] in bits 4*(k%8) .. 4*(k%8)+3 of
 *   qweight[n][k/8], two's complement in [-8, 7];
 *   scales[N][K/128] fp16 (IEEE half bits): W[n][k] = code * scales[n][k/128].
 * N and K must be multiples of 128.
 * ---------------------------------------------------------------------- */

/* Bytes of the prepacked weight / scale buffers for an N x K matrix
 * (equal to the canonical sizes: N*K/2 and N*K/64). 0 if N or K is invalid. */
size_t w4a16_packed_weight_bytes(int64_t N, int64_t K);
size_t w4a16_packed_scale_bytes(int64_t N, int64_t K);

/*
 * Group quantiser (device). w[N][K] fp32 (device) -> canonical qweight and
 * scales (device, caller-allocated). Per row n and group g:
 *   s = fp16_rne(max_j |w| / 7)  (fp32 quotient, then round to half),
 *   code = clamp(rne(w / s), -8, 7), or 0 when s == 0.
 * This is the spec's "scale = max|w|/7" symmetric int4 format; the rounding
 * rules are this library's reading. Bit-exact with the CPU oracle.
 */
w4a16_status w4a16_quantize(const float* w, int64_t N, int64_t K, uint32_t* qweight, uint16_t* scales,
                            void* stream);

/*
 * Prepack (device, one time per weight): canonical (qweight, scales) ->
 * the GPU streaming layout consumed by w4a16_linear. Both outputs are
 * caller-allocated device buffers of w4a16_packed_weight_bytes /
 * w4a16_packed_scale_bytes bytes, 16-byte aligned. The packed layout is
 * opaque: 128 x 128 tiles in (row-tile, group) order with the nibbles placed
 * where the tensor-core fragments want them, codes stored offset by +8.
 */
w4a16_status w4a16_prepack(const uint32_t* qweight, const uint16_t* scales, int64_t N, int64_t K,
                           void* qweight_packed, void* scales_packed, void* stream);

/* ------------------------------------------------------------------------
 * W4A16 verify linear: out[M][N] = bf16( x[M][K] . W^T ), W = code * scale.
 *
 * The verify forward of a speculative step runs every target linear at the
 * number of draft tokens being checked (the tutorial's section 3 Step 2: all
 * K positions in one forward; "Speculative Decoding Meets Quantization":
 * M = 1 decode, small M for a sequence draft, M up to 64 for a tree draft).
 * The dequantisation is fused into the contraction: codes are exact in bf16,
 * each 128-wide group is accumulated in fp32 and scaled once in fp32.
 *
 *   x            device, bf16 [M][K] row-major, 16-byte aligned
 *   M            1 .. 80
 *   K, N         multiples of 128, K >= 1024, N <= 2^20
 *   qweight_packed, scales_packed   from w4a16_prepack (device)
 *   out          device, bf16 [M][N] row-major
 *   workspace    device scratch of at least w4a16_linear_workspace_bytes(M,N,K)
 *                bytes, 256-byte aligned. Its first 262,400 bytes (256 KiB +
 *                256) hold counters (split-tile completions, accept steps):
 *                ZERO-FILL the workspace before its first use; every call
 *                leaves the counters zero again, so one workspace serves any
 *                later linear or accept call. After W4A16_ERR_DEVICE_TIMEOUT,
 *                zero it again before reuse. Calls that share a workspace must
 *                not overlap in time (calls on one stream never do).
 * Kernels are launched with programmatic dependent launch: one may start
 * while the previous kernel on the stream finishes (only a kernel that
 * signals programmatic completion early lets it, as this library's own
 * kernels do). It streams qweight_packed and scales_packed at once, but reads
 * x and the workspace and writes out only after that kernel has completed;
 * so a kernel that writes the packed weights must not signal early (the
 * library's quantize and prepack kernels do not).
 * Returns W4A16_ERR_INVALID_ARG / _WORKSPACE / _UNSUPPORTED before launching.
 */
size_t w4a16_linear_workspace_bytes(int M, int64_t N, int64_t K);
w4a16_status w4a16_linear(const void* x, int M, int64_t K, const void* qweight_packed,
                          const void* scales_packed, int64_t N, void* out, void* workspace,
                          size_t workspace_bytes, void* stream);

/* ------------------------------------------------------------------------
 * The target's lm_head for the verify pass with its softmax statistics
 * fused into the epilogue ("Speculative Decoding Meets Quantization": the
 * verify forward of the 4-bit target ends in the lm_head over every draft
 * position; the tutorial page, section 3 Step 3: the acceptance test needs
 * p = softmax of those logits). The accept step needs, per target row, the
 * maximum and sum of exp(l - max) over the vocabulary and the logits at the
 * drafted and drawn tokens. The epilogue produces the statistics of each
 * 32-logit slice while the logits are still in registers, so
 * spec_accept_prestat does not read the target rows to normalise them.
 *
 *   x, M, K, qweight_packed, scales_packed, N   as for w4a16_linear, with
 *                M in 1 .. 80 (this call always runs on the tcgen05 kernel)
 *   logits       device, fp32 [M][N] (4-byte aligned; 16-byte aligned lets
 *                the kernel write whole tiles with TMA stores): x . W^T, the
 *                fp32 sum unrounded
 *   row_stats    device, fp32 pairs [M][N / 32] (8-byte aligned): for row m
 *                and slice s, (max_j l, sum_j exp(l - max)) over the logits
 *                l = logits[m][32 s + j], j = 0..31; the exponential within a
 *                few ulp, the sum in fp32 (four partial sums over j mod 4,
 *                added pairwise)
 *   workspace    as for w4a16_linear, of w4a16_linear_logits_workspace_bytes
 * Same launch and error rules as w4a16_linear.
 */
size_t w4a16_linear_logits_workspace_bytes(int M, int64_t N, int64_t K);
w4a16_status w4a16_linear_logits(const void* x, int M, int64_t K, const void* qweight_packed,
                                 const void* scales_packed, int64_t N, float* logits, float* row_stats,
                                 void* workspace, size_t workspace_bytes, void* stream);

/* ------------------------------------------------------------------------
 * Speculative accept step (the tutorial page, section 3 Steps 3-4 and
 * section 6; greedy mode: section 5, "greedy decoding result identical").
 *
 * Modes (chosen by which pointers are NULL):
 *   stochastic sequence  q_logits != NULL, tree_parents == NULL
 *       p_logits [B][n+1][V] fp32: row i = target logits for draft position
 *                i+1 (row n: the extra position after all drafts)
 *       q_logits [B][n][V] fp32: draft logits for draft position i+1
 *       draft_ids [B][n] int32, uniforms [B][n+1] fp32 in [0, 1)
 *       For i = 1..n: alpha_i = min(1, P_i(d_i) / Q_i(d_i)) (P, Q = softmax
 *       at temperature 1; Q(d) == 0 gives alpha = 1); d_i is accepted iff
 *       u_i < alpha_i; stop at the first rejection r. next_token is drawn
 *       with u_{n+1} from normalize(max(0, P_r - Q_r)) (P_r itself if that
 *       sums to 0), or from P_{n+1} when all n are accepted. A draw is the
 *       smallest x whose ascending running sum exceeds u * total.
 *       accepted_len in [0, n].
 *   greedy sequence      q_logits == NULL, tree_parents == NULL
 *       p_logits [B][n+1][V], draft_ids [B][n]; uniforms may be NULL.
 *       accepted while d_i == argmax(p row i-1); next = argmax of the row
 *       after the last accepted token. argmax ties go to the smallest id.
 *   greedy tree          q_logits == NULL, tree_parents != NULL
 *       p_logits [B][n][V] (row j: after the path root..j), draft_ids [B][n]
 *       (slot 0 = root, ignored), tree_parents [B][n] int32 with
 *       parent[0] = -1 and 0 <= parent[j] < j. Node j is accepted iff its
 *       parent is and draft[j] == argmax(parent's row); accepted_len is the
 *       depth of the deepest accepted node (smallest index on ties) and
 *       next_token the argmax of its row.
 *   stochastic tree      q_logits != NULL, tree_parents != NULL
 *       p_logits, q_logits [B][n][V] (row j: target / draft distribution
 *       after the path root..j; node j's children were drawn from q row j),
 *       draft_ids [B][n] (slot 0 = root), tree_parents as above, uniforms
 *       [B][n] (u_j tests node j, u_0 draws the next token); V <= 131072
 *       (else W4A16_ERR_UNSUPPORTED). The pages give no rule for a tree:
 *       multi-step speculative sampling as SpecInfer defines it for children
 *       drawn independently from the draft: at node u (from the root, with
 *       R = P_u) the children are tried in ascending index, child s with
 *       token x is accepted iff u_s < min(1, R(x) / Q_u(x)) (then u = s,
 *       R = P_s), a rejection replaces R by normalize(max(0, R - Q_u)) (kept
 *       when that sums to 0); with no child left next_token is drawn from R
 *       with u_0. accepted_len = the final node's depth.
 * Logits must be finite. Outputs accepted_len[B], next_token[B] int32
 * (device). An id outside [0, V) or a bad parent sets W4A16_ERR_DEVICE_INPUT
 * in the device error word (the row then reports accepted_len = 0).
 * All pointers are device pointers; p/q rows must be 16-byte aligned when
 * V % 4 == 0. workspace: device scratch of spec_accept_workspace_bytes(B,n,V)
 * bytes, 256-byte aligned, with the same zeroed counter region (256 KiB + 256
 * bytes) at its start as the linear's workspace (either can serve both).
 * Limits: 1 <= B <= 32768, 1 <= n <= 1024, B * (2n + 1) <= 65535, 2 <= V <= 2^20.
 * ---------------------------------------------------------------------- */
size_t spec_accept_workspace_bytes(int B, int n, int V);
w4a16_status spec_accept(const float* p_logits, const float* q_logits, const int32_t* draft_ids,
                         const int32_t* tree_parents, const float* uniforms, int B, int n, int V,
                         int32_t* accepted_len, int32_t* next_token, void* workspace,
                         size_t workspace_bytes, void* stream);

/* ------------------------------------------------------------------------
 * spec_accept that also reports the accepted node: accepted_node[B] int32
 * (device, required) = the final node of the accepted root path in the tree
 * modes (the deepest accepted node in greedy mode), accepted_len in the
 * sequence modes (a chain's node index is its depth).
 * kv_compact takes it. Everything else as spec_accept.
 */
w4a16_status spec_accept_node(const float* p_logits, const float* q_logits, const int32_t* draft_ids,
                              const int32_t* tree_parents, const float* uniforms, int B, int n, int V,
                              int32_t* accepted_len, int32_t* next_token, int32_t* accepted_node, void* workspace,
                              size_t workspace_bytes, void* stream);

/* ------------------------------------------------------------------------
 * Tree-masked attention of the verify pass (the tutorial page, section
 * 10.1: Medusa's tree-based attention verifies every candidate continuation
 * of a token tree in one target pass; section 10.4: ReDrafter's dynamic tree
 * attention; a sequence draft is the chain parent[j] = j - 1).
 *
 * Every tree node j is a query position. It attends to the whole committed
 * prefix of its batch row (cache positions 0 .. lens[b] - 1) and to the tree
 * nodes on its own root path, itself included, whose keys and values the
 * verify forward has written at cache positions lens[b] + node index.
 * out = softmax(scale * q . k over the allowed keys) . v, per query head;
 * query head h reads key/value head h / (H / Hkv).
 *
 *   q             device bf16 [B][n][H][D] (16-byte aligned)
 *   k_cache, v_cache  device bf16 [B][Hkv][Lcap][D] (16-byte aligned)
 *   lens          device int32 [B]: committed lengths, 0 <= lens[b] <= max_len
 *   tree_parents  device int32 [B][n] (parent[0] = -1, 0 <= parent[j] < j),
 *                 or NULL for a sequence draft (the chain)
 *   n             tree nodes, 1 .. 64; D = 128 (else W4A16_ERR_UNSUPPORTED)
 *   max_len       an upper bound of lens[] known to the caller (a larger
 *                 lens[b] is reported and clamped); max_len + n <= Lcap
 *   scale         softmax scale (1 / sqrt(D) for the model), finite, > 0
 *   out           device bf16 [B][n][H][D] (16-byte aligned)
 *   workspace     device scratch of tree_attention_workspace_bytes() bytes
 *                 (256-byte aligned; may be NULL when that is 0: nonzero only
 *                 for up to 64 sequences whose units leave at least half the
 *                 SMs free, which the kernel may cut into pieces); needs no
 *                 initialisation
 * Arithmetic: bf16 inputs, fp32 scores and sums; the softmax weights are
 * rounded to bf16 for the weighted sum of the values and normalised by the
 * sum of the fp32 weights; out rounded to bf16.
 * A lens[b] outside [0, max_len] or a bad parent sets W4A16_ERR_DEVICE_INPUT
 * in the device error word (the length is clamped, the node then attends to
 * itself and the prefix only). Launch rules as for w4a16_linear.
 */
size_t tree_attention_workspace_bytes(int B, int n, int H, int Hkv, int D, int Lcap, int max_len);
w4a16_status tree_attention(const void* q, const void* k_cache, const void* v_cache, const int32_t* lens,
                            const int32_t* tree_parents, int B, int n, int H, int Hkv, int D, int Lcap, int max_len,
                            float scale, void* out, void* workspace, size_t workspace_bytes, void* stream);

/* ------------------------------------------------------------------------
 * KV compaction after verification (the tutorial page, section 8.7: the
 * cache must not keep rejected tokens; section 10.4). The keys and values of
 * the nodes on the root path of accepted_node[b] (root first) move to cache
 * positions lens[b] + 0, 1, ..., depth, in every layer and head, and
 * new_lens[b] = lens[b] + depth + 1 (the root, node 0, is always kept).
 * Positions from new_lens[b] on keep stale values.
 *
 *   k_cache, v_cache  device bf16 [n_layers][B][Hkv][Lcap][D], updated in
 *                 place (16-byte aligned; D a multiple of 8,
 *                 2 * Hkv * D <= 32768)
 *   lens          device int32 [B], 0 <= lens[b] <= Lcap - n
 *   tree_parents  as for tree_attention (NULL: chain)
 *   accepted_node device int32 [B] in [0, n) (spec_accept_node)
 *   new_lens      device int32 [B] (may not alias lens)
 *   n             1 .. 64
 * Bad input sets W4A16_ERR_DEVICE_INPUT in the device error word (the row
 * then keeps the root only).
 */
w4a16_status kv_compact(void* k_cache, void* v_cache, const int32_t* lens, const int32_t* tree_parents,
                        const int32_t* accepted_node, int B, int n, int Hkv, int D, int Lcap, int n_layers,
                        int32_t* new_lens, void* stream);

/* ------------------------------------------------------------------------
 * Stochastic sequence accept with the target rows' statistics supplied
 * (from w4a16_linear_logits over the B * (n + 1) verify positions): the same
 * decisions, draw and outputs as spec_accept in stochastic sequence mode, but
 * the statistics pass reads only the draft rows q_logits.
 *   p_stats   device, fp32 pairs [B * (n + 1)][V / 32]: row_stats of
 *             w4a16_linear_logits for the rows of p_logits
 *   V         a multiple of 32
 *   other arguments, limits, workspace and errors as for spec_accept
 *   (q_logits and uniforms required).
 */
w4a16_status spec_accept_prestat(const float* p_logits, const float* p_stats, const float* q_logits,
                                 const int32_t* draft_ids, const float* uniforms, int B, int n, int V,
                                 int32_t* accepted_len, int32_t* next_token, void* workspace,
                                 size_t workspace_bytes, void* stream);

/* ------------------------------------------------------------------------
 * Allocation-free W4A16 linear. The pages have no counterpart to this call:
 * it exists for callers that cannot allocate device memory where they call
 * the linear — a plugin slot that passes only inputs and outputs, a runtime
 * that owns every device allocation, a hot path that must never reach
 * cudaMalloc. It computes exactly what w4a16_linear computes (same argument
 * rules, same kernels) but takes no workspace: its scratch is one static
 * device array of w4a16_linear_noalloc_scratch_bytes() bytes (24 MiB) that
 * every GPU this library is used on holds until the process exits. It calls
 * no cudaMalloc, cudaFree or allocating library routine.
 *  - The first call on a device looks up the array's device address
 *    (cudaGetSymbolAddress) with that device current; make that first call
 *    before any stream capture.
 *  - Each call clears the completion counters it needs (a cudaMemsetAsync on
 *    `stream`) before its kernel.
 *  - All calls share the array: calls that overlap on the GPU (other streams,
 *    other host threads) race and give wrong results. Serialise them.
 *  - A shape whose scratch would exceed the array returns W4A16_ERR_WORKSPACE.
 * ---------------------------------------------------------------------- */
size_t w4a16_linear_noalloc_scratch_bytes(void);
w4a16_status w4a16_linear_noalloc(const void* x, int M, int64_t K, const void* qweight_packed,
                                  const void* scales_packed, int64_t N, void* out, void* stream);

/* ------------------------------------------------------------------------
 * Device status: synchronises `stream`, reads and clears the device error
 * word of the current device. W4A16_OK, W4A16_ERR_DEVICE_TIMEOUT,
 * W4A16_ERR_DEVICE_INPUT or W4A16_ERR_CUDA.
 * ---------------------------------------------------------------------- */
w4a16_status w4a16_check_device_status(void* stream);

/* ------------------------------------------------------------------------
 * Host-side planning helpers (no GPU needed; exported so tests can check
 * the work split of the linear).
 * The linear cuts U = (N/128)*(K/128) (row-tile, group) units into R rounds
 * of C items (C = its grid size): round r covers units [rb[r], rb[r+1]) and
 * item i = r*C + j owns units [rb[r] + floor(j*len/C), rb[r] +
 * floor((j+1)*len/C)), len = rb[r+1] - rb[r]. Each round takes half of the
 * units left until items would hold fewer than min_units units, or
 * max_rounds (1..8) is reached; the last round takes the rest. CTA c takes
 * items c, c + C, ...; split tiles are summed in item order.
 *   w4a16_item_rounds  writes rb[0..R] (room for 9) and returns R, or 0 on
 *                      bad arguments (U < C, C < 1, min_units < 1).
 *   w4a16_item_begin   first unit of item i (i in [0, R*C]; R*C gives U),
 *                      -1 on bad arguments.
 *   w4a16_item_owner   item holding unit u (0 <= u < U), -1 on bad arguments.
 * ---------------------------------------------------------------------- */
int w4a16_item_rounds(int64_t U, int C, int min_units, int max_rounds, int64_t* rb);
int64_t w4a16_item_begin(int64_t U, int C, int min_units, int max_rounds, int i);
int64_t w4a16_item_owner(int64_t U, int C, int min_units, int max_rounds, int64_t u);

#ifdef __cplusplus
}
#endif

#endif /* W4A16SV_H_ */
