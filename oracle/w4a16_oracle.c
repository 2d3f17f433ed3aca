/*
 * Plain CPU oracle for the W4A16 speculative-verify hot path.
 *
 * TEST INFRASTRUCTURE ONLY. This file is the slow, obviously-correct statement
 * of what the GPU library computes. Only the tests, the smoke check and the
 * benchmark's CPU-baseline leg may load it. It shares no code, header, table
 * or helper with the CUDA library.
 *
 * Sources (page title, section):
 *  - "Speculative Decoding Meets Quantization" (Zhang et al. 2025; ordoresearch
 *    blog, menfem KB note and the shd-paper digest of arXiv:2505.22179):
 *    the target is a 4-bit *weight-only* quantised Llama-3-70B; the verify
 *    pass is a forward over several draft tokens; weight memory traffic is the
 *    bottleneck (abstract; "Research Landscape"; "The Compatibility Problem").
 *  - "Speculative Decoding이란?" (Korean tutorial), section 3 Steps 2-4,
 *    section 5 and section 6: per-position acceptance alpha_i =
 *    min(1, p(d_i)/q(d_i)), accept when u < alpha_i, sequential acceptance,
 *    and sampling from the corrected distribution at the first rejection;
 *    greedy decoding gives the target's own output.
 *  - "Speculative Decoding이란?", section 10.1 (Medusa tree-based attention),
 *    section 10.4 (ReDrafter dynamic tree attention) and section 8.7 (KV cache
 *    reuse in serving): the tree-masked attention of the verify pass and the
 *    compaction of the accepted path's keys and values.
 *  - The 4-bit format (int4 symmetric, group 128 along K, fp16 scale =
 *    max|w|/7, 8 nibbles per uint32) is fixed by the task specification, not
 *    by the pages.
 *
 * Readings where the pages are silent (each listed in the design notes):
 *  - nibble k%8 sits at bits 4*(k%8) of qweight[n][k/8], two's complement;
 *  - scale = fp16_rne(fp32(max|w| / 7)); q = clamp(rne(w / scale), -8, 7);
 *    a zero scale gives q = 0;
 *  - the linear accumulates in fp64 in ascending k and rounds the fp64 sum
 *    once, directly, to bf16 (round to nearest even);
 *  - softmax at temperature 1, no truncation, fp64 throughout;
 *  - the target supplies K+1 distributions; when all K drafts are accepted
 *    the extra token is drawn from the (K+1)-th;
 *  - sampling a distribution R with uniform u: the smallest x whose running
 *    sum (ascending x) exceeds u * sum(R);
 *  - the corrected distribution is max(0, P - Q) normalised; if it sums to 0
 *    the oracle samples P itself;
 *  - greedy: argmax over raw logits, ties to the smallest index; tree node j
 *    is accepted iff its parent is and draft[j] equals the argmax of the
 *    parent's row; the deepest accepted node wins, ties to the smaller index.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define GROUP 128

/* ---------------------------------------------------------------- numbers */

/* float -> bfloat16 bits, round to nearest even (NaN stays NaN). */
static uint16_t f32_to_bf16(float f) {
    uint32_t u;
    memcpy(&u, &f, 4);
    if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu)) return (uint16_t)((u >> 16) | 0x40);
    uint32_t lsb = (u >> 16) & 1u;
    u += 0x7FFFu + lsb;
    return (uint16_t)(u >> 16);
}

static float bf16_to_f32(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}

static float f16_to_f32(uint16_t h) {
    _Float16 v;
    memcpy(&v, &h, 2);
    return (float)v;
}

static uint16_t f32_to_f16(float f) {
    _Float16 v = (_Float16)f; /* IEEE round to nearest even */
    uint16_t h;
    memcpy(&h, &v, 2);
    return h;
}

/* double -> bfloat16 bits, round to nearest even in one step (no fp32
 * intermediate): the bf16 grid spacing at |v| = m * 2^e (m in [0.5, 1)) is
 * 2^(e - 8), never finer than the subnormal spacing 2^-133; |v| is scaled
 * onto that grid (exact: a power of two), rounded with rint (the default
 * rounding mode is to nearest, ties to even), and scaled back. The result has
 * at most 8 significant bits, so its conversion to float is exact (or inf
 * past the largest bf16). */
static uint16_t f64_to_bf16(double v) {
    if (isnan(v)) return 0x7FC0;
    int e;
    (void)frexp(fabs(v), &e);
    int q = e - 8;
    if (q < -133) q = -133;
    double r = ldexp(rint(ldexp(fabs(v), -q)), q);
    float f = (float)copysign(r, v); /* keeps the sign of -0 and of negatives that round to 0 */
    uint32_t u;
    memcpy(&u, &f, 4);
    return (uint16_t)(u >> 16);
}

uint16_t oracle_bf16_round(float f) { return f32_to_bf16(f); }
uint16_t oracle_bf16_round_f64(double v) { return f64_to_bf16(v); }
uint16_t oracle_f16_round(float f) { return f32_to_f16(f); }

/* ------------------------------------------------------------ 4-bit format */

/* Signed 4-bit code of weight (n, k) from the canonical packed array. */
static int code_at(const uint32_t* qweight, int64_t K, int64_t n, int64_t k) {
    uint32_t word = qweight[n * (K / 8) + k / 8];
    int nib = (int)((word >> (4 * (k % 8))) & 0xFu);
    return nib >= 8 ? nib - 16 : nib;
}

void oracle_unpack_codes(const uint32_t* qweight, int64_t N, int64_t K, int8_t* codes) {
    for (int64_t n = 0; n < N; ++n)
        for (int64_t k = 0; k < K; ++k) codes[n * K + k] = (int8_t)code_at(qweight, K, n, k);
}

void oracle_pack_codes(const int8_t* codes, int64_t N, int64_t K, uint32_t* qweight) {
    for (int64_t n = 0; n < N; ++n)
        for (int64_t w = 0; w < K / 8; ++w) {
            uint32_t word = 0;
            for (int j = 0; j < 8; ++j) word |= ((uint32_t)codes[n * K + w * 8 + j] & 0xFu) << (4 * j);
            qweight[n * (K / 8) + w] = word;
        }
}

/* w[n,k] = q * s; a 4-bit integer times an fp16 value is exact in fp32. */
void oracle_dequantize(const uint32_t* qweight, const uint16_t* scales, int64_t N, int64_t K, float* w) {
    for (int64_t n = 0; n < N; ++n)
        for (int64_t k = 0; k < K; ++k)
            w[n * K + k] = (float)code_at(qweight, K, n, k) * f16_to_f32(scales[n * (K / GROUP) + k / GROUP]);
}

/* Symmetric per-group quantiser: s = fp16(max|w| / 7), q = clamp(rne(w/s), -8, 7). */
void oracle_quantize(const float* w, int64_t N, int64_t K, uint32_t* qweight, uint16_t* scales) {
    int64_t G = K / GROUP;
    int8_t* codes = (int8_t*)malloc((size_t)(N * K));
    for (int64_t n = 0; n < N; ++n)
        for (int64_t g = 0; g < G; ++g) {
            const float* row = w + n * K + g * GROUP;
            float a = 0.0f;
            for (int j = 0; j < GROUP; ++j) a = fmaxf(a, fabsf(row[j]));
            uint16_t s16 = f32_to_f16(a / 7.0f);
            float s = f16_to_f32(s16);
            scales[n * G + g] = s16;
            for (int j = 0; j < GROUP; ++j) {
                int q = 0;
                if (s != 0.0f) {
                    float r = rintf(row[j] / s);
                    q = r > 7.0f ? 7 : (r < -8.0f ? -8 : (int)r);
                }
                codes[n * K + g * GROUP + j] = (int8_t)q;
            }
        }
    oracle_pack_codes(codes, N, K, qweight);
    free(codes);
}

/* ------------------------------------------------------------------ linear */

/* One output: y = sum_k x[m,k] * w[n,k] in fp64, ascending k. */
static double dot_row(const uint16_t* x, int64_t K, int64_t m, const uint32_t* qweight, const uint16_t* scales,
                      int64_t n) {
    double y = 0.0;
    for (int64_t k = 0; k < K; ++k) {
        float w = (float)code_at(qweight, K, n, k) * f16_to_f32(scales[n * (K / GROUP) + k / GROUP]);
        y += (double)bf16_to_f32(x[m * K + k]) * (double)w;
    }
    return y;
}

/* out[M,N] = bf16(x[M,K] . W^T), W dequantised from the canonical format.
 * y (optional, may be NULL) receives the unrounded fp64 sums. */
void oracle_linear(const uint16_t* x, int64_t M, int64_t K, const uint32_t* qweight, const uint16_t* scales,
                   int64_t N, uint16_t* out, double* y) {
#pragma omp parallel for schedule(static)
    for (int64_t n = 0; n < N; ++n)
        for (int64_t m = 0; m < M; ++m) {
            double v = dot_row(x, K, m, qweight, scales, n);
            out[m * N + n] = f64_to_bf16(v);
            if (y) y[m * N + n] = v;
        }
}

/* The same for a chosen set of output columns: out[M, ncols]. */
void oracle_linear_cols(const uint16_t* x, int64_t M, int64_t K, const uint32_t* qweight, const uint16_t* scales,
                        int64_t N, const int64_t* cols, int64_t ncols, uint16_t* out, double* y) {
    (void)N;
#pragma omp parallel for schedule(static)
    for (int64_t c = 0; c < ncols; ++c)
        for (int64_t m = 0; m < M; ++m) {
            double v = dot_row(x, K, m, qweight, scales, cols[c]);
            out[m * ncols + c] = f64_to_bf16(v);
            if (y) y[m * ncols + c] = v;
        }
}

/* ------------------------------------------------------------ accept step */

/* P = softmax(logits) in fp64 (temperature 1). */
static void softmax64(const float* logits, int V, double* P) {
    double mx = -INFINITY;
    for (int x = 0; x < V; ++x) mx = logits[x] > mx ? logits[x] : mx;
    double Z = 0.0;
    for (int x = 0; x < V; ++x) {
        P[x] = exp((double)logits[x] - mx);
        Z += P[x];
    }
    for (int x = 0; x < V; ++x) P[x] /= Z;
}

/* Inverse-CDF draw: smallest x with sum_{y<=x} R(y) > u * S (ascending x).
 * If rounding leaves no such x, the last x with R(x) > 0.
 * *margin receives the distance from t = u*S to the nearer end of the chosen
 * x's interval [sum_{y<x} R(y), sum_{y<=x} R(y)), divided by S: how far u
 * would have to move for the draw to change. */
static int sample_cdf(const double* R, int V, double S, double u, double* margin) {
    double t = u * S, c = 0.0;
    int last_pos = -1;
    for (int x = 0; x < V; ++x) {
        if (R[x] > 0.0) last_pos = x;
        double prev = c;
        c += R[x];
        if (c > t) {
            double m1 = fabs(t - prev), m2 = fabs(c - t);
            *margin = (m1 < m2 ? m1 : m2) / S;
            return x;
        }
    }
    *margin = 0.0;
    return last_pos < 0 ? 0 : last_pos;
}

/*
 * Stochastic speculative acceptance for a sequence draft.
 *  p [B][K+1][V] target logits, q [B][K][V] draft logits, d [B][K] draft ids,
 *  u [B][K+1] uniforms (u[.,0..K-1] for the tests, u[.,K] for the final draw).
 * Outputs accepted_len[B] in [0,K], next_token[B], alpha[B][K] (fp64, NAN for
 * positions not evaluated), margin_alpha[B] = the smallest |u_i - alpha_i|
 * over the evaluated positions (how close an accept decision came to going
 * the other way) and margin_cdf[B] = the final draw's CDF margin (see
 * sample_cdf), both fp64.
 */
void oracle_spec_accept_seq(const float* p, const float* q, const int32_t* d, const float* u, int B, int K, int V,
                            int32_t* accepted_len, int32_t* next_token, double* alpha, double* margin_alpha,
                            double* margin_cdf) {
#pragma omp parallel for schedule(dynamic)
    for (int b = 0; b < B; ++b) {
        double* P = (double*)malloc(sizeof(double) * (size_t)V);
        double* Q = (double*)malloc(sizeof(double) * (size_t)V);
        double* R = (double*)malloc(sizeof(double) * (size_t)V);
        const float* ub = u + (int64_t)b * (K + 1);
        double mg = INFINITY;
        int r = K;
        for (int i = 0; i < K; ++i) alpha[(int64_t)b * K + i] = NAN;
        for (int i = 0; i < K; ++i) {
            softmax64(p + ((int64_t)b * (K + 1) + i) * V, V, P);
            softmax64(q + ((int64_t)b * K + i) * V, V, Q);
            int di = d[(int64_t)b * K + i];
            double a = Q[di] > 0.0 ? fmin(1.0, P[di] / Q[di]) : 1.0;
            alpha[(int64_t)b * K + i] = a;
            double gap = fabs((double)ub[i] - a);
            mg = gap < mg ? gap : mg;
            if ((double)ub[i] < a) continue; /* accepted */
            r = i;
            break;
        }
        double S = 0.0;
        if (r < K) { /* P, Q hold row r: corrected distribution max(0, P - Q) */
            for (int x = 0; x < V; ++x) {
                R[x] = P[x] - Q[x] > 0.0 ? P[x] - Q[x] : 0.0;
                S += R[x];
            }
            if (S == 0.0) {
                for (int x = 0; x < V; ++x) R[x] = P[x];
                S = 0.0;
                for (int x = 0; x < V; ++x) S += R[x];
            }
        } else { /* all accepted: draw the extra token from the (K+1)-th row */
            softmax64(p + ((int64_t)b * (K + 1) + K) * V, V, R);
            for (int x = 0; x < V; ++x) S += R[x];
        }
        double cm;
        next_token[b] = sample_cdf(R, V, S, (double)ub[K], &cm);
        accepted_len[b] = r;
        margin_alpha[b] = mg;
        margin_cdf[b] = cm;
        free(P);
        free(Q);
        free(R);
    }
}

/*
 * Stochastic acceptance of a token tree. The pages give the rule for a
 * sequence draft only (the tutorial page, section 3 Steps 3-4); for a tree
 * this follows multi-step speculative sampling as SpecInfer (Miao et al.
 * 2024, "SpecInfer: Accelerating Large Language Model Serving with Tree-based
 * Speculative Inference and Verification", section 4.2) defines it, for
 * children drawn independently from the draft's distribution at their parent:
 *  - start at the root (node 0) with R = P_0, the target's distribution there;
 *  - at node u, try u's children in ascending index: child s with token x is
 *    accepted iff u_s < min(1, R(x) / Q_u(x)) (alpha = 1 when Q_u(x) = 0);
 *    on acceptance move to s with R = P_s; on rejection
 *    R <- max(0, R - Q_u) / sum (R is kept when that sums to 0) and try the
 *    next child;
 *  - when u has no child left, draw the next token from R with u_0.
 * p, q [B][n][V]: target and draft logits at every node (row j: after the
 * path root..j; q row j is the distribution j's children were drawn from);
 * d [B][n] (slot 0 unused), parents [B][n], u [B][n] (u_j tests node j,
 * u_0 the final draw). Outputs accepted_len (the final node's depth),
 * next_token, accepted_node, margin_alpha (smallest |u_s - alpha| over the
 * tests made) and margin_cdf (see sample_cdf). fp64 throughout.
 */
void oracle_spec_accept_tree(const float* p, const float* q, const int32_t* d, const int32_t* parents, const float* u,
                             int B, int n, int V, int32_t* accepted_len, int32_t* next_token, int32_t* accepted_node,
                             double* margin_alpha, double* margin_cdf) {
#pragma omp parallel for schedule(dynamic)
    for (int b = 0; b < B; ++b) {
        double* R = (double*)malloc(sizeof(double) * (size_t)V);
        double* Q = (double*)malloc(sizeof(double) * (size_t)V);
        const int32_t* par = parents + (int64_t)b * n;
        const float* ub = u + (int64_t)b * n;
        int node = 0, depth = 0;
        double mg = INFINITY;
        softmax64(p + (int64_t)b * n * V, V, R);
        softmax64(q + (int64_t)b * n * V, V, Q);
        for (;;) {
            int accepted = -1;
            for (int s = node + 1; s < n; ++s) {
                if (par[s] != node) continue;
                const int x = d[(int64_t)b * n + s];
                const double a = Q[x] > 0.0 ? fmin(1.0, R[x] / Q[x]) : 1.0;
                const double gap = fabs((double)ub[s] - a);
                mg = gap < mg ? gap : mg;
                if ((double)ub[s] < a) {
                    accepted = s;
                    break;
                }
                double S = 0.0;
                for (int y = 0; y < V; ++y) S += R[y] - Q[y] > 0.0 ? R[y] - Q[y] : 0.0;
                if (S > 0.0)
                    for (int y = 0; y < V; ++y) R[y] = (R[y] - Q[y] > 0.0 ? R[y] - Q[y] : 0.0) / S;
            }
            if (accepted < 0) break;
            node = accepted;
            ++depth;
            softmax64(p + ((int64_t)b * n + node) * V, V, R);
            softmax64(q + ((int64_t)b * n + node) * V, V, Q);
        }
        double S = 0.0, cm;
        for (int y = 0; y < V; ++y) S += R[y];
        next_token[b] = sample_cdf(R, V, S, (double)ub[0], &cm);
        accepted_len[b] = depth;
        accepted_node[b] = node;
        margin_alpha[b] = mg;
        margin_cdf[b] = cm;
        free(R);
        free(Q);
    }
}

/* argmax over raw logits, ties to the smallest index. */
static int argmax_row(const float* row, int V) {
    int best = 0;
    for (int x = 1; x < V; ++x)
        if (row[x] > row[best]) best = x;
    return best;
}

/*
 * Greedy verification of a token tree. p [B][n][V]: row j is the target's
 * distribution after the path root..j. draft [B][n] (slot 0 unused), parents
 * [B][n] (parent[0] = -1, 0 <= parent[j] < j).
 * accepted_len = depth of the deepest accepted node; next = argmax of its row;
 * accepted_node (may be NULL) = that node's index.
 */
void oracle_greedy_tree(const float* p, const int32_t* draft, const int32_t* parents, int B, int n, int V,
                        int32_t* accepted_len, int32_t* next_token, int32_t* accepted_node) {
#pragma omp parallel for schedule(dynamic)
    for (int b = 0; b < B; ++b) {
        int* acc = (int*)malloc(sizeof(int) * (size_t)n);
        int* depth = (int*)malloc(sizeof(int) * (size_t)n);
        const float* pb = p + (int64_t)b * n * V;
        acc[0] = 1;
        depth[0] = 0;
        int best = 0;
        for (int j = 1; j < n; ++j) {
            int par = parents[(int64_t)b * n + j];
            depth[j] = depth[par] + 1;
            acc[j] = acc[par] && draft[(int64_t)b * n + j] == argmax_row(pb + (int64_t)par * V, V);
            if (acc[j] && depth[j] > depth[best]) best = j;
        }
        accepted_len[b] = depth[best];
        next_token[b] = argmax_row(pb + (int64_t)best * V, V);
        if (accepted_node) accepted_node[b] = best;
        free(acc);
        free(depth);
    }
}

/* Greedy verification of a sequence draft: p [B][K+1][V], draft [B][K]. */
void oracle_greedy_chain(const float* p, const int32_t* draft, int B, int K, int V, int32_t* accepted_len,
                         int32_t* next_token) {
#pragma omp parallel for schedule(dynamic)
    for (int b = 0; b < B; ++b) {
        const float* pb = p + (int64_t)b * (K + 1) * V;
        int r = K;
        for (int i = 0; i < K; ++i)
            if (draft[(int64_t)b * K + i] != argmax_row(pb + (int64_t)i * V, V)) {
                r = i;
                break;
            }
        accepted_len[b] = r;
        next_token[b] = argmax_row(pb + (int64_t)r * V, V);
    }
}

/* ------------------------------------------------ tree-masked attention */

/*
 * Attention of the verify pass over a token tree (the tutorial page, section
 * 10.1, Medusa "tree-based attention": the candidate continuations form a
 * tree and the target checks them in one pass; section 10.4, ReDrafter's
 * dynamic tree attention; a sequence draft is the chain parent[j] = j - 1).
 *
 * Readings (the pages give no formula):
 *  - every tree node j is one query position; it attends to the whole
 *    committed prefix (cache positions 0 .. lens[b] - 1) and to the tree
 *    nodes on its own root path, itself included, whose keys and values the
 *    verify forward has written at cache positions lens[b] + node index;
 *  - scaled dot-product attention, scale given (1/sqrt(D) in use), softmax at
 *    temperature 1 over the allowed keys;
 *  - grouped heads: query head h reads key/value head h / (H / Hkv).
 *
 * q bf16 bits [B][n][H][D]; k_cache, v_cache bf16 bits [B][Hkv][Lcap][D];
 * lens [B]; parents [B][n] (parent[0] = -1, 0 <= parent[j] < j) or NULL for
 * the chain; out fp64 [B][n][H][D]. Scores, softmax and the weighted sum in
 * fp64. absw (may be NULL) [B][n][H][D]: sum over the allowed keys of
 * softmax weight * |v|, the scale of the rounding errors a reduced-precision
 * weighted sum can make.
 */
void oracle_tree_attention(const uint16_t* q, const uint16_t* k_cache, const uint16_t* v_cache, const int32_t* lens,
                           const int32_t* parents, int B, int n, int H, int Hkv, int D, int Lcap, double scale,
                           double* out, double* absw) {
    const int G = H / Hkv;
#pragma omp parallel for collapse(2) schedule(dynamic)
    for (int b = 0; b < B; ++b)
        for (int j = 0; j < n; ++j) {
            const int L = lens[b];
            const int T = L + n;
            char* allowed = (char*)calloc((size_t)T, 1);
            double* s = (double*)malloc(sizeof(double) * (size_t)T);
            for (int x = 0; x < L; ++x) allowed[x] = 1;
            for (int i = j; i >= 0; i = parents ? parents[(int64_t)b * n + i] : i - 1) allowed[L + i] = 1;
            for (int h = 0; h < H; ++h) {
                const int kvh = h / G;
                const uint16_t* qr = q + (((int64_t)b * n + j) * H + h) * D;
                const uint16_t* kb = k_cache + ((int64_t)b * Hkv + kvh) * Lcap * D;
                const uint16_t* vb = v_cache + ((int64_t)b * Hkv + kvh) * Lcap * D;
                double m = -INFINITY;
                for (int x = 0; x < T; ++x) {
                    if (!allowed[x]) continue;
                    double dot = 0.0;
                    for (int d = 0; d < D; ++d)
                        dot += (double)bf16_to_f32(qr[d]) * (double)bf16_to_f32(kb[(int64_t)x * D + d]);
                    s[x] = dot * scale;
                    if (s[x] > m) m = s[x];
                }
                double* o = out + (((int64_t)b * n + j) * H + h) * D;
                double* a = absw ? absw + (((int64_t)b * n + j) * H + h) * D : NULL;
                for (int d = 0; d < D; ++d) o[d] = 0.0;
                if (a)
                    for (int d = 0; d < D; ++d) a[d] = 0.0;
                double Z = 0.0;
                for (int x = 0; x < T; ++x) {
                    if (!allowed[x]) continue;
                    const double w = exp(s[x] - m);
                    Z += w;
                    for (int d = 0; d < D; ++d) {
                        const double vv = (double)bf16_to_f32(vb[(int64_t)x * D + d]);
                        o[d] += w * vv;
                        if (a) a[d] += w * fabs(vv);
                    }
                }
                for (int d = 0; d < D; ++d) o[d] /= Z;
                if (a)
                    for (int d = 0; d < D; ++d) a[d] /= Z;
            }
            free(allowed);
            free(s);
        }
}

/*
 * KV compaction after verification (the tutorial page, section 8.7: the
 * serving stack must not waste cache on rejected tokens; ReDrafter's dynamic
 * tree attention). The tree nodes' keys and values sit at cache positions
 * lens[b] + node index; after acceptance the nodes on the root path of the
 * deepest accepted node (root first) move to positions lens[b] + 0, 1, ...,
 * depth, and the committed length becomes lens[b] + depth + 1. Reading: the
 * root (node 0, the last committed token, verified with the drafts) is
 * always kept; positions past the new length keep whatever they held.
 *
 * caches bf16 bits [n_layers][B][Hkv][Lcap][D], updated in place; parents
 * [B][n] or NULL (chain); accepted_node [B]; new_lens [B].
 */
void oracle_kv_compact(uint16_t* k_cache, uint16_t* v_cache, const int32_t* lens, const int32_t* parents,
                       const int32_t* accepted_node, int B, int n, int Hkv, int D, int Lcap, int n_layers,
                       int32_t* new_lens) {
    for (int b = 0; b < B; ++b) {
        int path[1025];
        int depth = 0;
        for (int i = accepted_node[b]; i >= 0 && depth < 1025; i = parents ? parents[(int64_t)b * n + i] : i - 1)
            path[depth++] = i;
        /* path[depth - 1] is the root: reverse into root-first order */
        for (int a = 0, z = depth - 1; a < z; ++a, --z) {
            const int t = path[a];
            path[a] = path[z];
            path[z] = t;
        }
        const int L = lens[b];
        new_lens[b] = L + depth;
        uint16_t* tmp = (uint16_t*)malloc(sizeof(uint16_t) * (size_t)n * D);
        for (int layer = 0; layer < n_layers; ++layer)
            for (int h = 0; h < Hkv; ++h)
                for (int c = 0; c < 2; ++c) {
                    uint16_t* base = (c ? v_cache : k_cache) + (((int64_t)layer * B + b) * Hkv + h) * Lcap * D;
                    memcpy(tmp, base + (int64_t)L * D, sizeof(uint16_t) * (size_t)n * D);
                    for (int d = 0; d < depth; ++d)
                        memcpy(base + (int64_t)(L + d) * D, tmp + (int64_t)path[d] * D, sizeof(uint16_t) * (size_t)D);
                }
        free(tmp);
    }
}

/* Threads the parallel loops use from now on (the timed CPU baseline runs
 * once on one thread and once on every host core); returns the new count. */
int oracle_set_num_threads(int n) {
#ifdef _OPENMP
    extern void omp_set_num_threads(int);
    extern int omp_get_max_threads(void);
    if (n > 0) omp_set_num_threads(n);
    return omp_get_max_threads();
#else
    (void)n;
    return 1;
#endif
}

int oracle_num_threads(void) {
#ifdef _OPENMP
    extern int omp_get_max_threads(void);
    return omp_get_max_threads();
#else
    return 1;
#endif
}
