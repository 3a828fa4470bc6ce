/*
 * oracle.c -- plain, slow fp64 CPU oracle for the DSA hot path.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the
 * benchmark's CPU-baseline leg call this library.  It shares no code,
 * header, table or helper with the CUDA library: every input arrives as a
 * raw array (bf16 as its 16-bit pattern, widened here exactly).
 *
 * What it computes, and where the pages define it:
 *
 *  oracle_indexer_scores  -- lightning-indexer score of query position t
 *      against every causal history position s <= t,
 *          I[t,s] = sum_h w[t,h] * ReLU( sum_d q_idx[t,h,d] * k_idx[s,d] ),
 *      32 heads x 128 dims, one shared 128-dim key per token, arithmetic in
 *      floating point wider than the bf16 inputs ("GLM-5.1 架构深度拆解",
 *      section 3.2 "Indexer 公式" Steps 4-5 and section 3.6 Step 5: two
 *      einsums in fp32 with a ReLU between them; the GLM-5 explainer page,
 *      indexer paragraph).  Any positive softmax_scale of the pages factors
 *      out of the ReLU and is taken to be folded into w.
 *  oracle_topk            -- causal top-k of one fp32 score row
 *      (section 3.6 Steps 6-7: mask s > t, keep min(index_topk, length);
 *      explainer page: "shorter than 2048 keeps all"; section 3.4: the
 *      top-k must be deterministic).  Reading used here: ties are broken
 *      toward the lower position, -0.0 equals +0.0, the chosen positions
 *      are emitted in ascending order and the tail is padded with -1.
 *  oracle_sparse_mla      -- attention of one query's 64 heads over the
 *      selected rows of the latent cache in absorbed form: logits
 *      sm_scale * q[h] . kv[s] over all 576 columns (512 latent + 64 RoPE
 *      key shared by every head), softmax over the selected rows, output
 *      the softmax-weighted sum of the first 512 columns (section 3.1
 *      "DSA 原理" step 2, section 4.2 shared single-head RoPE key, section
 *      2.5 576-wide cached row; explainer page: the top-2048 ids only
 *      drive the gather).  Also returns lse = m + log(sum exp(l - m)).
 *  oracle_masked_mla      -- the same attention written the way the pages'
 *      attention layer does it (section 4.5 Steps 6-7): a dense row of
 *      -inf with 0 scattered at the selected positions, plus the causal
 *      mask, added to the logits of *every* cached position before the
 *      softmax.  Used to check the gather form against the mask form.
 *
 * MLA around the path (section 4.5 Steps 1-4 and 7-8; section 4.1: the
 * cached row is the 512-dim compressed KV after kv_a_layernorm plus the
 * 64-dim RoPE key; kv_b_proj expands it to 64 heads x (192 nope + 256 v);
 * o_proj maps the 64 x 256 head outputs to the 6144-dim hidden state):
 *  oracle_mla_expanded    -- the pages' expanded path for selected rows:
 *      k_nope = W_UK[h] c, v = W_UV[h] c for every attended cached row
 *      (W_UK[h], W_UV[h] = rows h*448 .. +191 and h*448+192 .. +447 of
 *      kv_b_proj's weight), logits sm_scale*(q_nope.k_nope + q_pe.k_pe)
 *      plus the index mask and the causal mask, softmax, o[h] = sum p v,
 *      y = o_proj(o).
 *  oracle_mla_absorb_q    -- the absorbed query: q[h, 0:512] =
 *      W_UK[h]^T q_nope[h], q[h, 512:576] = q_pe[h] (the identity
 *      q_nope.(W_UK c) = (W_UK^T q_nope).c moves kv_b_proj's key half onto
 *      the query, so attention can run on the cached rows directly).
 *  oracle_mla_output      -- the absorbed output: o[h] = W_UV[h] o_lat[h]
 *      (sum p (W_UV c) = W_UV sum p c), then y = o_proj(o).
 *
 * The index-key producer ("GLM-5.1 架构深度拆解", section 3.6 Steps 2-4):
 *  oracle_index_key       -- for each new token with hidden state x:
 *      k = LayerNorm(wk x) over its 128 dims (k_norm: mean, biased
 *      variance, eps, then gamma and beta), RoPE on the first 64 dims with
 *      the caller's cos / sin of the token's position (the rotate-half
 *      form: pairs (i, i + 32)), the last 64 dims unchanged; and the head
 *      weights w = (weights_proj x) * 32^-1/2.  The pages give neither the
 *      rotary base nor the pairing; the cos / sin rows come in as inputs
 *      (the rotary table of the position embedding) and the pairing is the
 *      rotate-half one of the pages' apply_rotary_pos_emb.
 *
 * Reduced-precision index keys (the pages give no recipe; the reading used
 * here is stated once and followed by the GPU path):
 *  oracle_e4m3_decode / oracle_e4m3_encode -- the OCP 8-bit floating point
 *      E4M3 format: 1 sign, 4 exponent (bias 7), 3 mantissa bits; normals
 *      (1 + m/8) 2^(e-7), subnormals (m/8) 2^-6, S.1111.111 is NaN, no
 *      infinities, largest finite 448; encoding rounds to nearest, ties to
 *      the even code, and saturates finite values beyond 448 to +-448.
 *  oracle_quantize_fp8    -- one scale per row of n values: amax / 448 (1 when
 *      the row is all zero); codes = encode(v / scale), scale and quotient
 *      in single precision.  Index keys use one row per key (128 dims),
 *      indexer queries one row per (token, head).
 *  oracle_indexer_scores_fp8 -- the lightning-indexer score on the
 *      dequantised values: I[t,s] = sum_h w[t,h] ReLU(sq[t,h] sk[s]
 *      sum_d q8[t,h,d] k8[s,d]) with q8, k8 decoded exactly.
 *
 * Plain loops, no blocking, no reordering; OpenMP only splits query rows.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { O_HIDX = 32, O_DIDX = 128, O_H = 64, O_DQK = 576, O_DV = 512 };
enum { O_DNOPE = 192, O_DROPE = 64, O_DVH = 256, O_KVB = 448, O_HID = 6144 };
enum { O_KROPE = 64 };   /* the RoPE part of an index key: its first 64 dims */

static double widen_bf16(uint16_t b) {
    uint32_t u = ((uint32_t)b) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* sequence b and position t of packed query row r */
static void locate_row(int B, const int32_t* q_off, const int32_t* ctx_len, int32_t r,
                       int* b_out, int64_t* t_out) {
    int b = 0;
    while (b + 1 < B && q_off[b + 1] <= r) b++;
    int64_t nq = (int64_t)q_off[b + 1] - q_off[b];
    *b_out = b;
    *t_out = (int64_t)ctx_len[b] - nq + ((int64_t)r - q_off[b]);
}

int oracle_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

void oracle_set_num_threads(int n) {
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

/* out[j*ld + s] = I[t,s] for s in [0, t] of requested row rows[j]; other
 * entries of the row are left untouched. */
void oracle_indexer_scores(int B, const int32_t* q_off, const int32_t* ctx_len, int64_t stride,
                           const uint16_t* q_idx, const float* w, const uint16_t* k_idx,
                           int nrows, const int32_t* rows, double* out, int64_t ld) {
#pragma omp parallel for schedule(dynamic, 1)
    for (int j = 0; j < nrows; j++) {
        int b;
        int64_t t;
        locate_row(B, q_off, ctx_len, rows[j], &b, &t);
        const uint16_t* qr = q_idx + (int64_t)rows[j] * O_HIDX * O_DIDX;
        const float* wr = w + (int64_t)rows[j] * O_HIDX;
        for (int64_t s = 0; s <= t; s++) {
            const uint16_t* ks = k_idx + ((int64_t)b * stride + s) * O_DIDX;
            double score = 0.0;
            for (int h = 0; h < O_HIDX; h++) {
                double dot = 0.0;
                for (int d = 0; d < O_DIDX; d++)
                    dot += widen_bf16(qr[h * O_DIDX + d]) * widen_bf16(ks[d]);
                double relu = dot > 0.0 ? dot : 0.0;
                score += (double)wr[h] * relu;
            }
            out[(int64_t)j * ld + s] = score;
        }
    }
}

typedef struct {
    float v;
    int32_t s;
} cand_t;

/* larger score first; equal scores (-0.0 == +0.0) -> lower position first */
static int by_score_then_pos(const void* pa, const void* pb) {
    const cand_t* a = (const cand_t*)pa;
    const cand_t* b = (const cand_t*)pb;
    if (a->v > b->v) return -1;
    if (a->v < b->v) return 1;
    return (a->s > b->s) - (a->s < b->s);
}

static int by_pos(const void* pa, const void* pb) {
    int32_t a = *(const int32_t*)pa, b = *(const int32_t*)pb;
    return (a > b) - (a < b);
}

/* idx_out[j*k + i]: for requested row rows[j] (position t) the min(k, t+1)
 * positions with the largest scores[j*ld + s], s <= t, ascending, then -1. */
void oracle_topk(int B, const int32_t* q_off, const int32_t* ctx_len,
                 const float* scores, int64_t ld, int nrows, const int32_t* rows, int k,
                 int32_t* idx_out) {
#pragma omp parallel for schedule(dynamic, 1)
    for (int j = 0; j < nrows; j++) {
        int b;
        int64_t t;
        locate_row(B, q_off, ctx_len, rows[j], &b, &t);
        int64_t n = t + 1;
        int64_t m = n < k ? n : k;
        cand_t* c = (cand_t*)malloc((size_t)(n > 0 ? n : 1) * sizeof(cand_t));
        for (int64_t s = 0; s < n; s++) {
            c[s].v = scores[(int64_t)j * ld + s];
            c[s].s = (int32_t)s;
        }
        qsort(c, (size_t)n, sizeof(cand_t), by_score_then_pos);
        int32_t* o = idx_out + (int64_t)j * k;
        for (int64_t i = 0; i < m; i++) o[i] = c[i].s;
        qsort(o, (size_t)m, sizeof(int32_t), by_pos);
        for (int64_t i = m; i < k; i++) o[i] = -1;
        free(c);
    }
}

/* out[j, h, 0:512], lse[j, h] for requested row rows[j], attending over the
 * positions idx[j*k + i] >= 0. */
void oracle_sparse_mla(int B, const int32_t* q_off, const int32_t* ctx_len, int64_t stride,
                       const uint16_t* q, const uint16_t* kv, const int32_t* idx, int k,
                       double sm_scale, int nrows, const int32_t* rows, double* out,
                       double* lse) {
#pragma omp parallel for schedule(dynamic, 1)
    for (int j = 0; j < nrows; j++) {
        int b;
        int64_t t;
        locate_row(B, q_off, ctx_len, rows[j], &b, &t);
        const int32_t* sel = idx + (int64_t)j * k;
        double* logit = (double*)malloc((size_t)k * sizeof(double));
        for (int h = 0; h < O_H; h++) {
            const uint16_t* qh = q + ((int64_t)rows[j] * O_H + h) * O_DQK;
            double mx = -INFINITY;
            for (int i = 0; i < k; i++) {
                if (sel[i] < 0) continue;
                const uint16_t* row = kv + ((int64_t)b * stride + sel[i]) * O_DQK;
                double dot = 0.0;
                for (int d = 0; d < O_DQK; d++) dot += widen_bf16(qh[d]) * widen_bf16(row[d]);
                logit[i] = sm_scale * dot;
                if (logit[i] > mx) mx = logit[i];
            }
            double* o = out + ((int64_t)j * O_H + h) * O_DV;
            for (int d = 0; d < O_DV; d++) o[d] = 0.0;
            double z = 0.0;
            for (int i = 0; i < k; i++) {
                if (sel[i] < 0) continue;
                const uint16_t* row = kv + ((int64_t)b * stride + sel[i]) * O_DQK;
                double p = exp(logit[i] - mx);
                z += p;
                for (int d = 0; d < O_DV; d++) o[d] += p * widen_bf16(row[d]);
            }
            if (z > 0.0) {
                for (int d = 0; d < O_DV; d++) o[d] /= z;
                lse[(int64_t)j * O_H + h] = mx + log(z);
            } else {
                lse[(int64_t)j * O_H + h] = -INFINITY;
            }
        }
        free(logit);
    }
}

/* The mask formulation: logits over every cached position s < ctx_len[b]
 * plus index_mask[s] (0 where s is selected, -inf elsewhere) plus the
 * causal mask (0 for s <= t, -inf for s > t); softmax over the whole row. */
void oracle_masked_mla(int B, const int32_t* q_off, const int32_t* ctx_len, int64_t stride,
                       const uint16_t* q, const uint16_t* kv, const int32_t* idx, int k,
                       double sm_scale, int nrows, const int32_t* rows, double* out,
                       double* lse) {
#pragma omp parallel for schedule(dynamic, 1)
    for (int j = 0; j < nrows; j++) {
        int b;
        int64_t t;
        locate_row(B, q_off, ctx_len, rows[j], &b, &t);
        int64_t ctx = ctx_len[b];
        double* index_mask = (double*)malloc((size_t)(ctx > 0 ? ctx : 1) * sizeof(double));
        double* logit = (double*)malloc((size_t)(ctx > 0 ? ctx : 1) * sizeof(double));
        for (int64_t s = 0; s < ctx; s++) index_mask[s] = -INFINITY;
        for (int i = 0; i < k; i++)
            if (idx[(int64_t)j * k + i] >= 0 && idx[(int64_t)j * k + i] < ctx)
                index_mask[idx[(int64_t)j * k + i]] = 0.0;
        for (int h = 0; h < O_H; h++) {
            const uint16_t* qh = q + ((int64_t)rows[j] * O_H + h) * O_DQK;
            double mx = -INFINITY;
            for (int64_t s = 0; s < ctx; s++) {
                const uint16_t* row = kv + ((int64_t)b * stride + s) * O_DQK;
                double dot = 0.0;
                for (int d = 0; d < O_DQK; d++) dot += widen_bf16(qh[d]) * widen_bf16(row[d]);
                double causal = s <= t ? 0.0 : -INFINITY;
                logit[s] = sm_scale * dot + index_mask[s] + causal;
                if (logit[s] > mx) mx = logit[s];
            }
            double* o = out + ((int64_t)j * O_H + h) * O_DV;
            for (int d = 0; d < O_DV; d++) o[d] = 0.0;
            double z = 0.0;
            for (int64_t s = 0; s < ctx; s++) {
                double p = isinf(logit[s]) && logit[s] < 0 ? 0.0 : exp(logit[s] - mx);
                if (p == 0.0) continue;
                const uint16_t* row = kv + ((int64_t)b * stride + s) * O_DQK;
                z += p;
                for (int d = 0; d < O_DV; d++) o[d] += p * widen_bf16(row[d]);
            }
            if (z > 0.0) {
                for (int d = 0; d < O_DV; d++) o[d] /= z;
                lse[(int64_t)j * O_H + h] = mx + log(z);
            } else {
                lse[(int64_t)j * O_H + h] = -INFINITY;
            }
        }
        free(index_mask);
        free(logit);
    }
}

/* q_out[t, h, 0:512] = W_UK[h]^T q_nope[t, h]; q_out[t, h, 512:576] = q_pe[t, h]. */
void oracle_mla_absorb_q(int T, const uint16_t* q_nope, const uint16_t* q_pe, const uint16_t* w_kvb,
                         double* q_out) {
#pragma omp parallel for schedule(dynamic, 1)
    for (int t = 0; t < T; t++) {
        for (int h = 0; h < O_H; h++) {
            double* o = q_out + ((int64_t)t * O_H + h) * O_DQK;
            for (int d = 0; d < O_DV; d++) o[d] = 0.0;
            for (int i = 0; i < O_DNOPE; i++) {
                double qn = widen_bf16(q_nope[((int64_t)t * O_H + h) * O_DNOPE + i]);
                const uint16_t* wrow = w_kvb + ((int64_t)h * O_KVB + i) * O_DV;
                for (int d = 0; d < O_DV; d++) o[d] += qn * widen_bf16(wrow[d]);
            }
            for (int d = 0; d < O_DROPE; d++)
                o[O_DV + d] = widen_bf16(q_pe[((int64_t)t * O_H + h) * O_DROPE + d]);
        }
    }
}

/* o_mid[t, h, e] = sum_d W_UV[h][e, d] o_lat[t, h, d];
 * y[t, n] = sum_{h, e} W_o[n, h*256 + e] o_mid[t, h, e]. */
void oracle_mla_output(int T, const double* o_lat, const uint16_t* w_kvb, const uint16_t* w_o, double* o_mid,
                       double* y) {
#pragma omp parallel for schedule(dynamic, 1)
    for (int t = 0; t < T; t++) {
        double* om = o_mid + (int64_t)t * O_H * O_DVH;
        for (int h = 0; h < O_H; h++) {
            const double* ol = o_lat + ((int64_t)t * O_H + h) * O_DV;
            for (int e = 0; e < O_DVH; e++) {
                const uint16_t* wrow = w_kvb + ((int64_t)h * O_KVB + O_DNOPE + e) * O_DV;
                double acc = 0.0;
                for (int d = 0; d < O_DV; d++) acc += widen_bf16(wrow[d]) * ol[d];
                om[h * O_DVH + e] = acc;
            }
        }
        for (int n = 0; n < O_HID; n++) {
            const uint16_t* wrow = w_o + (int64_t)n * (O_H * O_DVH);
            double acc = 0.0;
            for (int c = 0; c < O_H * O_DVH; c++) acc += widen_bf16(wrow[c]) * om[c];
            y[(int64_t)t * O_HID + n] = acc;
        }
    }
}

/* The expanded path for requested rows: every cached position s < ctx_len[b]
 * gets index_mask[s] + causal[s]; where both are 0 the logit is
 * sm_scale * (q_nope . k_nope[s] + q_pe . k_pe[s]) with k_nope, v expanded
 * from the cached latent row by kv_b_proj; elsewhere the logit is -inf (its
 * finite part does not matter and is not computed).  o_mid[j, h, 0:256],
 * y[j, 0:6144]. */
void oracle_mla_expanded(int B, const int32_t* q_off, const int32_t* ctx_len, int64_t stride,
                         const uint16_t* q_nope, const uint16_t* q_pe, const uint16_t* kv, const uint16_t* w_kvb,
                         const uint16_t* w_o, const int32_t* idx, int k, double sm_scale, int nrows,
                         const int32_t* rows, double* o_mid, double* y) {
#pragma omp parallel for schedule(dynamic, 1)
    for (int j = 0; j < nrows; j++) {
        int b;
        int64_t t;
        locate_row(B, q_off, ctx_len, rows[j], &b, &t);
        int64_t ctx = ctx_len[b];
        double* mask = (double*)malloc((size_t)(ctx > 0 ? ctx : 1) * sizeof(double));
        double* logit = (double*)malloc((size_t)(ctx > 0 ? ctx : 1) * sizeof(double));
        double* kn = (double*)malloc(O_DNOPE * sizeof(double));
        double* v = (double*)malloc(O_DVH * sizeof(double));
        for (int64_t s = 0; s < ctx; s++) mask[s] = -INFINITY;
        for (int i = 0; i < k; i++) {
            int32_t s = idx[(int64_t)j * k + i];
            if (s >= 0 && s < ctx) mask[s] = 0.0;
        }
        double* om = o_mid + (int64_t)j * O_H * O_DVH;
        for (int h = 0; h < O_H; h++) {
            const uint16_t* qn = q_nope + ((int64_t)rows[j] * O_H + h) * O_DNOPE;
            const uint16_t* qp = q_pe + ((int64_t)rows[j] * O_H + h) * O_DROPE;
            double mx = -INFINITY;
            for (int64_t s = 0; s < ctx; s++) {
                double causal = s <= t ? 0.0 : -INFINITY;
                if (mask[s] + causal < 0.0) {
                    logit[s] = -INFINITY;
                    continue;
                }
                const uint16_t* row = kv + ((int64_t)b * stride + s) * O_DQK;
                double dot = 0.0;
                for (int i = 0; i < O_DNOPE; i++) {
                    const uint16_t* wrow = w_kvb + ((int64_t)h * O_KVB + i) * O_DV;
                    double acc = 0.0;
                    for (int d = 0; d < O_DV; d++) acc += widen_bf16(wrow[d]) * widen_bf16(row[d]);
                    kn[i] = acc;
                }
                for (int i = 0; i < O_DNOPE; i++) dot += widen_bf16(qn[i]) * kn[i];
                for (int d = 0; d < O_DROPE; d++) dot += widen_bf16(qp[d]) * widen_bf16(row[O_DV + d]);
                logit[s] = sm_scale * dot + mask[s] + causal;
                if (logit[s] > mx) mx = logit[s];
            }
            for (int e = 0; e < O_DVH; e++) om[h * O_DVH + e] = 0.0;
            double z = 0.0;
            for (int64_t s = 0; s < ctx; s++) {
                if (logit[s] == -INFINITY) continue;
                const uint16_t* row = kv + ((int64_t)b * stride + s) * O_DQK;
                double p = exp(logit[s] - mx);
                z += p;
                for (int e = 0; e < O_DVH; e++) {
                    const uint16_t* wrow = w_kvb + ((int64_t)h * O_KVB + O_DNOPE + e) * O_DV;
                    double acc = 0.0;
                    for (int d = 0; d < O_DV; d++) acc += widen_bf16(wrow[d]) * widen_bf16(row[d]);
                    v[e] = acc;
                }
                for (int e = 0; e < O_DVH; e++) om[h * O_DVH + e] += p * v[e];
            }
            for (int e = 0; e < O_DVH; e++) om[h * O_DVH + e] = z > 0.0 ? om[h * O_DVH + e] / z : 0.0;
        }
        for (int n = 0; n < O_HID; n++) {
            const uint16_t* wrow = w_o + (int64_t)n * (O_H * O_DVH);
            double acc = 0.0;
            for (int c = 0; c < O_H * O_DVH; c++) acc += widen_bf16(wrow[c]) * om[c];
            y[(int64_t)j * O_HID + n] = acc;
        }
        free(mask);
        free(logit);
        free(kn);
        free(v);
    }
}

/* k_out[t, 0:128] and w_out[t, 0:32] for T tokens. */
void oracle_index_key(int T, const uint16_t* x, const uint16_t* wk, const double* gamma, const double* beta,
                      double eps, const double* cos_t, const double* sin_t, const uint16_t* ww, double* k_out,
                      double* w_out) {
#pragma omp parallel for schedule(dynamic, 1)
    for (int t = 0; t < T; t++) {
        const uint16_t* xt = x + (int64_t)t * O_HID;
        double y[O_DIDX], z[O_DIDX];
        for (int j = 0; j < O_DIDX; j++) {
            double acc = 0.0;
            for (int c = 0; c < O_HID; c++) acc += widen_bf16(wk[(int64_t)j * O_HID + c]) * widen_bf16(xt[c]);
            y[j] = acc;
        }
        double mean = 0.0;
        for (int j = 0; j < O_DIDX; j++) mean += y[j];
        mean /= O_DIDX;
        double var = 0.0;
        for (int j = 0; j < O_DIDX; j++) var += (y[j] - mean) * (y[j] - mean);
        var /= O_DIDX;
        for (int j = 0; j < O_DIDX; j++) z[j] = (y[j] - mean) / sqrt(var + eps) * gamma[j] + beta[j];
        double* kt = k_out + (int64_t)t * O_DIDX;
        const double* ct = cos_t + (int64_t)t * O_KROPE;
        const double* st = sin_t + (int64_t)t * O_KROPE;
        for (int i = 0; i < O_KROPE; i++) {
            /* rotate_half: (-z[i + 32], z[i - 32]) */
            double rh = i < O_KROPE / 2 ? -z[i + O_KROPE / 2] : z[i - O_KROPE / 2];
            kt[i] = z[i] * ct[i] + rh * st[i];
        }
        for (int j = O_KROPE; j < O_DIDX; j++) kt[j] = z[j];
        for (int h = 0; h < O_HIDX; h++) {
            double acc = 0.0;
            for (int c = 0; c < O_HID; c++) acc += widen_bf16(ww[(int64_t)h * O_HID + c]) * widen_bf16(xt[c]);
            w_out[(int64_t)t * O_HIDX + h] = acc / sqrt((double)O_HIDX);
        }
    }
}

/* ---- E4M3 (OCP FP8) ---- */
double oracle_e4m3_decode(uint8_t c) {
    int sgn = c >> 7, e = (c >> 3) & 15, m = c & 7;
    double v;
    if (e == 15 && m == 7) return NAN;
    if (e == 0) v = ldexp((double)m / 8.0, -6);
    else v = ldexp(1.0 + (double)m / 8.0, e - 7);
    return sgn ? -v : v;
}

/* Nearest E4M3 code, ties to the even code; finite values beyond 448
 * saturate to +-448.  (Reference by exhaustive search over the 126 finite
 * non-negative magnitudes, so no rounding arithmetic can slip.) */
uint8_t oracle_e4m3_encode(double x) {
    if (isnan(x)) return 0x7F;
    uint8_t sgn = x < 0 ? 0x80 : 0x00;
    double a = fabs(x);
    if (a >= 448.0) return (uint8_t)(sgn | 0x7E);
    int best = 0;
    double best_d = INFINITY;
    for (int c = 0; c < 0x7F; c++) {          /* codes 0x00 .. 0x7E: +0 .. 448 */
        double d = fabs(oracle_e4m3_decode((uint8_t)c) - a);
        if (d < best_d || (d == best_d && (c & 1) == 0)) {
            best = c;
            best_d = d;
        }
    }
    return (uint8_t)(sgn | best);
}

/* rows of n bf16 values -> n codes per row and one scale per row.  The
 * scale amax / 448 and each quotient v / scale are single-precision (IEEE
 * round to nearest) values: the code is an integer decided by floating
 * point, so it is decided in the precision the GPU path uses. */
void oracle_quantize_fp8(int64_t rows, int n, const uint16_t* v, uint8_t* codes, double* scale) {
#pragma omp parallel for schedule(dynamic, 64)
    for (int64_t r = 0; r < rows; r++) {
        float amax = 0.0f;
        for (int d = 0; d < n; d++) {
            float a = (float)fabs(widen_bf16(v[r * n + d]));
            if (a > amax) amax = a;
        }
        volatile float sc = amax > 0.0f ? amax / 448.0f : 1.0f;
        scale[r] = (double)sc;
        for (int d = 0; d < n; d++) {
            volatile float q = (float)widen_bf16(v[r * n + d]) / sc;
            codes[r * n + d] = oracle_e4m3_encode((double)q);
        }
    }
}

/* Scores of requested rows on FP8 queries / keys (row layouts as
 * oracle_indexer_scores; q8 [total_q, 32, 128], qs [total_q, 32],
 * k8 [B*stride, 128], ks [B*stride]). */
void oracle_indexer_scores_fp8(int B, const int32_t* q_off, const int32_t* ctx_len, int64_t stride,
                               const uint8_t* q8, const double* qs, const float* w, const uint8_t* k8,
                               const double* ks, int nrows, const int32_t* rows, double* out, int64_t ld) {
    double val[256];                 /* every code's value, from the definition above */
    for (int c = 0; c < 256; c++) val[c] = oracle_e4m3_decode((uint8_t)c);
#pragma omp parallel for schedule(dynamic, 1)
    for (int j = 0; j < nrows; j++) {
        int b;
        int64_t t;
        locate_row(B, q_off, ctx_len, rows[j], &b, &t);
        for (int64_t s = 0; s <= t; s++) {
            const uint8_t* kr = k8 + ((int64_t)b * stride + s) * O_DIDX;
            double ksc = ks[(int64_t)b * stride + s];
            double score = 0.0;
            for (int h = 0; h < O_HIDX; h++) {
                const uint8_t* qr = q8 + ((int64_t)rows[j] * O_HIDX + h) * O_DIDX;
                double dot = 0.0;
                for (int d = 0; d < O_DIDX; d++) dot += val[qr[d]] * val[kr[d]];
                double x = qs[(int64_t)rows[j] * O_HIDX + h] * ksc * dot;
                score += (double)w[(int64_t)rows[j] * O_HIDX + h] * (x > 0.0 ? x : 0.0);
            }
            out[(int64_t)j * ld + s] = score;
        }
    }
}

void oracle_e4m3_decode_array(int64_t n, const uint8_t* c, double* out) {
    for (int64_t i = 0; i < n; i++) out[i] = oracle_e4m3_decode(c[i]);
}

void oracle_e4m3_encode_array(int64_t n, const double* x, uint8_t* out) {
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; i++) out[i] = oracle_e4m3_encode(x[i]);
}
