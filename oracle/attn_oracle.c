/*
 * attn_oracle.c -- plain, slow, fp64 CPU oracle for exact scaled-dot-product
 * attention (prefill forward) and paged-KV decode attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or
 * call this file; only the tests, the smoke check and the benchmark's CPU
 * baseline leg use it.  It shares no code, header or constant with the CUDA
 * library.
 *
 * What it computes (the plain definition, written out):
 *   The pages describe FlashAttention as *exact* attention that reaches the
 *   same result as naive attention which materialises the full N x N score
 *   matrix (NanoInfer README, "Flash Attention v1" bullet and the naive vs
 *   flash paragraph; inference-kernel-cookbook README, recipe 01 "Same
 *   result").  The online-softmax recurrence is stated there to be identical
 *   to the safe three-pass softmax (NanoInfer README, online softmax
 *   paragraph).  So this oracle is the three-pass form:
 *
 *     for every batch b, head h, query row i:
 *       J   = { j < Nkv : j < kv_len[b]  and  (not causal or j <= i + Nkv - Nq) }
 *       s_j = scale * sum_k q[i,k] * k[j,k]                 (pass 1, with m = max s_j)
 *       l   = sum_{j in J} exp(s_j - m)                     (pass 2)
 *       O_i = sum_{j in J} exp(s_j - m) * v[j,:] / l        (pass 3)
 *       LSE_i = m + ln(l)         (natural log of the sum of exp of the scaled scores)
 *
 *   The log-sum-exp per row is the statistic the FlashAttention-2 forward
 *   saves for the backward (gpu-inference blog, section 02).  The causal mask
 *   is combined with the key-padding mask before the softmax (same section).
 *   Causal alignment when Nq != Nkv is bottom-right (query i sees keys up to
 *   i + Nkv - Nq); the pages are silent on it and it is the reading that
 *   matches decoding after a prefill.  A row with no valid key yields O = 0
 *   and LSE = -inf (pages silent; chosen so the value is well defined).
 *
 *   Paged decode: one query per sequence attends over all ctx_len[b] cached
 *   tokens, which live in fixed-size pages found through a page table, and
 *   must give exactly the result of a contiguous cache (inference-kernel-
 *   cookbook README, recipe 03 "Paged Attention").  The oracle gathers the
 *   pages into a contiguous [ctx_len, d] buffer and applies the definition
 *   above with Nq = 1, Nkv = ctx_len, non-causal.
 *
 * Inputs are bf16 bit patterns (uint16); each is widened exactly to fp64
 * (bf16 -> fp32 by a 16-bit shift, fp32 -> fp64 exactly), so the oracle sees
 * the very values the GPU reads.  All arithmetic is in fp64.
 *
 * Layouts (row-major, contiguous):
 *   q [B,H,Nq,d], k/v [B,H,Nkv,d], o [B,H,Nq,d] (fp64), lse [B,H,Nq] (fp64)
 *   paged: q [B,H,d]; k_pages/v_pages [num_pages,H,page_size,d];
 *          page_table [B,max_pages] int32; ctx_lens [B] int32
 *
 * The backward (gradients of the same definition) is at the end of the file.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

static double bf16_to_f64(uint16_t bits) {
    uint32_t u = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* One query row against a contiguous K/V block of n_keys rows.
 * valid[j] != 0 marks the keys in J.  srow is caller scratch of n_keys doubles. */
static void attend_row(const uint16_t *qrow, const uint16_t *kb, const uint16_t *vb,
                       const unsigned char *valid, int n_keys, int d, double scale,
                       double *srow, double *out, double *lse_out) {
    /* pass 1: scores and their maximum over the valid keys */
    double m = -INFINITY;
    int any = 0;
    for (int j = 0; j < n_keys; ++j) {
        if (!valid[j]) continue;
        double dot = 0.0;
        for (int c = 0; c < d; ++c)
            dot += bf16_to_f64(qrow[c]) * bf16_to_f64(kb[(size_t)j * d + c]);
        srow[j] = scale * dot;
        if (!any || srow[j] > m) m = srow[j];
        any = 1;
    }
    if (!any) {
        for (int c = 0; c < d; ++c) out[c] = 0.0;
        *lse_out = -INFINITY;
        return;
    }
    /* pass 2: normaliser */
    double l = 0.0;
    for (int j = 0; j < n_keys; ++j)
        if (valid[j]) l += exp(srow[j] - m);
    /* pass 3: probabilities times V */
    for (int c = 0; c < d; ++c) out[c] = 0.0;
    for (int j = 0; j < n_keys; ++j) {
        if (!valid[j]) continue;
        double p = exp(srow[j] - m) / l;
        for (int c = 0; c < d; ++c) out[c] += p * bf16_to_f64(vb[(size_t)j * d + c]);
    }
    *lse_out = m + log(l);
}

static int key_valid(int i, int j, int Nq, int Nkv, int kv_len, int causal) {
    if (j >= Nkv || j >= kv_len) return 0;
    if (causal && (long)j > (long)i + (long)Nkv - (long)Nq) return 0;
    return 1;
}

/* Grouped-query form (grouped-query / multi-query attention, the variants compared in the
 * llm-kernel-lib README's attention ablation): Hq query heads share Hkv key/value heads,
 * query head h reading key/value head h / (Hq / Hkv).  q [B,Hq,Nq,d], k/v [B,Hkv,Nkv,d].
 * Rows are selected by flat index r = (b*Hq + h)*Nq + i.  o_rows [nrows,d], lse_rows [nrows].
 * Hkv == Hq is ordinary multi-head attention. */
int oracle_attn_gqa_rows_f64(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                             const int32_t *kv_lens, int B, int Hq, int Hkv, int Nq, int Nkv, int d,
                             int causal, double scale, const int64_t *rows, int64_t nrows,
                             double *o_rows, double *lse_rows, int nthreads) {
    if (B <= 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || Nq <= 0 || Nkv <= 0 || d <= 0 || nrows < 0)
        return 1;
    const int group = Hq / Hkv;
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
    int err = 0;
#pragma omp parallel
    {
        double *srow = (double *)malloc(sizeof(double) * (size_t)Nkv);
        unsigned char *valid = (unsigned char *)malloc((size_t)Nkv);
        if (!srow || !valid) {
#pragma omp atomic write
            err = 2;
        } else {
#pragma omp for schedule(dynamic, 4)
            for (int64_t t = 0; t < nrows; ++t) {
                int64_t r = rows[t];
                if (r < 0 || r >= (int64_t)B * Hq * Nq) {
#pragma omp atomic write
                    err = 1;
                    continue;
                }
                int i = (int)(r % Nq);
                int64_t bh = r / Nq;
                int b = (int)(bh / Hq), h = (int)(bh % Hq);
                int64_t bhkv = (int64_t)b * Hkv + h / group;
                int kv_len = kv_lens ? kv_lens[b] : Nkv;
                for (int j = 0; j < Nkv; ++j) valid[j] = (unsigned char)key_valid(i, j, Nq, Nkv, kv_len, causal);
                attend_row(q + (size_t)r * d, k + (size_t)bhkv * Nkv * d, v + (size_t)bhkv * Nkv * d,
                           valid, Nkv, d, scale, srow, o_rows + (size_t)t * d, lse_rows + t);
            }
        }
        free(srow);
        free(valid);
    }
    return err;
}

/* Rows selected by flat index r = (b*H + h)*Nq + i (multi-head: Hkv = H). */
int oracle_attn_rows_f64(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                         const int32_t *kv_lens, int B, int H, int Nq, int Nkv, int d,
                         int causal, double scale, const int64_t *rows, int64_t nrows,
                         double *o_rows, double *lse_rows, int nthreads) {
    return oracle_attn_gqa_rows_f64(q, k, v, kv_lens, B, H, H, Nq, Nkv, d, causal, scale, rows, nrows,
                                    o_rows, lse_rows, nthreads);
}

/* Every row: o [B,H,Nq,d], lse [B,H,Nq]. */
int oracle_attn_fwd_f64(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                        const int32_t *kv_lens, int B, int H, int Nq, int Nkv, int d, int causal,
                        double scale, double *o, double *lse, int nthreads) {
    if (B <= 0 || H <= 0 || Nq <= 0 || Nkv <= 0 || d <= 0) return 1;
    int64_t n = (int64_t)B * H * Nq;
    int64_t *rows = (int64_t *)malloc(sizeof(int64_t) * (size_t)n);
    if (!rows) return 2;
    for (int64_t r = 0; r < n; ++r) rows[r] = r;
    int err = oracle_attn_rows_f64(q, k, v, kv_lens, B, H, Nq, Nkv, d, causal, scale, rows, n,
                                   o, lse, nthreads);
    free(rows);
    return err;
}

/* Page ids outside [0, num_pages).  The pages describe the page table as an operating
 * system's page table over the KV cache (inference-kernel-cookbook README, recipe 03) and are
 * silent on an entry that maps no page.  With skip_bad_pages = 0 such an entry is an error
 * (return 1).  With skip_bad_pages = 1 it is read as an unmapped page that holds no tokens: the
 * positions it covers are left out of J (their keys get no weight and their values add
 * nothing), the other positions keep their places, so causal masks are unchanged. */

/* Paged decode, grouped-query form: q [B,Hq,d]; k_pages/v_pages [num_pages,Hkv,page_size,d];
 * query head h reads key/value head h / (Hq / Hkv).  o [B,Hq,d], lse [B,Hq]. */
int oracle_paged_decode_gqa_f64(const uint16_t *q, const uint16_t *k_pages, const uint16_t *v_pages,
                                const int32_t *page_table, const int32_t *ctx_lens, int page_size,
                                int B, int Hq, int Hkv, int d, int max_pages, int num_pages, double scale,
                                double *o, double *lse, int nthreads, int skip_bad_pages) {
    if (B <= 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || d <= 0 || page_size <= 0 || max_pages <= 0 ||
        num_pages <= 0)
        return 1;
    const int H = Hq, group = Hq / Hkv;
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
    int err = 0;
    int cap = max_pages * page_size;
#pragma omp parallel
    {
        uint16_t *kc = (uint16_t *)malloc(sizeof(uint16_t) * (size_t)cap * d);
        uint16_t *vc = (uint16_t *)malloc(sizeof(uint16_t) * (size_t)cap * d);
        double *srow = (double *)malloc(sizeof(double) * (size_t)cap);
        unsigned char *valid = (unsigned char *)malloc((size_t)cap);
        if (!kc || !vc || !srow || !valid) {
#pragma omp atomic write
            err = 2;
        } else {
#pragma omp for schedule(dynamic, 1)
            for (int64_t bh = 0; bh < (int64_t)B * H; ++bh) {
                int b = (int)(bh / H), h = (int)(bh % H);
                int n = ctx_lens[b];
                if (n < 0 || n > cap) {
#pragma omp atomic write
                    err = 1;
                    continue;
                }
                /* gather: logical token t lives in page page_table[b][t / page_size],
                 * slot t % page_size, of head h */
                int bad = 0;
                for (int t = 0; t < n; ++t) {
                    int32_t pg = page_table[(size_t)b * max_pages + t / page_size];
                    valid[t] = 1;
                    if (pg < 0 || pg >= num_pages) {
                        if (!skip_bad_pages) { bad = 1; break; }
                        valid[t] = 0;  /* an unmapped page: no token here */
                        memset(kc + (size_t)t * d, 0, sizeof(uint16_t) * (size_t)d);
                        memset(vc + (size_t)t * d, 0, sizeof(uint16_t) * (size_t)d);
                        continue;
                    }
                    size_t src = (((size_t)pg * Hkv + h / group) * page_size + (size_t)(t % page_size)) * d;
                    memcpy(kc + (size_t)t * d, k_pages + src, sizeof(uint16_t) * (size_t)d);
                    memcpy(vc + (size_t)t * d, v_pages + src, sizeof(uint16_t) * (size_t)d);
                }
                if (bad) {
#pragma omp atomic write
                    err = 1;
                    continue;
                }
                attend_row(q + (size_t)bh * d, kc, vc, valid, n, d, scale, srow,
                           o + (size_t)bh * d, lse + bh);
            }
        }
        free(kc);
        free(vc);
        free(srow);
        free(valid);
    }
    return err;
}

/* Chunked prefill over the paged cache (prefill into a KV cache, inference-kernel-cookbook
 * README recipes 02-03; KV-cache append path of the Kernel-Inference-Engine README's
 * roadmap): sequence b has ctx_lens[b] cached tokens in its pages, the last Nq of which are
 * the new queries q[b, :, i] at positions ctx_lens[b] - Nq + i.  Query i sees keys
 * j < ctx_lens[b] and, if causal, j <= i + ctx_lens[b] - Nq (bottom-right).  Pages are
 * gathered into a contiguous cache and the plain definition applied per row.
 * q [B,Hq,Nq,d]; k_pages/v_pages [num_pages,Hkv,page_size,d]; o [B,Hq,Nq,d]; lse [B,Hq,Nq]. */
int oracle_paged_prefill_gqa_f64(const uint16_t *q, const uint16_t *k_pages, const uint16_t *v_pages,
                                 const int32_t *page_table, const int32_t *ctx_lens, int page_size, int B,
                                 int Hq, int Hkv, int Nq, int d, int max_pages, int num_pages, int causal,
                                 double scale, double *o, double *lse, int nthreads, int skip_bad_pages) {
    if (B <= 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || Nq <= 0 || d <= 0 || page_size <= 0 ||
        max_pages <= 0 || num_pages <= 0)
        return 1;
    const int group = Hq / Hkv;
    const int cap = max_pages * page_size;
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
    int err = 0;
#pragma omp parallel
    {
        uint16_t *kc = (uint16_t *)malloc(sizeof(uint16_t) * (size_t)cap * d);
        uint16_t *vc = (uint16_t *)malloc(sizeof(uint16_t) * (size_t)cap * d);
        double *srow = (double *)malloc(sizeof(double) * (size_t)cap);
        unsigned char *valid = (unsigned char *)malloc((size_t)cap);
        unsigned char *mapped = (unsigned char *)malloc((size_t)cap);
        if (!kc || !vc || !srow || !valid || !mapped) {
#pragma omp atomic write
            err = 2;
        } else {
#pragma omp for schedule(dynamic, 1)
            for (int64_t bh = 0; bh < (int64_t)B * Hq; ++bh) {
                int b = (int)(bh / Hq), h = (int)(bh % Hq);
                int n = ctx_lens[b];
                if (n < 0 || n > cap) {
#pragma omp atomic write
                    err = 1;
                    continue;
                }
                int bad = 0;
                for (int t = 0; t < n; ++t) {
                    int32_t pg = page_table[(size_t)b * max_pages + t / page_size];
                    mapped[t] = 1;
                    if (pg < 0 || pg >= num_pages) {
                        if (!skip_bad_pages) { bad = 1; break; }
                        mapped[t] = 0;  /* an unmapped page: no token here */
                        memset(kc + (size_t)t * d, 0, sizeof(uint16_t) * (size_t)d);
                        memset(vc + (size_t)t * d, 0, sizeof(uint16_t) * (size_t)d);
                        continue;
                    }
                    size_t src = (((size_t)pg * Hkv + h / group) * page_size + (size_t)(t % page_size)) * d;
                    memcpy(kc + (size_t)t * d, k_pages + src, sizeof(uint16_t) * (size_t)d);
                    memcpy(vc + (size_t)t * d, v_pages + src, sizeof(uint16_t) * (size_t)d);
                }
                if (bad) {
#pragma omp atomic write
                    err = 1;
                    continue;
                }
                for (int i = 0; i < Nq; ++i) {
                    for (int j = 0; j < n; ++j)
                        valid[j] = (unsigned char)(mapped[j] && key_valid(i, j, Nq, n, n, causal));
                    size_t r = (size_t)bh * Nq + i;
                    attend_row(q + r * d, kc, vc, valid, n, d, scale, srow, o + r * d, lse + r);
                }
            }
        }
        free(kc);
        free(vc);
        free(srow);
        free(valid);
        free(mapped);
    }
    return err;
}

/* Paged decode, multi-head (Hkv = H): o [B,H,d], lse [B,H]. */
int oracle_paged_decode_f64(const uint16_t *q, const uint16_t *k_pages, const uint16_t *v_pages,
                            const int32_t *page_table, const int32_t *ctx_lens, int page_size,
                            int B, int H, int d, int max_pages, int num_pages, double scale,
                            double *o, double *lse, int nthreads) {
    return oracle_paged_decode_gqa_f64(q, k_pages, v_pages, page_table, ctx_lens, page_size, B, H, H, d,
                                       max_pages, num_pages, scale, o, lse, nthreads, 0);
}

/* ------------------------------------------------------------------------------------------
 * Backward pass.  The gpu-inference blog, section 02 ("FlashAttention-2 in Triton"), trains with
 * a backward that recomputes the probabilities from the forward's saved log-sum-exp and splits
 * the work into a row-wise D preprocessing pass, a dK/dV pass and a dQ pass.  What that backward
 * reaches is the exact gradient of the definition above for an upstream gradient dO of O, which
 * this oracle writes out directly (no tiling, no saved statistics; everything recomputed):
 *
 *   P_ij  = exp(s_ij - m_i) / l_i  for j in J_i, 0 otherwise        (the forward's softmax row)
 *   dV_j  = sum_i P_ij dO_i                                          (O = P V)
 *   dP_ij = dO_i . v_j
 *   D_i   = sum_j P_ij dP_ij                                         (= dO_i . O_i)
 *   dS_ij = P_ij (dP_ij - D_i)                                       (softmax Jacobian)
 *   dQ_i  = scale sum_j dS_ij k_j,     dK_j = scale sum_i dS_ij q_i  (s = scale q . k)
 *
 * Grouped-query form: key/value head g is read by query heads g*group .. g*group+group-1, so its
 * dK and dV sum over those heads.  A row with no valid key has P = 0: it adds nothing and its dQ
 * is 0.  Inputs are fp64 here (the Python wrapper widens bf16 exactly) so that the same function
 * also serves finite-difference checks with perturbations bf16 cannot hold.  Optional outputs o,
 * lse (the forward of these fp64 inputs) and Drow may be NULL.
 * q, dout, dq [B,Hq,Nq,d]; k, v, dk, dv [B,Hkv,Nkv,d]; o [B,Hq,Nq,d]; lse, Drow [B,Hq,Nq].
 */
int oracle_attn_bwd_gqa_f64(const double *q, const double *k, const double *v, const double *dout,
                            const int32_t *kv_lens, int B, int Hq, int Hkv, int Nq, int Nkv, int d,
                            int causal, double scale, double *dq, double *dk, double *dv,
                            double *o, double *lse, double *Drow, int nthreads) {
    if (B <= 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || Nq <= 0 || Nkv <= 0 || d <= 0) return 1;
    const int group = Hq / Hkv;
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
    int err = 0;
#pragma omp parallel
    {
        double *P = (double *)malloc(sizeof(double) * (size_t)Nkv);
        double *dP = (double *)malloc(sizeof(double) * (size_t)Nkv);
        unsigned char *valid = (unsigned char *)malloc((size_t)Nkv);
        if (!P || !dP || !valid) {
#pragma omp atomic write
            err = 2;
        } else {
            /* one (batch, key/value head) per iteration: it owns dK/dV of that head */
#pragma omp for schedule(dynamic, 1)
            for (int64_t bg = 0; bg < (int64_t)B * Hkv; ++bg) {
                const int b = (int)(bg / Hkv), g = (int)(bg % Hkv);
                const double *kb = k + (size_t)bg * Nkv * d;
                const double *vb = v + (size_t)bg * Nkv * d;
                double *dkb = dk + (size_t)bg * Nkv * d;
                double *dvb = dv + (size_t)bg * Nkv * d;
                for (size_t x = 0; x < (size_t)Nkv * d; ++x) dkb[x] = dvb[x] = 0.0;
                const int kv_len = kv_lens ? kv_lens[b] : Nkv;
                for (int hh = 0; hh < group; ++hh) {
                    const int h = g * group + hh;
                    for (int i = 0; i < Nq; ++i) {
                        const size_t r = ((size_t)b * Hq + h) * Nq + i;
                        const double *qi = q + r * d, *doi = dout + r * d;
                        double *dqi = dq + r * d;
                        for (int c = 0; c < d; ++c) dqi[c] = 0.0;
                        /* the forward's softmax row, three passes */
                        double m = -INFINITY;
                        int any = 0;
                        for (int j = 0; j < Nkv; ++j) {
                            valid[j] = (unsigned char)key_valid(i, j, Nq, Nkv, kv_len, causal);
                            if (!valid[j]) continue;
                            double dot = 0.0;
                            for (int c = 0; c < d; ++c) dot += qi[c] * kb[(size_t)j * d + c];
                            P[j] = scale * dot;
                            if (!any || P[j] > m) m = P[j];
                            any = 1;
                        }
                        if (!any) {
                            if (o) for (int c = 0; c < d; ++c) o[r * d + c] = 0.0;
                            if (lse) lse[r] = -INFINITY;
                            if (Drow) Drow[r] = 0.0;
                            continue;
                        }
                        double l = 0.0;
                        for (int j = 0; j < Nkv; ++j)
                            if (valid[j]) l += exp(P[j] - m);
                        for (int j = 0; j < Nkv; ++j) P[j] = valid[j] ? exp(P[j] - m) / l : 0.0;
                        if (o) {
                            for (int c = 0; c < d; ++c) o[r * d + c] = 0.0;
                            for (int j = 0; j < Nkv; ++j)
                                if (valid[j])
                                    for (int c = 0; c < d; ++c) o[r * d + c] += P[j] * vb[(size_t)j * d + c];
                        }
                        if (lse) lse[r] = m + log(l);
                        /* dP and the row term D */
                        double Di = 0.0;
                        for (int j = 0; j < Nkv; ++j) {
                            if (!valid[j]) continue;
                            double dot = 0.0;
                            for (int c = 0; c < d; ++c) dot += doi[c] * vb[(size_t)j * d + c];
                            dP[j] = dot;
                            Di += P[j] * dot;
                        }
                        if (Drow) Drow[r] = Di;
                        /* dS, then the three products */
                        for (int j = 0; j < Nkv; ++j) {
                            if (!valid[j]) continue;
                            const double dS = P[j] * (dP[j] - Di);
                            for (int c = 0; c < d; ++c) {
                                dqi[c] += scale * dS * kb[(size_t)j * d + c];
                                dkb[(size_t)j * d + c] += scale * dS * qi[c];
                                dvb[(size_t)j * d + c] += P[j] * doi[c];
                            }
                        }
                    }
                }
            }
        }
        free(P);
        free(dP);
        free(valid);
    }
    return err;
}

/* The backward's preprocessing step as the method computes it: D_i = dO_i . O_i from the stored
 * (bf16) forward output.  o, dout [nrows, d] bf16 bit patterns; Drow [nrows]. */
int oracle_bwd_rowdot_f64(const uint16_t *o, const uint16_t *dout, int64_t nrows, int d, double *Drow) {
    if (nrows < 0 || d <= 0) return 1;
    for (int64_t r = 0; r < nrows; ++r) {
        double acc = 0.0;
        for (int c = 0; c < d; ++c)
            acc += bf16_to_f64(dout[(size_t)r * d + c]) * bf16_to_f64(o[(size_t)r * d + c]);
        Drow[r] = acc;
    }
    return 0;
}

/* ------------------------------------------------------------------------------------------
 * FP8 (E4M3) key/value cache.  The NanoInfer README's roadmap names FP8 e4m3 storage (Hopper and
 * later, cuda_fp8.h) as the successor of INT8 with the quantisation math unchanged; applied to the
 * attention path that is a KV cache stored as e4m3 codes with one scale per tensor:
 *   value(code) = e4m3(code) * scale,
 *   code(x)     = e4m3 rounding of fp32(x) * fp32(1/scale), to nearest with ties to even,
 *                 saturating at the largest finite magnitude (448).
 * E4M3 (the OCP FP8 "E4M3" format): 1 sign bit, 4 exponent bits with bias 7, 3 mantissa bits;
 * exponent field 0 holds the subnormals m * 2^-9; no infinities; S.1111.111 is NaN, so the
 * largest finite value is 1.75 * 2^8 = 448.
 */
double oracle_e4m3_value(uint8_t code) {
    const int sign = code >> 7, e = (code >> 3) & 15, m = code & 7;
    if (e == 15 && m == 7) return NAN;
    const double mag = e == 0 ? ldexp((double)m, -9) : ldexp(1.0 + m / 8.0, e - 7);
    return sign ? -mag : mag;
}

/* Nearest e4m3 code to y (ties to the even code, i.e. mantissa bit 0 clear), saturating:
 * magnitudes above 448 give 448.  The sign bit is y's (E4M3 has a signed zero: -0 -> 0x80).  A brute-force search over the 127 non-negative finite codes,
 * which saturates by construction (every candidate is finite). */
uint8_t oracle_e4m3_code(float y) {
    if (y != y) return 0x7F;
    const double a = fabs((double)y);
    int best = 0;
    double best_err = INFINITY;
    for (int c = 0; c <= 0x7E; ++c) {
        const double err = fabs(oracle_e4m3_value((uint8_t)c) - a);
        if (err < best_err || (err == best_err && (c & 1) == 0)) {
            best = c;
            best_err = err;
        }
    }
    return (uint8_t)((signbit(y) ? 0x80 : 0) | best);  /* the sign is kept, -0 included */
}

/* codes[i] = code(fp32(x[i]) * inv_scale): x bf16 bit patterns, the product rounded to fp32.
 * The code depends only on x[i]'s bit pattern, so it is worked out once per pattern (65536
 * calls of oracle_e4m3_code) and looked up. */
int oracle_e4m3_quantize(const uint16_t *x, int64_t n, float inv_scale, uint8_t *codes) {
    if (n < 0) return 1;
    uint8_t *table = (uint8_t *)malloc(65536);
    if (!table) return 2;
    for (int b = 0; b < 65536; ++b) {
        const float y = (float)bf16_to_f64((uint16_t)b) * inv_scale;
        table[b] = oracle_e4m3_code(y);
    }
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) codes[i] = table[x[i]];
    free(table);
    return 0;
}

/* One query row against n_keys fp64 keys/values with a validity mask (valid[j] != 0 marks the
 * keys in J): the three passes of attend_row, in the same order. */
static void attend_row_f64kv_masked(const uint16_t *qrow, const double *kb, const double *vb,
                                    const unsigned char *valid, int n_keys, int d, double scale, double *srow,
                                    double *out, double *lse_out) {
    double m = -INFINITY;
    int any = 0;
    for (int j = 0; j < n_keys; ++j) {
        if (!valid[j]) continue;
        double dot = 0.0;
        for (int c = 0; c < d; ++c) dot += bf16_to_f64(qrow[c]) * kb[(size_t)j * d + c];
        srow[j] = scale * dot;
        if (!any || srow[j] > m) m = srow[j];
        any = 1;
    }
    for (int c = 0; c < d; ++c) out[c] = 0.0;
    if (!any) {
        *lse_out = -INFINITY;
        return;
    }
    double l = 0.0;
    for (int j = 0; j < n_keys; ++j)
        if (valid[j]) l += exp(srow[j] - m);
    for (int j = 0; j < n_keys; ++j) {
        if (!valid[j]) continue;
        double p = exp(srow[j] - m) / l;
        for (int c = 0; c < d; ++c) out[c] += p * vb[(size_t)j * d + c];
    }
    *lse_out = m + log(l);
}

/* One query row against n_keys fp64 keys/values (all valid): the three passes of attend_row. */
static void attend_row_f64kv(const uint16_t *qrow, const double *kb, const double *vb, int n_keys, int d,
                             double scale, double *srow, double *out, double *lse_out) {
    double m = -INFINITY;
    for (int j = 0; j < n_keys; ++j) {
        double dot = 0.0;
        for (int c = 0; c < d; ++c) dot += bf16_to_f64(qrow[c]) * kb[(size_t)j * d + c];
        srow[j] = scale * dot;
        if (j == 0 || srow[j] > m) m = srow[j];
    }
    for (int c = 0; c < d; ++c) out[c] = 0.0;
    if (n_keys == 0) {
        *lse_out = -INFINITY;
        return;
    }
    double l = 0.0;
    for (int j = 0; j < n_keys; ++j) l += exp(srow[j] - m);
    for (int j = 0; j < n_keys; ++j) {
        const double p = exp(srow[j] - m) / l;
        for (int c = 0; c < d; ++c) out[c] += p * vb[(size_t)j * d + c];
    }
    *lse_out = m + log(l);
}

/* Paged decode over an e4m3 cache: as oracle_paged_decode_gqa_f64 with k_pages/v_pages holding
 * e4m3 codes [num_pages, Hkv, page_size, d]; each cached value is e4m3(code) * k_scale (keys) or
 * * v_scale (values), dequantised exactly in fp64 before the plain definition is applied. */
int oracle_paged_decode_fp8_gqa_f64(const uint16_t *q, const uint8_t *k_pages, const uint8_t *v_pages,
                                    double k_scale, double v_scale, const int32_t *page_table,
                                    const int32_t *ctx_lens, int page_size, int B, int Hq, int Hkv, int d,
                                    int max_pages, int num_pages, double scale, double *o, double *lse,
                                    int nthreads, int skip_bad_pages) {
    if (B <= 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || d <= 0 || page_size <= 0 || max_pages <= 0 ||
        num_pages <= 0)
        return 1;
    const int group = Hq / Hkv;
    const int cap = max_pages * page_size;
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
    int err = 0;
#pragma omp parallel
    {
        double *kc = (double *)malloc(sizeof(double) * (size_t)cap * d);
        double *vc = (double *)malloc(sizeof(double) * (size_t)cap * d);
        double *srow = (double *)malloc(sizeof(double) * (size_t)cap);
        if (!kc || !vc || !srow) {
#pragma omp atomic write
            err = 2;
        } else {
#pragma omp for schedule(dynamic, 1)
            for (int64_t bh = 0; bh < (int64_t)B * Hq; ++bh) {
                const int b = (int)(bh / Hq), h = (int)(bh % Hq);
                const int n = ctx_lens[b];
                if (n < 0 || n > cap) {
#pragma omp atomic write
                    err = 1;
                    continue;
                }
                /* the decode query has no position-dependent mask, so the tokens of mapped pages
                 * are gathered back to back (unmapped pages, when skipped, contribute none) */
                int bad = 0, kept = 0;
                for (int t = 0; t < n && !bad; ++t) {
                    const int32_t pg = page_table[(size_t)b * max_pages + t / page_size];
                    if (pg < 0 || pg >= num_pages) {
                        if (skip_bad_pages) continue;
                        bad = 1;
                        break;
                    }
                    const size_t src = (((size_t)pg * Hkv + h / group) * page_size + (size_t)(t % page_size)) * d;
                    for (int c = 0; c < d; ++c) {
                        kc[(size_t)kept * d + c] = oracle_e4m3_value(k_pages[src + c]) * k_scale;
                        vc[(size_t)kept * d + c] = oracle_e4m3_value(v_pages[src + c]) * v_scale;
                    }
                    ++kept;
                }
                if (bad) {
#pragma omp atomic write
                    err = 1;
                    continue;
                }
                attend_row_f64kv(q + (size_t)bh * d, kc, vc, kept, d, scale, srow, o + (size_t)bh * d, lse + bh);
            }
        }
        free(kc);
        free(vc);
        free(srow);
    }
    return err;
}

/* Chunked prefill over an e4m3 cache: oracle_paged_prefill_gqa_f64 with k_pages/v_pages holding
 * e4m3 codes [num_pages, Hkv, page_size, d]; each cached value is e4m3(code) * k_scale (keys) or
 * * v_scale (values), dequantised exactly in fp64, after which the plain definition is applied
 * per query row exactly as in the bf16 form (same masks, same order of operations).  Page ids
 * outside [0, num_pages) follow skip_bad_pages as in the bf16 form. */
int oracle_paged_prefill_fp8_gqa_f64(const uint16_t *q, const uint8_t *k_pages, const uint8_t *v_pages,
                                     double k_scale, double v_scale, const int32_t *page_table,
                                     const int32_t *ctx_lens, int page_size, int B, int Hq, int Hkv, int Nq,
                                     int d, int max_pages, int num_pages, int causal, double scale, double *o,
                                     double *lse, int nthreads, int skip_bad_pages) {
    if (B <= 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || Nq <= 0 || d <= 0 || page_size <= 0 ||
        max_pages <= 0 || num_pages <= 0)
        return 1;
    const int group = Hq / Hkv;
    const int cap = max_pages * page_size;
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
    int err = 0;
#pragma omp parallel
    {
        double *kc = (double *)malloc(sizeof(double) * (size_t)cap * d);
        double *vc = (double *)malloc(sizeof(double) * (size_t)cap * d);
        double *srow = (double *)malloc(sizeof(double) * (size_t)cap);
        unsigned char *valid = (unsigned char *)malloc((size_t)cap);
        unsigned char *mapped = (unsigned char *)malloc((size_t)cap);
        if (!kc || !vc || !srow || !valid || !mapped) {
#pragma omp atomic write
            err = 2;
        } else {
#pragma omp for schedule(dynamic, 1)
            for (int64_t bh = 0; bh < (int64_t)B * Hq; ++bh) {
                const int b = (int)(bh / Hq), h = (int)(bh % Hq);
                const int n = ctx_lens[b];
                if (n < 0 || n > cap) {
#pragma omp atomic write
                    err = 1;
                    continue;
                }
                int bad = 0;
                for (int t = 0; t < n; ++t) {
                    const int32_t pg = page_table[(size_t)b * max_pages + t / page_size];
                    mapped[t] = 1;
                    if (pg < 0 || pg >= num_pages) {
                        if (!skip_bad_pages) { bad = 1; break; }
                        mapped[t] = 0;  /* an unmapped page: no token here */
                        for (int c = 0; c < d; ++c) kc[(size_t)t * d + c] = vc[(size_t)t * d + c] = 0.0;
                        continue;
                    }
                    const size_t src = (((size_t)pg * Hkv + h / group) * page_size + (size_t)(t % page_size)) * d;
                    for (int c = 0; c < d; ++c) {
                        kc[(size_t)t * d + c] = oracle_e4m3_value(k_pages[src + c]) * k_scale;
                        vc[(size_t)t * d + c] = oracle_e4m3_value(v_pages[src + c]) * v_scale;
                    }
                }
                if (bad) {
#pragma omp atomic write
                    err = 1;
                    continue;
                }
                for (int i = 0; i < Nq; ++i) {
                    for (int j = 0; j < n; ++j)
                        valid[j] = (unsigned char)(mapped[j] && key_valid(i, j, Nq, n, n, causal));
                    const size_t r = (size_t)bh * Nq + i;
                    attend_row_f64kv_masked(q + r * d, kc, vc, valid, n, d, scale, srow, o + r * d, lse + r);
                }
            }
        }
        free(kc);
        free(vc);
        free(srow);
        free(valid);
        free(mapped);
    }
    return err;
}

/* Number of threads OpenMP would use (for reporting the CPU baseline's cores). */
int oracle_num_threads(int nthreads) {
#ifdef _OPENMP
    if (nthreads > 0) return nthreads;
    return omp_get_max_threads();
#else
    (void)nthreads;
    return 1;
#endif
}
