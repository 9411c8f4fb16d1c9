/*
 * CPU oracle for the attention hot path -- TEST INFRASTRUCTURE ONLY.
 *
 * Only tests/, the smoke check and the benchmark's CPU-baseline leg may load
 * this library.  The product path never calls it; it shares no code, header or
 * helper with the CUDA library.
 *
 * Everything here is the plain definition of what the method computes, written
 * as slow loops, following the article "SLM 生成式高并发推理引擎：延迟约束下的有效吞吐优化":
 *
 *   - section 3.1 (packed prefill): Q [sum L_i, N_q, D], K/V [sum L_i, N_kv, D];
 *     the sequence boundary implies a block-diagonal causal mask; a query sees
 *     only positions of its own sequence that are not later than itself.
 *   - section 3.2 (shared prefix): O_b = Attention(Q_b, [prefix_K; suffix_K[b]],
 *     [prefix_V; suffix_V[b]]); the suffix K/V is reordered by parent index.
 *     The oracle builds the concatenation that the method avoids.
 *   - section 3.3 (two-stage candidate selection): FP32 log-softmax over the full
 *     vocabulary, scores = cumulative beam score + log-probability, global
 *     candidates from the flattened beams.  The oracle sorts ALL W x V
 *     entries instead of taking the 2W-per-beam shortcut.
 *
 * Inputs are bf16 bit patterns (uint16) widened exactly; attention arithmetic is
 * fp64.  Selection arithmetic is fp32 where the article fixes FP32 (the
 * log-softmax and the scores); the log-normaliser is computed in fp64 and
 * rounded once to fp32.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------------- */
/* bf16 widening: a bf16 value is the upper 16 bits of an IEEE binary32.      */
/* ------------------------------------------------------------------------- */
static float bf16_bits_to_f32(uint16_t b) {
    uint32_t u = ((uint32_t)b) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

static double bf16_bits_to_f64(uint16_t b) { return (double)bf16_bits_to_f32(b); }

int oracle_abi_version(void) { return 1; }

/* ------------------------------------------------------------------------- */
/* Single-query attention over an explicit key/value list (fp64).            */
/*   keys[j], vals[j] point to D contiguous bf16 values, j = 0..n-1.          */
/*   out[D] = sum_j softmax_j(scale * q.k_j) * v_j ;  *lse = log sum exp.     */
/* ------------------------------------------------------------------------- */
static void attend_list(const uint16_t *qrow, const uint16_t *const *keys,
                        const uint16_t *const *vals, int64_t n, int D,
                        double scale, double *score_buf, double *out, double *lse) {
    double m = -INFINITY;
    for (int64_t j = 0; j < n; ++j) {
        double dot = 0.0;
        for (int d = 0; d < D; ++d)
            dot += bf16_bits_to_f64(qrow[d]) * bf16_bits_to_f64(keys[j][d]);
        double s = scale * dot;
        score_buf[j] = s;
        if (s > m) m = s;
    }
    double l = 0.0;
    for (int64_t j = 0; j < n; ++j) {
        double p = exp(score_buf[j] - m);
        score_buf[j] = p;
        l += p;
    }
    for (int d = 0; d < D; ++d) {
        double acc = 0.0;
        for (int64_t j = 0; j < n; ++j) acc += score_buf[j] * bf16_bits_to_f64(vals[j][d]);
        out[d] = acc / l;
    }
    if (lse) *lse = m + log(l);
}

/* ------------------------------------------------------------------------- */
/* Packed varlen causal GQA prefill (section 3.1).                            */
/*                                                                           */
/*   q [T, Hq, D], k/v [T, Hkv, D] bf16 bits; cu_seqlens int32 [B+1].          */
/*   Query head h reads KV head h / (Hq/Hkv) (contiguous head groups).        */
/*   o [T, Hq, D] fp64; lse [Hq, T] fp64 (nullable).                           */
/*   Returns 0, or -1 on malformed arguments.                                 */
/* ------------------------------------------------------------------------- */
static int64_t seq_of_token(const int32_t *cu, int B, int64_t t) {
    for (int b = 0; b < B; ++b)
        if (t >= cu[b] && t < cu[b + 1]) return b;
    return -1;
}

static int prefill_row(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                       const int32_t *cu, int B, int Hq, int Hkv, int D, double scale,
                       int64_t t, int h, double *out, double *lse) {
    int G = Hq / Hkv;
    int kvh = h / G;
    int64_t b = seq_of_token(cu, B, t);
    if (b < 0) return -1;
    int64_t s0 = cu[b];
    int64_t n = t - s0 + 1; /* keys s0..t: same sequence, not later than t */
    const uint16_t **keys = (const uint16_t **)malloc(sizeof(void *) * (size_t)n);
    const uint16_t **vals = (const uint16_t **)malloc(sizeof(void *) * (size_t)n);
    double *buf = (double *)malloc(sizeof(double) * (size_t)n);
    if (!keys || !vals || !buf) { free(keys); free(vals); free(buf); return -1; }
    for (int64_t j = 0; j < n; ++j) {
        keys[j] = k + ((s0 + j) * Hkv + kvh) * (int64_t)D;
        vals[j] = v + ((s0 + j) * Hkv + kvh) * (int64_t)D;
    }
    attend_list(q + (t * Hq + h) * (int64_t)D, keys, vals, n, D, scale, buf, out, lse);
    free(keys); free(vals); free(buf);
    return 0;
}

static int check_boundary(const int32_t *cu, int B) {
    if (B < 0 || cu[0] != 0) return -1;
    for (int b = 0; b < B; ++b)
        if (cu[b + 1] < cu[b]) return -1;
    return 0;
}

int oracle_packed_prefill(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                          const int32_t *cu_seqlens, int B, int Hq, int Hkv, int D,
                          double scale, double *o, double *lse, int n_threads) {
    if (Hkv <= 0 || Hq % Hkv != 0 || D <= 0) return -1;
    if (check_boundary(cu_seqlens, B)) return -1;
    int64_t T = cu_seqlens[B];
    int64_t n_rows = T * Hq;
    int bad = 0;
    (void)n_threads;
#pragma omp parallel for schedule(dynamic, 16) num_threads(n_threads > 0 ? n_threads : 1) reduction(| : bad)
    for (int64_t r = 0; r < n_rows; ++r) {
        int64_t t = r / Hq;
        int h = (int)(r % Hq);
        double l;
        if (prefill_row(q, k, v, cu_seqlens, B, Hq, Hkv, D, scale, t, h,
                        o + (t * Hq + h) * (int64_t)D, &l)) bad = 1;
        if (lse) lse[(int64_t)h * T + t] = l;
    }
    return bad ? -1 : 0;
}

/* Selected rows only: rows[2*i] = token, rows[2*i+1] = q head.
 * o_rows [n, D], lse_rows [n] (nullable).  For sizes where a full pass is slow. */
int oracle_packed_prefill_rows(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                               const int32_t *cu_seqlens, int B, int Hq, int Hkv, int D,
                               double scale, const int64_t *rows, int64_t n_sel,
                               double *o_rows, double *lse_rows, int n_threads) {
    if (Hkv <= 0 || Hq % Hkv != 0 || D <= 0) return -1;
    if (check_boundary(cu_seqlens, B)) return -1;
    int bad = 0;
    (void)n_threads;
#pragma omp parallel for schedule(dynamic, 4) num_threads(n_threads > 0 ? n_threads : 1) reduction(| : bad)
    for (int64_t i = 0; i < n_sel; ++i) {
        double l;
        if (prefill_row(q, k, v, cu_seqlens, B, Hq, Hkv, D, scale, rows[2 * i],
                        (int)rows[2 * i + 1], o_rows + i * D, &l)) bad = 1;
        if (lse_rows) lse_rows[i] = l;
    }
    return bad ? -1 : 0;
}

/* ------------------------------------------------------------------------- */
/* Shared-prefix beam decode (section 3.2).                                   */
/*                                                                           */
/*   q [W, Hq, D]; kp/vp [Lp, Hkv, D]; ks/vs [W, Smax, Hkv, D] with rows       */
/*   s < L_prev valid in the previous beam order; k_new/v_new [W, Hkv, D] in  */
/*   the new beam order (nullable together: then nothing is appended);        */
/*   parent [W] (nullable: identity).                                         */
/*                                                                           */
/*   Suffix reorder: ks_out[b, s] = ks[parent[b], s] for s < L_prev and       */
/*   ks_out[b, L_prev] = k_new[b] (same for V); rows beyond L_s are copied    */
/*   as zero.  Attention of beam b, head h reads the explicit concatenation   */
/*   [kp[:, kvh]; ks_out[b, :L_s, kvh]] with L_s = L_prev (+1 if appended).   */
/*   o [W, Hq, D] fp64; lse [W, Hq] fp64 (nullable).                           */
/* ------------------------------------------------------------------------- */
int oracle_shared_prefix_decode(const uint16_t *q, const uint16_t *kp, const uint16_t *vp,
                                const uint16_t *ks, const uint16_t *vs,
                                const uint16_t *k_new, const uint16_t *v_new,
                                const int32_t *parent, int W, int Lp, int L_prev, int Smax,
                                int Hq, int Hkv, int D, double scale,
                                uint16_t *ks_out, uint16_t *vs_out, double *o, double *lse,
                                int n_threads) {
    if (Hkv <= 0 || Hq % Hkv != 0 || D <= 0 || W < 0 || Lp < 0 || L_prev < 0) return -1;
    int append = (k_new != NULL && v_new != NULL);
    int Ls = L_prev + (append ? 1 : 0);
    if (Ls > Smax) return -1;
    if (Lp + Ls <= 0) return -1;
    for (int b = 0; b < W; ++b)
        if (parent && (parent[b] < 0 || parent[b] >= W)) return -1;

    /* 1. reorder + append into the output suffix buffers */
    int64_t row = (int64_t)Hkv * D;
    for (int b = 0; b < W; ++b) {
        int src = parent ? parent[b] : b;
        for (int s = 0; s < Smax; ++s) {
            uint16_t *dk = ks_out + ((int64_t)b * Smax + s) * row;
            uint16_t *dv = vs_out + ((int64_t)b * Smax + s) * row;
            if (s < L_prev) {
                memcpy(dk, ks + ((int64_t)src * Smax + s) * row, sizeof(uint16_t) * (size_t)row);
                memcpy(dv, vs + ((int64_t)src * Smax + s) * row, sizeof(uint16_t) * (size_t)row);
            } else if (s == L_prev && append) {
                memcpy(dk, k_new + (int64_t)b * row, sizeof(uint16_t) * (size_t)row);
                memcpy(dv, v_new + (int64_t)b * row, sizeof(uint16_t) * (size_t)row);
            } else {
                memset(dk, 0, sizeof(uint16_t) * (size_t)row);
                memset(dv, 0, sizeof(uint16_t) * (size_t)row);
            }
        }
    }

    /* 2. attention over the explicit concatenation */
    int G = Hq / Hkv;
    int n = Lp + Ls;
    int bad = 0;
    (void)n_threads;
#pragma omp parallel for schedule(dynamic, 1) num_threads(n_threads > 0 ? n_threads : 1) reduction(| : bad)
    for (int64_t r = 0; r < (int64_t)W * Hq; ++r) {
        int b = (int)(r / Hq), h = (int)(r % Hq), kvh = h / G;
        const uint16_t **keys = (const uint16_t **)malloc(sizeof(void *) * (size_t)n);
        const uint16_t **vals = (const uint16_t **)malloc(sizeof(void *) * (size_t)n);
        double *buf = (double *)malloc(sizeof(double) * (size_t)n);
        if (!keys || !vals || !buf) { bad = 1; free(keys); free(vals); free(buf); continue; }
        for (int j = 0; j < Lp; ++j) {
            keys[j] = kp + ((int64_t)j * Hkv + kvh) * D;
            vals[j] = vp + ((int64_t)j * Hkv + kvh) * D;
        }
        for (int s = 0; s < Ls; ++s) {
            keys[Lp + s] = ks_out + (((int64_t)b * Smax + s) * Hkv + kvh) * D;
            vals[Lp + s] = vs_out + (((int64_t)b * Smax + s) * Hkv + kvh) * D;
        }
        double l;
        attend_list(q + ((int64_t)b * Hq + h) * D, keys, vals, n, D, scale, buf,
                    o + ((int64_t)b * Hq + h) * D, &l);
        if (lse) lse[(int64_t)b * Hq + h] = l;
        free(keys); free(vals); free(buf);
    }
    return bad ? -1 : 0;
}

/* ------------------------------------------------------------------------- */
/* Beam candidate selection (section 3.3).                                    */
/* ------------------------------------------------------------------------- */

/* Row log-normaliser: lse_b = m + log sum_v exp(x_bv - m), fp64, rounded to fp32. */
int oracle_row_lse(const uint16_t *logits, int W_in, int64_t V, float *lse_out) {
    if (W_in < 0 || V <= 0) return -1;
    for (int b = 0; b < W_in; ++b) {
        const uint16_t *row = logits + (int64_t)b * V;
        double m = -INFINITY;
        for (int64_t v = 0; v < V; ++v) {
            double x = bf16_bits_to_f64(row[v]);
            if (x > m) m = x;
        }
        double s = 0.0;
        for (int64_t v = 0; v < V; ++v) s += exp(bf16_bits_to_f64(row[v]) - m);
        lse_out[b] = (float)(m + log(s));
    }
    return 0;
}

typedef struct {
    float score;  /* fl32(cum_b + fl32(x - lse_b)) */
    float x;      /* the bf16 logit, widened */
    int32_t b;    /* source beam (parent) */
    int32_t v;    /* token id */
} cand_t;

/* Total order of the flattened candidates: higher score first; equal scores
 * by lower parent; then by higher logit, then lower token id.  Within one beam
 * this is the per-beam Top-K order (logit descending, lowest id on ties), so
 * it equals "flat index ascending" of the two-stage method. */
static int cand_cmp(const void *pa, const void *pb) {
    const cand_t *a = (const cand_t *)pa, *c = (const cand_t *)pb;
    if (a->score > c->score) return -1;
    if (a->score < c->score) return 1;
    if (a->b != c->b) return a->b < c->b ? -1 : 1;
    if (a->x > c->x) return -1;
    if (a->x < c->x) return 1;
    if (a->v != c->v) return a->v < c->v ? -1 : 1;
    return 0;
}

/* Full sort of all W_in x V candidates; returns the first n_keep in order.
 *   logits [W_in, V] bf16 bits; cum [W_in] fp32; lse [W_in] fp32 (nullable:
 *   computed here by oracle_row_lse).  Outputs [n_keep]: token, parent, score.
 *   Returns 0, -1 on bad arguments, -2 on allocation failure. */
int oracle_beam_select(const uint16_t *logits, const float *cum, int W_in, int64_t V,
                       int n_keep, const float *lse_in, int32_t *out_token,
                       int32_t *out_parent, float *out_score, float *out_lse) {
    if (W_in <= 0 || V <= 0 || n_keep < 0 || (int64_t)n_keep > (int64_t)W_in * V) return -1;
    float *lse = (float *)malloc(sizeof(float) * (size_t)W_in);
    if (!lse) return -2;
    if (lse_in) memcpy(lse, lse_in, sizeof(float) * (size_t)W_in);
    else oracle_row_lse(logits, W_in, V, lse);
    if (out_lse) memcpy(out_lse, lse, sizeof(float) * (size_t)W_in);

    int64_t N = (int64_t)W_in * V;
    cand_t *c = (cand_t *)malloc(sizeof(cand_t) * (size_t)N);
    if (!c) { free(lse); return -2; }
    for (int b = 0; b < W_in; ++b) {
        for (int64_t v = 0; v < V; ++v) {
            float x = bf16_bits_to_f32(logits[(int64_t)b * V + v]);
            float lp = x - lse[b];          /* FP32 log-probability */
            float sc = cum[b] + lp;         /* plus the beam's cumulative score */
            cand_t *e = &c[(int64_t)b * V + v];
            e->score = sc; e->x = x; e->b = b; e->v = (int32_t)v;
        }
    }
    qsort(c, (size_t)N, sizeof(cand_t), cand_cmp);
    for (int i = 0; i < n_keep; ++i) {
        out_token[i] = c[i].v;
        out_parent[i] = c[i].b;
        out_score[i] = c[i].score;
    }
    free(c);
    free(lse);
    return 0;
}
