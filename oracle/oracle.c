/*
 * oracle.c -- plain, slow, obviously correct CPU oracle of one batch-1 decode
 * step of a Llama-style decoder.
 *
 * TEST INFRASTRUCTURE. Only the test suite, the smoke check and the benchmark's
 * CPU-baseline leg may link, load or call this code. The product path never
 * does, and the two share no code.
 *
 * Source of the method: the page "Hazy Research Llama-3.2-1B Megakernel"
 * (a Chinese write-up at w2o.qhhnjy.cn/html/17f999973.html). Its instruction
 * list names, per layer, (1) RMSNorm fused with the QKV projection and RoPE,
 * (2) attention as a matrix product plus a reduction, with GQA and long
 * sequences, (3) the O projection plus the residual add, (4) the MLP RMSNorm,
 * the SiLU-gated activation and the up projection, (5) the down projection plus
 * the final residual, and after the last layer (6) RMSNorm plus the language
 * modelling head. The megakernel only reorders and fuses this computation, so
 * the oracle is the standard Llama decode forward written out in that order,
 * with the token embedding lookup in front and a greedy argmax at the end.
 *
 * Readings where the page is silent (each also listed in the design notes):
 *   - RMSNorm: x * 1/sqrt(mean(x^2) + eps) * g, no bias.
 *   - RoPE: "rotate half" pairing (i with i + hd/2), angle pos * theta^(-2i/hd),
 *     no frequency scaling; the angle and its cos/sin are taken in double.
 *   - Attention: scale 1/sqrt(hd), softmax with max subtraction, causal by
 *     construction (only cache entries 0..pos exist); query head h reads KV
 *     head floor(h / (n_q / n_kv)).
 *   - The new k (after RoPE) and v are rounded to bf16 (round to nearest even),
 *     stored in the cache at pos, and attention reads every entry 0..pos back
 *     from the bf16 cache, the new one included.
 *   - MLP: down( silu(gate(h)) * up(h) ), silu(z) = z / (1 + exp(-z)).
 *   - Greedy argmax returns the lowest index among equal maxima.
 *
 * Arithmetic: every step runs in REAL (float for orc32_, double for orc64_) on
 * bf16 weights widened exactly. Dot products accumulate left to right.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#include "oracle.h"

#ifndef ORC_REAL
#error "compile with -DORC_REAL=float|double -DORC_PREFIX=orc32_|orc64_"
#endif
#define ORC_CAT2(a, b) a##b
#define ORC_CAT(a, b) ORC_CAT2(a, b)
#define F(name) ORC_CAT(ORC_PREFIX, name)

typedef ORC_REAL real;

#if ORC_IS_DOUBLE
#define R_EXP exp
#define R_SQRT sqrt
#else
#define R_EXP expf
#define R_SQRT sqrtf
#endif

/* bf16 is the upper half of an IEEE binary32; widening is exact. */
real F(from_bf16)(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (real)f;
}

static uint16_t float_to_bf16_rne(float f) {
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    if ((u & 0x7f800000u) == 0x7f800000u && (u & 0x007fffffu)) return 0x7fc0; /* NaN */
    u += 0x7fffu + ((u >> 16) & 1u); /* round to nearest, ties to even */
    return (uint16_t)(u >> 16);
}

/* Round to the nearest bf16 value, ties to even. */
uint16_t F(to_bf16)(real v) {
#if ORC_IS_DOUBLE
    /* Round the double directly to 8 significant bits, so that no float
     * rounding happens in between. Values below the bf16 normal range go
     * through float, where bf16 subnormals are handled bit-wise. */
    if (isnan(v)) return 0x7fc0;
    if (v == 0.0 || isinf(v) || fabs(v) < 0x1p-126) return float_to_bf16_rne((float)v);
    int e;
    double m = frexp(v, &e);                 /* v = m * 2^e, 0.5 <= |m| < 1 */
    double r = ldexp(nearbyint(ldexp(m, 8)), e - 8); /* default mode: ties to even */
    return float_to_bf16_rne((float)r);      /* exact: r has 8 significant bits */
#else
    return float_to_bf16_rne(v);
#endif
}

/* RMSNorm, instruction list steps 1, 4 and 6: out = x / sqrt(mean(x^2) + eps) * g. */
void F(rmsnorm)(const real *x, const uint16_t *g, int n, double eps, real *out) {
    real ss = 0;
    for (int i = 0; i < n; i++) ss += x[i] * x[i];
    real r = (real)1 / R_SQRT(ss / (real)n + (real)eps);
    for (int i = 0; i < n; i++) out[i] = x[i] * r * F(from_bf16)(g[i]);
}

/* y = W x for a row-major [rows][cols] bf16 matrix (every projection). Rows are
 * independent, so they may run on several threads; each row sums left to right. */
void F(matvec)(const uint16_t *w, const real *x, int rows, int cols, real *y) {
#ifdef _OPENMP
#pragma omp parallel for schedule(static)
#endif
    for (int r = 0; r < rows; r++) {
        const uint16_t *wr = w + (size_t)r * (size_t)cols;
        real acc = 0;
        for (int c = 0; c < cols; c++) acc += F(from_bf16)(wr[c]) * x[c];
        y[r] = acc;
    }
}

/* RoPE on one head, in place (instruction list step 1). */
void F(rope)(real *v, int head_dim, int pos, double theta) {
    int half = head_dim / 2;
    for (int i = 0; i < half; i++) {
        double ang = (double)pos * pow(theta, -2.0 * (double)i / (double)head_dim);
        real c = (real)cos(ang), s = (real)sin(ang);
        real a = v[i], b = v[i + half];
        v[i] = a * c - b * s;
        v[i + half] = a * s + b * c;
    }
}

/* SiLU gate of the MLP (instruction list step 4). */
real F(silu)(real z) { return z / ((real)1 + R_EXP(-z)); }

/* One query head attending over n_pos cached entries k[j], v[j] (bf16, [n_pos][hd]),
 * instruction list step 2. */
void F(attention)(const real *q, const uint16_t *k, const uint16_t *v, int n_pos,
                  int head_dim, real *out) {
    real *s = (real *)malloc((size_t)n_pos * sizeof(real));
    real scale = (real)1 / R_SQRT((real)head_dim);
    real m = -INFINITY;
    for (int j = 0; j < n_pos; j++) {
        real acc = 0;
        for (int d = 0; d < head_dim; d++) acc += q[d] * F(from_bf16)(k[(size_t)j * head_dim + d]);
        s[j] = acc * scale;
        if (s[j] > m) m = s[j];
    }
    real l = 0;
    for (int j = 0; j < n_pos; j++) {
        s[j] = R_EXP(s[j] - m);
        l += s[j];
    }
    for (int d = 0; d < head_dim; d++) {
        real acc = 0;
        for (int j = 0; j < n_pos; j++) acc += s[j] * F(from_bf16)(v[(size_t)j * head_dim + d]);
        out[d] = acc / l;
    }
    free(s);
}

/* Greedy decoding: index of the largest value, lowest index on ties. */
int F(argmax)(const real *v, int n) {
    int best = 0;
    for (int i = 1; i < n; i++)
        if (v[i] > v[best]) best = i;
    return best;
}

/* One decode step at position pos for input token `token`: writes the new k, v
 * into the caches ([L][n_kv][max_seq][hd] bf16), the logits into `logits` [V],
 * and returns the greedy next token (negative on a bad argument). */
int F(decode_step)(const orc_config *cfg, const orc_weights *w, uint16_t *k_cache,
                   uint16_t *v_cache, int token, int pos, real *logits) {
    const int H = cfg->hidden, nq = cfg->n_q_heads, nkv = cfg->n_kv_heads;
    const int hd = cfg->head_dim, I = cfg->inter, V = cfg->vocab, S = cfg->max_seq;
    if (token < 0 || token >= V || pos < 0 || pos >= S) return -1;
    if (nkv <= 0 || nq % nkv != 0 || hd % 2 != 0) return -2;
    const int G = nq / nkv;

    real *x = (real *)calloc((size_t)H, sizeof(real));
    real *h = (real *)calloc((size_t)(H > I ? H : I), sizeof(real));
    real *q = (real *)calloc((size_t)nq * hd, sizeof(real));
    real *k = (real *)calloc((size_t)nkv * hd, sizeof(real));
    real *v = (real *)calloc((size_t)nkv * hd, sizeof(real));
    real *o = (real *)calloc((size_t)nq * hd, sizeof(real));
    real *t = (real *)calloc((size_t)H, sizeof(real));
    real *gt = (real *)calloc((size_t)I, sizeof(real));
    real *up = (real *)calloc((size_t)I, sizeof(real));
    real *a = (real *)calloc((size_t)I, sizeof(real));

    /* token embedding lookup */
    for (int i = 0; i < H; i++) x[i] = F(from_bf16)(w->embed[(size_t)token * H + i]);

    for (int l = 0; l < cfg->n_layers; l++) {
        /* (1) RMSNorm + QKV projection + RoPE, then the KV cache write at pos */
        F(rmsnorm)(x, w->attn_norm[l], H, cfg->rms_eps, h);
        F(matvec)(w->wq[l], h, nq * hd, H, q);
        F(matvec)(w->wk[l], h, nkv * hd, H, k);
        F(matvec)(w->wv[l], h, nkv * hd, H, v);
        for (int qh = 0; qh < nq; qh++) F(rope)(q + (size_t)qh * hd, hd, pos, cfg->rope_theta);
        for (int g = 0; g < nkv; g++) F(rope)(k + (size_t)g * hd, hd, pos, cfg->rope_theta);
        for (int g = 0; g < nkv; g++) {
            size_t base = (((size_t)l * nkv + g) * S + pos) * hd;
            for (int d = 0; d < hd; d++) {
                k_cache[base + d] = F(to_bf16)(k[(size_t)g * hd + d]);
                v_cache[base + d] = F(to_bf16)(v[(size_t)g * hd + d]);
            }
        }
        /* (2) attention of each query head over cache entries 0..pos of its KV head */
        for (int qh = 0; qh < nq; qh++) {
            int g = qh / G;
            size_t base = ((size_t)l * nkv + g) * S * hd;
            F(attention)(q + (size_t)qh * hd, k_cache + base, v_cache + base, pos + 1, hd,
                         o + (size_t)qh * hd);
        }
        /* (3) O projection + residual */
        F(matvec)(w->wo[l], o, H, nq * hd, t);
        for (int i = 0; i < H; i++) x[i] += t[i];
        /* (4) MLP RMSNorm + SiLU-gated gate/up projections */
        F(rmsnorm)(x, w->mlp_norm[l], H, cfg->rms_eps, h);
        F(matvec)(w->wg[l], h, I, H, gt);
        F(matvec)(w->wu[l], h, I, H, up);
        for (int i = 0; i < I; i++) a[i] = F(silu)(gt[i]) * up[i];
        /* (5) down projection + residual */
        F(matvec)(w->wd[l], a, H, I, t);
        for (int i = 0; i < H; i++) x[i] += t[i];
    }
    /* (6) final RMSNorm + LM head, then greedy argmax */
    F(rmsnorm)(x, w->final_norm, H, cfg->rms_eps, h);
    F(matvec)(cfg->tied ? w->embed : w->lm_head, h, V, H, logits);
    int next = F(argmax)(logits, V);

    free(x); free(h); free(q); free(k); free(v); free(o); free(t); free(gt); free(up); free(a);
    return next;
}

#if !ORC_IS_DOUBLE
int orc_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Threads for the row-parallel loops from now on (n >= 1); timing only, the
 * results do not depend on it (each output row is one thread's sum). */
void orc_set_threads(int n) {
#ifdef _OPENMP
    if (n >= 1) omp_set_num_threads(n);
#else
    (void)n;
#endif
}
#endif
