/*
 * oracle.h -- declarations of the plain CPU oracle for one batch-1 decode step
 * of a Llama-style decoder.
 *
 * TEST INFRASTRUCTURE. Only the test suite, the smoke check and the benchmark's
 * CPU-baseline leg may link, load or call this code. The product path (the CUDA
 * library under decode_megakernel_persistent_gb300/) never does, and shares no
 * code, header, table or helper with it.
 *
 * The same source (oracle.c) is compiled twice: once with float arithmetic
 * (symbols prefixed orc32_) and once with double arithmetic (prefixed orc64_).
 * Weights and the KV cache are bf16 bit patterns held in uint16_t arrays.
 */
#ifndef ORACLE_H
#define ORACLE_H

#include <stdint.h>

typedef struct {
    int n_layers;    /* decoder layers L */
    int hidden;      /* model width H */
    int n_q_heads;   /* query heads */
    int n_kv_heads;  /* key/value heads (GQA groups) */
    int head_dim;    /* per-head width */
    int inter;       /* SwiGLU intermediate width I */
    int vocab;       /* vocabulary size V */
    int max_seq;     /* positions held by the KV cache */
    int tied;        /* 1: LM head is the embedding matrix */
    double rms_eps;  /* RMSNorm epsilon */
    double rope_theta; /* RoPE base */
} orc_config;

/* Host pointers to bf16 bit patterns, row-major [out][in] for every matrix.
 * Per-layer tensors are arrays of n_layers pointers. */
typedef struct {
    const uint16_t *embed;       /* [V][H] */
    const uint16_t *lm_head;     /* [V][H], ignored when tied */
    const uint16_t *final_norm;  /* [H] */
    const uint16_t *const *attn_norm; /* [H] */
    const uint16_t *const *wq;   /* [nq*hd][H] */
    const uint16_t *const *wk;   /* [nkv*hd][H] */
    const uint16_t *const *wv;   /* [nkv*hd][H] */
    const uint16_t *const *wo;   /* [H][nq*hd] */
    const uint16_t *const *mlp_norm; /* [H] */
    const uint16_t *const *wg;   /* [I][H] */
    const uint16_t *const *wu;   /* [I][H] */
    const uint16_t *const *wd;   /* [H][I] */
} orc_weights;

#define ORC_DECLARE(P, REAL)                                                         \
    uint16_t P##to_bf16(REAL v);                                                     \
    REAL P##from_bf16(uint16_t b);                                                   \
    void P##rmsnorm(const REAL *x, const uint16_t *g, int n, double eps, REAL *out); \
    void P##matvec(const uint16_t *w, const REAL *x, int rows, int cols, REAL *y);   \
    void P##rope(REAL *v, int head_dim, int pos, double theta);                      \
    REAL P##silu(REAL z);                                                            \
    void P##attention(const REAL *q, const uint16_t *k, const uint16_t *v,           \
                      int n_pos, int head_dim, REAL *out);                           \
    int P##argmax(const REAL *v, int n);                                             \
    int P##decode_step(const orc_config *cfg, const orc_weights *w,                  \
                       uint16_t *k_cache, uint16_t *v_cache, int token, int pos,     \
                       REAL *logits);

ORC_DECLARE(orc32_, float)
ORC_DECLARE(orc64_, double)

int orc_num_threads(void);
void orc_set_threads(int n);

#endif
