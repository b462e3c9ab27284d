/*
 * ll.h -- C ABI of libll.so: batch-1 autoregressive decode of a Llama-style
 * decoder on one NVIDIA GB300 (sm_103a), one decode step per launch of a
 * persistent megakernel.
 *
 * Source of the method: the page "Hazy Research Llama-3.2-1B Megakernel" (a
 * Chinese write-up at w2o.qhhnjy.cn/html/17f999973.html). Its instruction list
 * defines what one step computes: per layer (1) RMSNorm fused with the QKV
 * projection and RoPE, (2) attention as matrix product plus reduction with GQA
 * over long sequences, (3) O projection plus residual, (4) MLP RMSNorm with the
 * SiLU-gated gate and up projections, (5) down projection plus residual; after
 * the last layer (6) RMSNorm plus the language-modelling head. In front of the
 * layers the step looks up the token embedding, and after the head it takes
 * the greedy argmax. The page's paragraphs on the instruction interpreter, the
 * shared-memory pages and the global-memory counters describe how the library
 * runs that step as one kernel; the page defines no programming interface, so
 * the calls below are this library's own.
 *
 * Conventions shared by every call:
 *   - bf16 tensors are passed as uint16_t bit patterns; every matrix is
 *     row-major [out][in]. All tensor pointers are DEVICE pointers and must be
 *     16-byte aligned.
 *   - The caller owns the weights, the KV caches and every output buffer; they
 *     must stay allocated and unchanged (weights) while the handle lives. The
 *     library owns its schedule, scratch, counters and status word.
 *   - All GPU work is enqueued on the stream given to ll_init (a cudaStream_t
 *     passed as void*; NULL means the legacy default stream).
 *   - Return codes are LL_OK (0) or one of the negative LL_ERR_* values; after
 *     an error ll_last_error() holds a one-line explanation.
 *   - A handle is not thread-safe: calls on one handle must not overlap.
 */
#ifndef LL_H
#define LL_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define LL_OK 0
#define LL_ERR_ARG (-1)          /* bad argument: null/misaligned pointer, token or pos out of range */
#define LL_ERR_SHAPE (-2)        /* model shape the kernels do not support */
#define LL_ERR_CUDA (-3)         /* a CUDA runtime call failed */
#define LL_ERR_DEP_TIMEOUT (-4)  /* a device-side wait ran past its time limit; the step was abandoned */
#define LL_ERR_OOM (-5)          /* library scratch could not be allocated */
#define LL_ERR_DEVICE (-6)       /* device is not sm_103 or cannot co-schedule one block per SM */
#define LL_ERR_NUMERIC (-7)      /* the logits held no orderable value (all NaN): no greedy token (the
                                    token outputs read -1, and a multi-step launch stops there) */

#define LL_BACKEND_MEGAKERNEL 0  /* one persistent kernel per decode step */
#define LL_BACKEND_CHAIN 1       /* one kernel per operation, for comparison */

typedef struct ll_handle ll_handle;

/* Model shape. Constraints checked by ll_init (LL_ERR_SHAPE otherwise):
 * n_q_heads % n_kv_heads == 0 and n_q_heads / n_kv_heads <= 8; head_dim 64 or
 * 128; hidden, n_q_heads*head_dim and inter multiples of 256 and at most 16384;
 * n_q_heads*head_dim at most 4096; each of those widths must split into at most
 * 16 slices of 256, 512, 768 or 1024 elements; max_seq >= 1. */
typedef struct {
    int32_t n_layers;
    int32_t hidden;
    int32_t n_q_heads;
    int32_t n_kv_heads;
    int32_t head_dim;
    int32_t inter;      /* SwiGLU intermediate width */
    int32_t vocab;
    int32_t max_seq;    /* positions the KV caches hold */
    int32_t tied;       /* nonzero: the LM head is the embedding matrix */
    int32_t backend;    /* LL_BACKEND_MEGAKERNEL or LL_BACKEND_CHAIN */
    float rms_eps;
    float rope_theta;
} ll_config;

/* Weight pointers. The per-layer members are HOST arrays of n_layers DEVICE
 * pointers; ll_init copies them, so the host arrays may be freed afterwards. */
typedef struct {
    const uint16_t *embed;        /* [vocab][hidden] */
    const uint16_t *lm_head;      /* [vocab][hidden]; ignored (may be NULL) when tied */
    const uint16_t *final_norm;   /* [hidden] */
    const uint16_t *const *attn_norm; /* [hidden] */
    const uint16_t *const *wq;    /* [n_q_heads*head_dim][hidden] */
    const uint16_t *const *wk;    /* [n_kv_heads*head_dim][hidden] */
    const uint16_t *const *wv;    /* [n_kv_heads*head_dim][hidden] */
    const uint16_t *const *wo;    /* [hidden][n_q_heads*head_dim] */
    const uint16_t *const *mlp_norm; /* [hidden] */
    const uint16_t *const *wg;    /* [inter][hidden] */
    const uint16_t *const *wu;    /* [inter][hidden] */
    const uint16_t *const *wd;    /* [hidden][inter] */
} ll_weights;

/* Create a decoder for one sequence on the current CUDA device.
 *   k_cache, v_cache: caller-owned device buffers, bf16,
 *     [n_layers][n_kv_heads][max_seq][head_dim]. Step `pos` writes entry pos and
 *     reads entries 0..pos; entries the caller filled beforehand are used as is.
 *   stream: cudaStream_t (as void*) that every later call enqueues on.
 * Builds the per-SM instruction schedule and the RoPE table, allocates library
 * scratch, and checks that the device is sm_103 and can keep one block resident
 * on every SM. On success *out receives the handle; on failure *out is NULL and
 * the code says why (no handle exists to query, so the reason is printed by
 * ll_init_error()). */
int ll_init(const ll_config *cfg, const ll_weights *w, uint16_t *k_cache, uint16_t *v_cache,
            void *stream, ll_handle **out);

/* Reason for the last ll_init failure in this process (static string). */
const char *ll_init_error(void);

/* One decode step, synchronous: input token `token` at position `pos`
 * (0 <= token < vocab, 0 <= pos < max_seq). Writes K/V entry pos, writes the
 * fp32 logits [vocab] to logits_dev when it is not NULL, stores the greedy next
 * token (lowest index among equal maxima) to *next_token_host when it is not
 * NULL, waits for the stream, and returns the step's status. */
int ll_decode_step(ll_handle *h, int32_t token, int32_t pos, float *logits_dev,
                   int32_t *next_token_host);

/* One decode step, enqueued only: the input token is read on the device from
 * *token_dev and the next token written to *next_token_dev (both device int32;
 * they may be the same address, which chains steps without the host). pos is
 * checked on the host; a token out of range is caught on the device and ends
 * the step with LL_ERR_ARG. Errors on the device are sticky: later steps return
 * at once, and ll_synchronize() reports and clears them. */
int ll_decode_step_async(ll_handle *h, const int32_t *token_dev, int32_t pos, float *logits_dev,
                         int32_t *next_token_dev);

/* n_steps greedy decode steps in one launch of the persistent kernel, enqueued
 * only (the page's interpreter keeps its per-SM schedule for every token; here
 * it also keeps running from one token to the next, so the weight pages of a
 * step stream in while the previous step's LM head and argmax finish). Step i
 * decodes at position pos + i: step 0 reads its token from *token_dev, step
 * i > 0 the token step i - 1 chose, and step i writes its next token to
 * tokens_dev[i] and, when logits_dev is not NULL, its fp32 logits to
 * logits_dev + i * vocab (so logits_dev holds n_steps * vocab floats).
 * token_dev and tokens_dev are device int32 and must not be NULL; tokens_dev
 * holds n_steps values, and token_dev may point into it (every block reads
 * *token_dev before step 0 can finish). Requires
 * n_steps >= 1 and pos + n_steps <= max_seq (LL_ERR_ARG otherwise). Results are
 * bit-identical to n_steps calls of ll_decode_step_async chained on the device.
 * Errors are sticky as for ll_decode_step_async; ll_synchronize() reports them.
 * The per-operation backend runs the same steps as separate launches. */
int ll_decode_steps(ll_handle *h, const int32_t *token_dev, int32_t pos, int32_t n_steps, float *logits_dev,
                    int32_t *tokens_dev);

/* Prefill: the n prompt tokens tokens_dev[0..n) (device int32) at positions
 * pos0 .. pos0 + n - 1 through every layer at once, writing their K/V entries to
 * the cache, then the last position's final RMSNorm, LM head and greedy token:
 * logits_dev (device [vocab] fp32, or NULL) and next_token_dev (device int32).
 * The same computation as n ll_decode_step calls at those positions (what the
 * page's decode step computes, for many positions: the instruction list's
 * projections become matrix products), here as tcgen05 GEMMs with TMA-staged
 * bf16 operands and tensor-memory accumulators, the activations as three
 * bf16 terms, plus a causal attention (mma.sync tiles) over the cache entries
 * 0..pos0 + t of each position t. Asynchronous on the handle's stream; a token out of range is
 * reported by ll_synchronize (LL_ERR_ARG). Single-sequence handles only (LL_ERR_ARG
 * on a batched one); needs hidden, n_q_heads*head_dim and inter multiples of 64
 * (LL_ERR_SHAPE). The first call, and any call with more positions than before,
 * allocates the prefill buffers (cudaMalloc, about n x (10 hidden + 10 q + 8 kv
 * + 6 inter) bytes plus the weight tensor maps; LL_ERR_OOM if that fails);
 * ll_free releases them. */
int ll_prefill(ll_handle *h, const int32_t *tokens_dev, int32_t n, int32_t pos0, float *logits_dev,
               int32_t *next_token_dev);

/* Small-batch decode: n_seq independent sequences (1, 2, 4 or 8) share every
 * pass over the weights. The page's method is batch 1; it says a batch turns the
 * matrix-vector products into skinny matrix products, where tensor cores pay
 * (its paragraph on CUDA-core against tensor-core matvec), so these handles run
 * the tensor-core kernel: each weight page is multiplied with all sequences'
 * inputs in the same m16n8k16 products, while every sequence keeps its own KV
 * cache, position, attention items, logits and greedy tokens. Two sequences
 * whose widths give at most 16 input floats per sequence and lane (hidden,
 * n_q_heads*head_dim and inter of 1024, 2048 or 8192) run on CUDA-core pages
 * instead, each page multiplied with both inputs (measured faster; the
 * environment variable LL_BATCH_CC=0 at ll_init_batch keeps tensor-core pages;
 * ll_query LL_Q_BATCH_CC reports which).
 *
 * ll_init_batch: as ll_init, with k_caches / v_caches host arrays of n_seq
 * device pointers, one cache pair per sequence, each laid out as ll_init's
 * (caller-owned, 16-byte aligned). Needs the two-sequence CUDA-core widths
 * above, or hidden, n_q_heads*head_dim and inter multiples of 1024, the
 * megakernel backend, and rows per SM x n_seq within the kernel's accumulator
 * (LL_ERR_SHAPE otherwise); attention uses the block-wide
 * softmax variant and about max_seq / 128 KV splits, at most n_sm / (n_kv *
 * n_seq). A batched handle is stepped only by ll_decode_steps_batch (the other
 * step calls return LL_ERR_ARG); ll_synchronize, ll_set_timeout_ns,
 * ll_set_trace, ll_query (LL_Q_BATCH) and ll_free apply as to any handle. */
int ll_init_batch(const ll_config *cfg, const ll_weights *w, uint16_t *const *k_caches, uint16_t *const *v_caches,
                  int32_t n_seq, void *stream, ll_handle **out);

/* n_steps greedy steps of every sequence of a batched handle in one launch.
 * tokens_in_dev: device [n_seq] input tokens of the first step. pos_host: host
 * [n_seq] first positions (sequence b decodes at pos_host[b] + i in step i;
 * every pos_host[b] + n_steps <= max_seq, LL_ERR_ARG otherwise). logits_dev:
 * device [n_steps][n_seq][vocab] fp32, or NULL. tokens_dev: device
 * [n_steps][n_seq] greedy tokens; step i of sequence b reads the token step i - 1
 * chose for it. Asynchronous on the handle's stream, errors as ll_decode_steps. */
int ll_decode_steps_batch(ll_handle *h, const int32_t *tokens_in_dev, const int32_t *pos_host, int32_t n_steps,
                          float *logits_dev, int32_t *tokens_dev);

/* Wait for the handle's stream, then return and clear the device status of the
 * steps enqueued since the last check (LL_OK if all of them succeeded). After
 * an error the library clears its device state, so the next step starts clean. */
int ll_synchronize(ll_handle *h);

/* Upper bound, in nanoseconds, on any single device-side wait (for tagged
 * activations from other SMs, and the shared-memory page handoff). Past it the kernel records
 * LL_ERR_DEP_TIMEOUT, lets its own copies land, and returns. Default 1 s. */
int ll_set_timeout_ns(ll_handle *h, uint64_t ns);

/* Timing trace of the megakernel (the page's time breakdown of one forward pass
 * is what it is for). trace_dev is a caller-owned device buffer of at least
 * LL_Q_TRACE_BYTES bytes. Its first part, [sm][instr][12] uint64 (max_instr from
 * ll_plan), holds per instruction: consumer begin, dependency met and input
 * loaded, pages consumed, end, the producer's first and last page issue, the
 * first page in the consumers' hands, the compute on the pages done, and for
 * attention the ends of the scores, softmax and P.V phases and of its signal.
 * The second part, [sm][4096][3] uint64, holds per shared-memory page (page
 * number modulo 4096): producer issue, consumer start, release. All values are
 * %globaltimer nanoseconds; each traced step (every step of a multi-step
 * launch) overwrites them. NULL turns tracing
 * off (the default). Returns LL_ERR_ARG if the buffer is too small or misaligned. */
int ll_set_trace(ll_handle *h, uint64_t *trace_dev, size_t bytes);

/* Schedule and memory facts, for tests and reports. */
#define LL_Q_NUM_SMS 0          /* blocks of the persistent kernel (one per SM) */
#define LL_Q_ATTN_SPLITS 1      /* KV splits per KV head in the attention instruction */
#define LL_Q_PAGE_BYTES 2       /* bytes of one shared-memory page */
#define LL_Q_NUM_PAGES 3        /* pages per SM */
#define LL_Q_SCRATCH_BYTES 4    /* device bytes the library allocated */
#define LL_Q_MAX_INSTRS 5       /* longest per-SM instruction list */
#define LL_Q_LAUNCHES_PER_STEP 6 /* kernel launches one decode step makes (ll_decode_steps: one launch for all its steps) */
#define LL_Q_SMEM_BYTES 7       /* dynamic shared memory per block */
#define LL_Q_TRACE_BYTES 8      /* size of the buffer ll_set_trace needs */
#define LL_Q_BATCH 10           /* sequences a handle decodes together */
#define LL_Q_MV_TC 9            /* matrix-vector widths on tensor-core pages: bit 0 hidden, bit 1 n_q*head_dim, bit 2 inter */
#define LL_Q_BATCH_CC 12        /* 1: a batch of two on CUDA-core pages (each page read once for both sequences) */
int ll_query(const ll_handle *h, int what, int64_t *value);

/* Fault injection for tests (host side only; nothing faults on the device):
 * LL_FAULT_DROP_SIGNAL removes the completion signal of every instruction of
 * kind `op` (0 QKV, 1 attention, 2 O projection, 3 gate/up, 4 down) in layer
 * `layer`: those instructions store their outputs with a tag no reader accepts,
 * so the instruction waiting on them runs into its time limit and the step
 * returns LL_ERR_DEP_TIMEOUT. LL_FAULT_NONE restores the schedule. */
#define LL_FAULT_NONE 0
#define LL_FAULT_DROP_SIGNAL 1
int ll_debug_inject(ll_handle *h, int kind, int layer, int op);

/* The per-SM instruction schedule ll_init would build for `cfg` on a device
 * with `nsm` SMs; host only, needs no GPU. *max_instr receives the longest list.
 * When out is not NULL it must hold nsm*max_instr*7 int32, filled [sm][i] with
 * (op, layer, r0, r1, wait_counter, wait_count, signal_counter); op is 0 QKV,
 * 1 attention, 2 O projection, 3 gate/up, 4 down, 5 LM head, -1 an unused slot;
 * [r0, r1) is the SM's row range, or (KV head, split) for attention. The
 * counter fields name the dependency: the instruction reads the outputs that
 * wait_count instructions marked signal_counter produce (the kernel finds
 * them ready by their tags); -1 where there is none. */
int ll_plan(const ll_config *cfg, int32_t nsm, int32_t *out, size_t out_len, int32_t *max_instr);

/* The handle's own per-SM instruction lists, in ll_plan's format (for a batched
 * handle they hold its sequences' attention items and LM-head pieces). */
int ll_handle_plan(const ll_handle *h, int32_t *out, size_t out_len, int32_t *max_instr);

/* Explanation of the last error on this handle (never NULL). */
const char *ll_last_error(const ll_handle *h);

/* Release library memory (not the caller's weights, caches or buffers). NULL is a no-op. */
void ll_free(ll_handle *h);

/* One decode step that allocates no device memory, for callers that cannot
 * call cudaMalloc. The pages define no such call (they have no counterpart to
 * it): it is the one-kernel-per-operation path of LL_BACKEND_CHAIN with all of
 * its scratch (activations, attention partials, the RoPE row of pos, the status
 * word and the next token) in one file-scope device array of
 * LL_STATIC_SCRATCH_BYTES bytes per device, shared by every call.
 *   cfg, w: as for ll_init (cfg->backend is ignored); the per-layer host arrays
 *     are read during the call only. n_layers is at most LL_STATIC_MAX_LAYERS.
 *   k_cache, v_cache, token, pos, logits_dev, next_token_host: as for
 *     ll_decode_step; logits_dev may be NULL (the logits then use the array).
 *   stream: cudaStream_t (as void*) the work is enqueued on; the call waits for
 *     it before returning.
 *   err, err_len: optional caller buffer that receives a one-line reason on
 *     failure (truncated to err_len bytes, NUL-terminated); NULL for none.
 * Returns LL_OK or LL_ERR_ARG / LL_ERR_SHAPE / LL_ERR_CUDA / LL_ERR_DEVICE. A
 * shape whose scratch would exceed LL_STATIC_SCRATCH_BYTES is rejected with
 * LL_ERR_SHAPE and a message giving the bytes it needs; nothing is launched.
 * The first call on a device (the device current at the call) sets up that
 * device: it looks up the array's device address (cudaGetSymbolAddress) and
 * the SM count. Make that first call before any stream capture. The call
 * itself calls no cudaMalloc, cudaFree or other allocating routine; it clears
 * the status word at the start of every step (everything else is written
 * before it is read). Calls whose GPU work overlaps in time, on any streams or
 * threads, race on the shared array: serialise them. */
#define LL_STATIC_SCRATCH_BYTES 4194304
#define LL_STATIC_MAX_LAYERS 256
int ll_decode_step_static(const ll_config *cfg, const ll_weights *w, uint16_t *k_cache, uint16_t *v_cache,
                          int32_t token, int32_t pos, float *logits_dev, int32_t *next_token_host, void *stream,
                          char *err, size_t err_len);

#ifdef __cplusplus
}
#endif
#endif /* LL_H */
