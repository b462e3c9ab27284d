// ll_internal.h -- structures shared by the host runtime (api.cpp, schedule.cpp)
// and the device code (megakernel.cuh and its instantiations, chain.cu) of libll.so.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <vector>

#include "../../include/ll.h"

namespace ll {

// ---- persistent-kernel geometry -------------------------------------------------
// One block per SM: NCW consumer warps compute, one producer warp streams bytes
// from HBM into a ring of NPAGES shared-memory pages of PAGE_BYTES each.
constexpr int NCW = 16;
constexpr int NCT = NCW * 32;              // consumer threads
constexpr int NTHREADS = NCT + 32;         // + producer warp
// The ring geometry; another one can be built for comparison (LL_RING=12x16 or
// 8x24 before build(): pages x KB), the total held at 192 KB.
#ifndef LL_PAGE_BYTES
#define LL_PAGE_BYTES 32768
#endif
#ifndef LL_NPAGES
#define LL_NPAGES 6
#endif
constexpr int PAGE_BYTES = LL_PAGE_BYTES;
constexpr int NPAGES = LL_NPAGES;
constexpr int MAX_VPL = 4;                 // 16-byte input vectors per lane (register budget)
constexpr int MAX_GQA = 8;                 // query heads per KV head
constexpr int MAX_HD = 128;
constexpr int MAX_RPP = 64;                // rows per page (hidden 256 at one vector per lane)
constexpr int MAX_PART = 128;              // (row, k-slice) partial sums per page
constexpr int ACC_FLOATS = 2048;           // rows of one SM's matrix-vector instruction, at most
constexpr int XIN_FLOATS = 4096;           // largest O-projection input (n_q_heads * head_dim)
constexpr int KPART_FLOATS = XIN_FLOATS;   // (row, k-slice) partial sums of one instruction
constexpr int XOWN_MAX = 64;               // residual rows one SM owns (hidden / SMs, rounded up)
constexpr int ATTN_SPLIT_POS = 128;        // cached positions one attention split aims at
constexpr int ATT_WARPS = 8;               // warps that split an attention page's P.V
constexpr int TRACE_WORDS = 12;            // timestamps per traced instruction
#ifndef LL_MAX_B
#define LL_MAX_B 8
#endif
constexpr int MAX_B = LL_MAX_B;            // sequences one batched handle decodes together
constexpr int BACC_FLOATS = 1024;          // per-SM row results x sequences of a tensor-core instruction
constexpr int PTRACE_PAGES = 4096;         // pages per SM the page trace keeps (a ring)

// Instruction kinds, in the order they appear within a layer.
enum Op : uint8_t { OP_QKV = 0, OP_ATTN = 1, OP_OPROJ = 2, OP_GATEUP = 3, OP_DOWN = 4, OP_LMHEAD = 5 };

// One entry of an SM's instruction list. For matrix-vector instructions
// [r0, r1) is the SM's row range (for QKV in the stacked [q; k; v] rows, for
// gate/up in the intermediate rows of both matrices); for attention r0 is the KV
// head and r1 the split index. sub: the sequence of an attention item (batched
// handles); for the LM head, 1 on the SM's last LM-head instruction (batched
// handles cut an SM's vocabulary rows into several).
struct Instr {
    uint8_t op;
    uint8_t sub;
    uint16_t layer;
    int32_t r0, r1;
    int32_t wait_ctr;     // counter to wait on, -1 for none
    uint32_t wait_count;  // its increments per step (target = epoch * wait_count)
    int32_t sig_ctr;      // counter to bump when done, -1 for none
};

// Matrix-vector geometry for one input width K. The consumer warps form `teams`
// teams of NCW / teams warps; page number p of the SM goes to team p % teams, so
// several pages are worked on at once. A page holds rpp whole rows. Within a
// team the row is cut into ws k-slices of vpl groups of 256 elements, the groups
// of the slices interleaved (slice sw has groups sw, sw + ws, ...); team warp w
// works on slice w % ws of rows w / ws + q * rg (q < rw) of each of its pages,
// so ws * rg warps of the team are active and each lane keeps vpl 16-byte
// vectors of the input in registers.
//
// tc = 1 selects the tensor-core page instead (mv_shape_tc): the columns are cut
// into nch chunks of kc; a page holds up to TC_ROWS rows of one chunk, loaded by
// TMA in the 128-byte swizzle, and all NCW warps work on every page, each on its
// own kc / NCW columns of the chunk.
// Geometry families of the CUDA-core kernel instantiations (see geo_has): hidden
// 2048 with inter 8192 ((2, 8) and (4, 2)), hidden 4096 with inter 14336 ((4, 4)
// and (4, 1)).
enum : int { GEO_ALL = 0, GEO_2048 = 1, GEO_4096 = 2, GEO_BCC = 3 };  // GEO_BCC: two sequences on CUDA-core pages

struct MvShape {
    int32_t K, ws, vpl, rpp, rg, rw, teams, tc, kc, nch;
    // per consumer warp w (CUDA-core pages): its team, k-slice and row group, and
    // the arrivals it makes on a page's release (0: no work in its team); set by
    // mv_shape so that the kernel divides by none of the runtime sizes
    uint8_t w_team[NCW], w_sw[NCW], w_rgi[NCW], w_arrive[NCW];
};
constexpr int TC_ROWS = 8;        // rows of a tensor-core page (the MMA's n)
constexpr int TC_MATS_PER_LAYER = 7;  // wq, wk, wv, wo, wg, wu, wd: the matrices whose pages may be tensor-core pages

// One entry of an SM's producer list, in consumption order: a weight page
// (src, bytes), or an attention item whose K/V pages depend on pos and are
// expanded on the device (src then packs layer << 32 | kv_head << 16 | split).
struct PDesc {
    unsigned long long src;
    uint32_t bytes;
    uint16_t instr;  // index of the instruction the page belongs to
    uint16_t kind;   // PD_WEIGHTS or PD_ATTN
};
enum : uint16_t { PD_WEIGHTS = 0, PD_ATTN = 1, PD_TMA_W = 2 };
// PD_ATTN: src = (sequence << 48) | (layer << 32) | (KV head << 16) | split.
// PD_TMA_W: a tensor-core weight page, src = (tensor map index << 40) |
// (64-column block of its chunk << 32) | first row.
// Map index of matrix m (0..6: wq, wk, wv, wo, wg, wu, wd) of layer l, or of the
// LM head (l = L, m = 0), for a page of nr rows (1..TC_ROWS): every box height has
// its own map, so that a page never loads rows of another SM's range.
__host__ __device__ inline uint32_t wmap_index(int l, int m, int nr) {
    return (uint32_t(l) * TC_MATS_PER_LAYER + uint32_t(m)) * TC_ROWS + uint32_t(nr - 1);
}


// A TMA tensor map (CUtensorMap: 128 opaque bytes, 64-byte aligned), kept as
// bytes here so that this header needs no driver API types.
struct alignas(64) TensorMap {
    unsigned char bytes[128];
};
// KV tensor maps of the per-warp attention variant: the K or V cache as a 2-D
// tensor (head_dim, L * n_kv * max_seq rows), 64-dim boxes with the 128-byte
// swizzle; box height a whole page of positions or one 16-position tile.
enum : int { TM_K_PAGE = 0, TM_K_TILE = 1, TM_V_PAGE = 2, TM_V_TILE = 3, TM_COUNT = 4 };
constexpr int ATT_TILE = 16;  // positions per tensor-core attention tile

struct LayerW {
    const uint16_t *attn_norm, *wq, *wk, *wv, *wo, *mlp_norm, *wg, *wu, *wd;
};
constexpr int SMEM_LAYERS = 32;  // layers whose weight pointers the megakernel keeps in shared memory

// Counters, each on its own 128-byte line.
constexpr int CTR_STRIDE = 32;  // uint32 per counter slot
struct CtrLayout {
    // per layer: qkv, attn, oproj, gateup, down; then the LM-head ticket
    static __host__ __device__ inline int qkv(int l) { return l * 5 + 0; }
    static __host__ __device__ inline int attn(int l) { return l * 5 + 1; }
    static __host__ __device__ inline int oproj(int l) { return l * 5 + 2; }
    static __host__ __device__ inline int gateup(int l) { return l * 5 + 3; }
    static __host__ __device__ inline int down(int l) { return l * 5 + 4; }
    static __host__ __device__ inline int lm_ticket(int L) { return L * 5; }
    static __host__ __device__ inline int count(int L, int) { return L * 5 + 1; }
};

struct KParams {
    TensorMap kv_maps[TM_COUNT];  // (TM_*) used by the per-warp attention variant
    // schedule
    const Instr *instrs;      // [nsm][max_instr]
    const int32_t *n_instr;   // [nsm]
    const PDesc *pdesc;       // producer lists of all SMs, back to back
    const int32_t *pdesc_off; // [nsm + 1] start of each SM's list
    int32_t max_instr;
    int32_t nsm;
    // model
    const LayerW *layers;     // [L] (device)
    const uint16_t *embed, *lm_head, *final_norm;
    uint16_t *k_cache, *v_cache;
    const float2 *rope_cs;    // [max_seq][hd/2] (cos, sin)
    int32_t L, H, nq, nkv, hd, I, V, max_seq;
    float eps;
    int32_t attn_splits;
    int32_t attn_flash;       // kernel variant: per-warp softmax in attention (long items)
    MvShape mv_h, mv_q, mv_i; // input widths hidden, n_q*hd, inter
    const TensorMap *wmaps;   // weight tensor maps of tensor-core pages (wmap_index), global memory, or null
    // Batched handles (the tensor-core kernel): nb sequences, each with its own KV
    // cache and position; tagged activations, argmax keys, tokens and logits are
    // laid out sequence after sequence. Single-sequence handles: nb = 1 and entry 0.
    int32_t nb;
    int32_t pos_b[MAX_B];     // each sequence's position in the launch's first step
    uint16_t *kc_b[MAX_B], *vc_b[MAX_B];
    const TensorMap *kvmaps_b; // [nb][TM_COUNT] each sequence's KV tensor maps (global memory; the per-warp attention)
    // Activations between instructions, as tagged words: (tag << 32) | fp32 bits,
    // stored and loaded as single 8-byte accesses. A reader takes a word only
    // when its tag is the one of the current step and layer (tag_of), so the
    // data itself tells the reader it is ready.
    uint64_t *t_qkv;          // [nq*hd + 2*nkv*hd] QKV projection (before RoPE)
    uint64_t *t_part;         // [nq][splits][hd + 4] attention partials: o (unnormalised), m, l
    uint64_t *t_o;            // [nq*hd] attention output, the splits merged
    uint64_t *t_xmid;         // [H] residual stream after the O projection
    uint64_t *t_act;          // [I] silu(gate) * up
    uint64_t *t_xout;         // [H] residual stream after the down projection
    unsigned long long *lm_keys; // [nsm]
    uint32_t *ctr;            // counters, CTR_STRIDE apart
    int32_t *status;          // sticky status word
    int32_t *token_out;       // [1] library copy of the last next token
    uint64_t *t_token;        // each step's next token as a tagged word (tag = the step's epoch), read by the
                              // next step of the same launch
    // step
    int32_t token;            // used when token_dev is null
    const int32_t *token_dev;
    int32_t pos;              // position of the launch's first step (step i decodes at pos + i)
    uint32_t epoch;           // 1-based step count since the last reset, of the launch's first step
    int32_t n_steps;          // greedy steps in this launch, each fed the previous one's token
    int32_t *tokens_dev;      // [n_steps] every step's next token (multi-step launches), or null
    float *logits;            // [n_steps][V] or null
    int32_t *next_token_dev;  // or null
    unsigned long long timeout_ns;
    uint32_t l2_prefetch;     // pages the producer may prefetch into L2 beyond its ring
    uint32_t evict_first;     // weight pages loaded with an L2 evict-first hint
    uint32_t producer_sleep_ns; // back-off of the producer while the ring is full
    int32_t geo;                // GEO_*: the kernel instantiation whose geometries this handle uses
    uint32_t consumer_sleep_ns; // back-off of a consumer warp whose page is not issued yet
    uint32_t max_inflight;    // pages issued but not yet landed, at most (NPAGES: only the ring bounds it)
    // optional globaltimer trace, [nsm][max_instr][TRACE_WORDS]: consumer begin,
    // dependency met + input loaded, pages done, end; producer first and last issue;
    // first page in hand, compute on the pages done; for attention also the end
    // of the scores, softmax and P.V phases of its last block, and the partials written
    unsigned long long *trace;
    // optional page trace, [nsm][PTRACE_PAGES][3]: producer issue, consumer start,
    // release, indexed by page number modulo PTRACE_PAGES
    unsigned long long *ptrace;
    // debug builds (LL_DEBUG_CHECKS): first out-of-range access seen, else null
    long long *dbg;
};

// Host-side launchers (defined in the .cu files).
int launch_megakernel(const KParams &p, void *stream, int smem_bytes);
int megakernel_smem_bytes();
int megakernel_prepare(int smem_bytes);

struct ChainBufs {
    const LayerW *host_layers;  // [L], host memory
    float *x, *h, *qkv, *part, *o, *gate, *up, *act, *logits;
    int32_t splits;
    // the (cos, sin) row of the step's position, or null to take row pos of the
    // KParams table (rope_cs)
    const float2 *rope_row;
};

// KV splits per KV head: about ATTN_SPLIT_POS cached positions each at the
// longest context (tuning knob LL_ATTN_SPLIT_POS, read here), at most one
// attention item per SM. Every entry point picks its splits with this.
int attn_splits(int max_seq, int n_kv_heads, int nsm, int nb = 1);
int launch_chain_step(const KParams &p, const ChainBufs &b, void *stream);
// Final RMSNorm of the residual row x, LM head into logits (all vocab rows) and
// greedy argmax into next_dev and p.token_out (p.status on all-NaN logits):
// per-operation kernels of the chain, for the last position of a prefill.
int launch_chain_head(const KParams &p, const float *x, float *h, float *logits, int32_t *next_dev, void *stream);

// ---- prefill (prefill.cu): the prompt's positions through the model at once,
// every projection a tcgen05 GEMM. Buffers for up to n_alloc tokens.
struct PrefillBufs {
    static constexpr int T = 3;          // bf16 terms of an activation matrix
    int n_alloc = 0;
    float *x = nullptr;                  // [n][H] residual stream
    uint16_t *h[T] = {};                 // [n][H] normed input, as T bf16 terms
    float *qkv = nullptr;                // [n][qd + 2 kd]
    uint16_t *o[T] = {};                 // [n][qd] attention output, T terms
    uint16_t *a[T] = {};                 // [n][I] silu(gate) * up, T terms (gate and up: one GEMM)
    float *hrow = nullptr, *logits = nullptr;       // [H], [V]: the last position's head
    TensorMap m_h[T], m_o[T], m_a[T];    // A operands (activations), boxes of 128 rows x 64 columns
    std::vector<TensorMap> m_w;          // B operands: [L][7] wq, wk, wv, wo, wg, wu, wd, boxes of 128 rows x 64
    TensorMap m_k, m_v;                  // the K and V caches as [L * n_kv * max_seq][hd], boxes of 16 rows x 64
    void *mem = nullptr;
};
// Allocates (or grows) the buffers and encodes the maps; false on failure.
bool prefill_prepare(const KParams &p, const LayerW *host_layers, int n, PrefillBufs &b);
void prefill_release(PrefillBufs &b);
int launch_prefill(const KParams &p, const LayerW *host_layers, PrefillBufs &b, const int32_t *tokens_dev, int n,
                   int pos0, float *logits, int32_t *next_dev, void *stream);

// Host-side schedule construction (schedule.cpp). nb sequences (attention items
// per sequence); an SM's LM-head rows in instructions of at most lm_rows rows.
void build_schedule(int L, int H, int qd, int kd, int I, int V, int nkv, int nsm, int splits,
                    std::vector<std::vector<Instr>> &lists, int nb = 1, int lm_rows = 1 << 30);
// lane_floats: the most input floats a lane may hold per team copy of the
// input (16 or 32); more allows more teams (pages in progress at once).
bool mv_shape(int K, MvShape &m, int lane_floats = 16);
// CUDA-core geometry for width K with two sequences' inputs held per lane (at
// most 16 floats of each): only (vpl, rw) = (2, 8) or (2, 2); false otherwise.
bool mv_shape_bc(int K, MvShape &m);
// The tensor-core geometry for width K, if the kernel has it (K a multiple of
// 1024, at most 16384): chunks of 2048 columns (1024 when 2048 does not divide K),
// pages of TC_ROWS rows of one chunk, every warp on a whole number of 64-column
// blocks of each.
bool mv_shape_tc(int K, MvShape &m);
void build_pdesc(const std::vector<std::vector<Instr>> &lists, const std::vector<LayerW> &layers,
                 const uint16_t *lm_head, int H, int qd, int kd, int I, const MvShape &mh, const MvShape &mq,
                 const MvShape &mi, std::vector<PDesc> &out, std::vector<int32_t> &off);

}  // namespace ll
