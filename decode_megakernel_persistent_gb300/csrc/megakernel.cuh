// megakernel.cuh -- the persistent decode megakernel for sm_103a (device code;
// mk_cuda_cores.cu and mk_tensor_cores.cu instantiate its kernels).
//
// One decode step of a Llama-style decoder runs as one launch of this kernel,
// one block per SM, following the page "Hazy Research Llama-3.2-1B Megakernel"
// (Chinese write-up, w2o.qhhnjy.cn/html/17f999973.html):
//   * instruction interpreter: every SM walks its own static instruction list,
//     built on the host once and reused for every token (paragraphs on the
//     interpreter and the instruction list);
//   * shared-memory pages: the block's shared memory is a ring of pages; a
//     producer warp fills them with the bytes the next instructions will read,
//     so loads for later instructions start while earlier ones still wait
//     (paragraph on paging);
//   * dependencies in global memory instead of kernel boundaries (paragraph on
//     the counter system). The page counts finished instructions in integers;
//     here the data carries its own readiness: every activation an instruction
//     hands to another SM is stored as one 8-byte word holding the fp32 value
//     and a tag (step, layer), and the reader polls the words it needs until
//     their tags are current. Nothing is fenced or counted per instruction, and
//     the reader's wait and its input load are the same reads.
//
// GB300 choices (not from the page): pages are filled with one-dimensional
// bulk async copies (cp.async.bulk) completing on mbarriers; matrix-vector
// products run on CUDA cores with the input vector held in registers; the
// split-KV attention partials are merged by the attention SMs of each KV head
// between them, so the O projection reads one merged vector; the greedy argmax
// is reduced by the last SM to finish (an atomic ticket). Every wait is bounded
// by a time limit.
#pragma once
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "ll_internal.h"

namespace ll {
// Everything here has internal linkage: two translation units instantiate it.
namespace {

// ---------------------------------------------------------------------------------
// PTX helpers

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
                 : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive_cnt(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ bool mbar_test(uint64_t *bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return done != 0;
}

__device__ __forceinline__ void bulk_load(void *dst, const void *src, uint32_t bytes, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_addr(dst)),
        "l"(src), "r"(bytes), "r"(smem_addr(bar))
        : "memory");
}

__device__ __forceinline__ uint64_t gtimer() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ int32_t ld_relaxed(const int32_t *p) {
    int32_t v;
    asm volatile("ld.relaxed.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// Tagged activation words: (tag << 32) | fp32 bits, one 8-byte access each, so a
// reader that sees the tag also sees the value stored with it.
__device__ __forceinline__ void st_tag(uint64_t *p, float v, uint32_t tag) {
    const uint64_t w = (static_cast<uint64_t>(tag) << 32) | __float_as_uint(v);
    asm volatile("st.relaxed.gpu.global.b64 [%0], %1;" ::"l"(p), "l"(w) : "memory");
}

__device__ __forceinline__ uint64_t ld_tag(const uint64_t *p) {
    uint64_t w;
    asm volatile("ld.relaxed.gpu.global.b64 %0, [%1];" : "=l"(w) : "l"(p) : "memory");
    return w;
}

__device__ __forceinline__ void ld_tag2(const uint64_t *p, uint64_t &a, uint64_t &b) {
    asm volatile("ld.relaxed.gpu.global.v2.b64 {%0, %1}, [%2];" : "=l"(a), "=l"(b) : "l"(p) : "memory");
}

__device__ __forceinline__ float tag_val(uint64_t w) { return __uint_as_float(static_cast<uint32_t>(w)); }
__device__ __forceinline__ bool tag_ok(uint64_t w, uint32_t tag) { return static_cast<uint32_t>(w >> 32) == tag; }

__device__ __forceinline__ void consumer_sync() {
    asm volatile("bar.sync 1, %0;" ::"n"(NCT) : "memory");
}

// Consumer barrier that also returns, to every consumer thread alike, whether
// any of them passed true: failures leave an instruction together, so no
// thread is left waiting at a later barrier for threads that have gone.
__device__ __forceinline__ bool consumer_any(bool v) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\tbar.red.or.pred q, 1, %2, p;\n\tselp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"(static_cast<uint32_t>(v)), "n"(NCT)
        : "memory");
    return r != 0;
}

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
    return v;
}

__device__ __forceinline__ float4 lds_f4(uint32_t addr) {
    float4 v;
    asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(addr));
    return v;
}

__device__ __forceinline__ float bf_lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf_hi(uint32_t u) { return __uint_as_float(u & 0xffff0000u); }
__device__ __forceinline__ float bf16_to_f(uint16_t b) { return __uint_as_float(uint32_t(b) << 16); }

// fp32 -> bf16, round to nearest even (finite inputs; NaN maps to a quiet NaN).
__device__ __forceinline__ uint16_t f_to_bf16(float f) {
    uint32_t u = __float_as_uint(f);
    if ((u & 0x7f800000u) == 0x7f800000u && (u & 0x007fffffu)) return 0x7fc0;
    u += 0x7fffu + ((u >> 16) & 1u);
    return uint16_t(u >> 16);
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

__device__ __forceinline__ unsigned long long warp_max_u64(unsigned long long v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        unsigned long long w = __shfl_xor_sync(0xffffffffu, v, o);
        v = w > v ? w : v;
    }
    return v;
}

// Order-preserving key for the argmax: larger value first, then lower index.
__device__ __forceinline__ unsigned long long argmax_key(float v, int idx) {
    uint32_t u = __float_as_uint(v);
    uint32_t ord = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
    return (static_cast<unsigned long long>(ord) << 32) | (0xffffffffu - static_cast<uint32_t>(idx));
}

// ---------------------------------------------------------------------------------
// Shared memory

// One merge slot of the attention warps (per-warp softmax): o for up to 512
// (query head, dim) pairs (n_q / n_kv * head_dim <= 512), then m and l of up to
// 8 heads.
constexpr int AT_SLOT = 512 + 2 * MAX_GQA;

struct alignas(16) Smem {
    union {
        float xin[XIN_FLOATS];  // O-projection input: the merged attention output; also the
                                // attention P.V partials of the P.V warps
        float kpart[KPART_FLOATS];  // the current matrix-vector instruction's (row, k-slice) partial sums
        struct {                                // attention, block-wide softmax per page:
            float ared_lo[ATT_WARPS * 4 * 64];  // P.V partials of four heads of 64 dims
            float sc[MAX_GQA][132];             // scores of up to 129 positions
            float pt[132][MAX_GQA];             // their probabilities, position-major
        };
        uint4 qf[MAX_HD / 16][32];           // attention, per-warp softmax: query MMA A fragments (hi, lo rows)
        float ared[NCW / 2][AT_SLOT];        // attention, per-warp softmax: (o, m, l) of warps being merged
    };
    uint64_t full[NPAGES];   // page filled (tx bytes landed)
    uint64_t empty[NPAGES];  // page released by the consumers: NCW arrivals in all per page
    int32_t pcnt[NPAGES];    // warps done with the page in the slot
    volatile uint32_t slot_page[NPAGES];  // page number the producer last put in the slot
    float qr[MAX_GQA][MAX_HD];  // the attention item's rotated, scaled query heads
    alignas(16) uint16_t knew[MAX_HD];
    alignas(16) uint16_t vnew[MAX_HD];
    alignas(16) uint16_t zrow[64];  // zeros: the K / V row read for positions past a page's end
    float m_run[MAX_GQA], l_run[MAX_GQA], alpha[MAX_GQA];
    float xown[XOWN_MAX];  // this SM's rows of the residual stream (the O and down rows)
    LayerW lw[SMEM_LAYERS];  // weight pointers of the first SMEM_LAYERS layers, copied at kernel start
    float nred[NCW];
    unsigned long long kred[NCW];
    int32_t token;
    // the consumers' current step of a multi-step launch
    uint32_t c_epoch;          // its epoch (tags)
    int32_t c_pos;             // its position
    float *c_logits;           // where its logits go, or null
    volatile int32_t tok_step; // steps whose input token the consumers hold (the producer's gate)
    int32_t start_status;
    volatile int32_t flag;
    volatile int32_t abort;
    // the tensor-core kernel (batched handles; one sequence is a batch of one)
    float bacc[BACC_FLOATS];        // row results of the current instruction, [row][sequence]
    float bxown[MAX_B][XOWN_MAX];   // each sequence's residual rows this SM owns
    float nredb[NCW][MAX_B];        // per warp and sequence: sum of squares of the input
    int32_t btoken[MAX_B];          // each sequence's input token of the current step
    int32_t bpos[MAX_B];            // and its position
};

static_assert(offsetof(Smem, xin) % 16 == 0 && offsetof(Smem, pt) % 16 == 0, "alignment");
static_assert(ATT_WARPS * 4 * MAX_HD <= XIN_FLOATS, "P.V partials of four heads fit the O input space");

constexpr int SMEM_BYTES = NPAGES * PAGE_BYTES + static_cast<int>(sizeof(Smem));

// ---------------------------------------------------------------------------------
// Bounded waits. A wait that runs past p.timeout_ns records LL_ERR_DEP_TIMEOUT in
// the status word; any wait that sees a nonzero status gives up as well.

__device__ __forceinline__ void raise_status(const KParams &p, Smem &s, int32_t code) {
    atomicCAS(p.status, 0, code);
    s.abort = 1;
}

__device__ __forceinline__ void trace_put(const KParams &p, int ii, int k) {
    if (p.trace) p.trace[(size_t(blockIdx.x) * p.max_instr + ii) * TRACE_WORDS + k] = gtimer();
}

// Debug builds check every shared- and global-memory index of the hot paths;
// the first out-of-range access is recorded in p.dbg (code, sm, thread, index,
// limit) and skipped. Release builds compile the checks away.
#ifdef LL_DEBUG_CHECKS
__device__ __noinline__ bool ll_check_fail(const KParams &p, int code, long long a, long long b) {
    if (p.dbg && atomicCAS(reinterpret_cast<unsigned long long *>(p.dbg), 0ull, 1ull) == 0ull) {
        p.dbg[1] = code;
        p.dbg[2] = blockIdx.x;
        p.dbg[3] = threadIdx.x;
        p.dbg[4] = a;
        p.dbg[5] = b;
    }
    return false;
}
#define LL_OK_IDX(code, idx, lim) \
    ((static_cast<long long>(idx) >= 0 && static_cast<long long>(idx) < static_cast<long long>(lim)) || \
     ll_check_fail(p, (code), static_cast<long long>(idx), static_cast<long long>(lim)))
#else
#define LL_OK_IDX(code, idx, lim) true
#endif

__device__ __forceinline__ void ptrace_put(const KParams &p, uint32_t page, int k) {
    if (p.ptrace) p.ptrace[(size_t(blockIdx.x) * PTRACE_PAGES + page % PTRACE_PAGES) * 3 + k] = gtimer();
}

__device__ bool wait_mbar(const KParams &p, Smem &s, uint64_t *bar, uint32_t parity) {
    if (mbar_test(bar, parity)) return true;
    const uint64_t t0 = gtimer();
    for (uint32_t it = 1;; ++it) {
        if (mbar_test(bar, parity)) return true;
        if ((it & 15u) == 0) {
            if (s.abort) return false;
            if (gtimer() - t0 > p.timeout_ns) {
                raise_status(p, s, LL_ERR_DEP_TIMEOUT);
                return false;
            }
        }
    }
}

// Consumer wait for page number `page` in its ring slot. A phase-parity wait is
// only unambiguous once the slot holds this page (consumers of different teams
// may run more than one ring lap apart), so first wait until the producer has
// put the page in the slot, then for its bytes.
__device__ bool wait_page(const KParams &p, Smem &s, uint32_t page) {
    const uint32_t slot = page % NPAGES;
    if (s.slot_page[slot] != page) {
        const uint64_t t0 = gtimer();
        for (uint32_t it = 1; s.slot_page[slot] != page; ++it) {
            // back off, so that the warps working on landed pages keep the issue slots
            if (p.consumer_sleep_ns) __nanosleep(p.consumer_sleep_ns);
            if ((it & 15u) == 0) {
                if (s.abort) return false;
                if (gtimer() - t0 > p.timeout_ns) {
                    raise_status(p, s, LL_ERR_DEP_TIMEOUT);
                    return false;
                }
            }
        }
    }
    return wait_mbar(p, s, &s.full[slot], (page / NPAGES) & 1u);
}

// Tag of the words an instruction of `layer` writes in the current step (never 0
// for a live step, so cleared memory never passes).
//
// Each tagged buffer is rewritten once per layer, and no untagged signal orders
// a rewrite after the last read of the previous layer's words; the data flow
// does. Every SM's QKV rows feed some attention item, every attention item
// feeds every O-projection SM (the full merged vector), every O-projection SM
// feeds every gate/up SM (the full residual), every gate/up SM feeds every
// down SM (the full act vector), and every down SM feeds every QKV SM (the full
// residual). So before any SM can write a buffer for layer l + 1 it has waited,
// through this chain, on words that every reader of the layer-l words produced
// after reading them:
//   qkv    (QKV -> attention):  rewrite needs x_out(l) from all down SMs;
//   part   (attention -> merge): rewrite needs qkv(l+1), i.e. x_out(l), i.e. o(l) merged;
//   o      (merge -> O):        rewrite needs qkv(l+1), i.e. every O-projection SM done;
//   x_mid  (O -> gate/up):      rewrite needs o(l+1), i.e. every gate/up SM done with layer l;
//   act    (gate/up -> down):   rewrite needs x_mid(l+1), i.e. every down SM done with layer l;
//   x_out  (down -> QKV, LM):   rewrite needs act(l+1), i.e. every QKV SM done with layer l
// The LM head reads the last layer's x_out before any write of the next step:
// that step runs in a later launch, or, in a multi-step launch, only once its
// input token is published, which the last SM does after every SM has finished
// its LM head (and so every read of this step's words).
__device__ __forceinline__ uint32_t tag_of(const KParams &p, const Smem &s, int layer) {
    return s.c_epoch * static_cast<uint32_t>(p.L + 1) + static_cast<uint32_t>(layer) + 1u;
}

// The tag an instruction writes: its layer's, or 0 when its completion has been
// removed from the schedule (fault injection), so that its readers time out.
__device__ __forceinline__ uint32_t write_tag(const KParams &p, const Smem &s, const Instr &ins) {
    return ins.sig_ctr >= 0 ? tag_of(p, s, ins.layer) : 0u;
}

// Bounded polling of tagged words: called after a round of loads found a stale
// tag (it > 0; round 0 only starts the clock). Returns true once the thread
// should give up: another thread or block failed (s.abort, the status word), or
// the time limit passed (then it records LL_ERR_DEP_TIMEOUT). The caller's
// threads learn of it through consumer_any(s.abort).
__device__ __forceinline__ bool poll_give_up(const KParams &p, Smem &s, uint32_t it, uint64_t &t0) {
    if (it == 0) {
        t0 = gtimer();
        return false;
    }
    if (s.abort) return true;
    if ((it & 7u) == 0) {
        if (ld_relaxed(p.status) != 0) {
            s.abort = 1;
            return true;
        }
        if (gtimer() - t0 > p.timeout_ns) {
            raise_status(p, s, LL_ERR_DEP_TIMEOUT);
            return true;
        }
    }
    return false;
}

// Load N tagged words with `load(w)` (which fills every entry; entries it does
// not need it sets to a word with the expected tag) until all carry `tag`. Every
// round reloads them all: whichever word turns current first, the thread sees
// the rest within the same round trip.
template <int N, class Load>
__device__ __forceinline__ void poll_words(const KParams &p, Smem &s, uint64_t (&w)[N], uint32_t tag, Load load) {
    uint64_t t0 = 0;
    for (uint32_t it = 0;; ++it) {
        load(w);
        bool ok = true;
#pragma unroll
        for (int i = 0; i < N; i++) ok = ok && tag_ok(w[i], tag);
        if (ok || poll_give_up(p, s, it, t0)) return;
    }
}

// Instruction boundary: every consumer thread is done with the shared-memory
// scratch of this instruction before the next one writes it; reports, to all
// alike, a failure any thread saw.
__device__ __forceinline__ bool instr_sync(Smem &s) { return !consumer_any(s.abort); }

// ---------------------------------------------------------------------------------
// Matrix-vector instructions: the rows an SM owns are cut into segments (one per
// weight matrix) and each segment into pages of at most mv.rpp whole rows.

enum OutKind : int { OUT_QKV, OUT_RESID, OUT_GATE, OUT_UP, OUT_LOGITS };

struct Seg {
    const uint16_t *w;  // row 0 of the matrix
    int32_t row0;       // first row of the segment within the matrix
    int32_t nrows;
    int32_t out0;       // output index of matrix row 0
    int32_t kind;
};

__device__ __forceinline__ const MvShape &mv_of(const KParams &p, int op) {
    return op == OP_OPROJ ? p.mv_q : (op == OP_DOWN ? p.mv_i : p.mv_h);
}

// A layer's weight pointers, from shared memory for the first SMEM_LAYERS layers:
// an instruction then does not start with a dependent global load.
__device__ __forceinline__ const LayerW &layer_w(const KParams &p, const Smem &s, int l) {
    return l < SMEM_LAYERS ? s.lw[l] : p.layers[l];
}

__device__ int mv_segments(const KParams &p, const Smem &s, const Instr &ins, Seg *seg) {
    const LayerW *lw = ins.op == OP_LMHEAD ? nullptr : &layer_w(p, s, ins.layer);
    const int r0 = ins.r0, r1 = ins.r1;
    int n = 0;
    switch (ins.op) {
        case OP_QKV: {
            const int qd = p.nq * p.hd, kd = p.nkv * p.hd;
            const int b[4] = {0, qd, qd + kd, qd + 2 * kd};
            const uint16_t *m[3] = {lw->wq, lw->wk, lw->wv};
            for (int i = 0; i < 3; i++) {
                int a = max(r0, b[i]), e = min(r1, b[i + 1]);
                if (a < e) seg[n++] = Seg{m[i], a - b[i], e - a, b[i], OUT_QKV};
            }
            break;
        }
        case OP_OPROJ:
            if (r0 < r1) seg[n++] = Seg{lw->wo, r0, r1 - r0, 0, OUT_RESID};
            break;
        case OP_GATEUP:
            if (r0 < r1) {
                seg[n++] = Seg{lw->wg, r0, r1 - r0, 0, OUT_GATE};
                seg[n++] = Seg{lw->wu, r0, r1 - r0, 0, OUT_UP};
            }
            break;
        case OP_DOWN:
            if (r0 < r1) seg[n++] = Seg{lw->wd, r0, r1 - r0, 0, OUT_RESID};
            break;
        case OP_LMHEAD:
            if (r0 < r1) seg[n++] = Seg{p.lm_head, r0, r1 - r0, 0, OUT_LOGITS};
            break;
        default:
            break;
    }
    return n;
}

// Attention: cached positions [c0, c1) of split c, PP of them per page (K then V).
__device__ __forceinline__ void attn_range(const KParams &p, int pos, int c, int &c0, int &c1) {
    const long long S = p.attn_splits;
    c0 = static_cast<int>((static_cast<long long>(c) * pos) / S);
    c1 = static_cast<int>((static_cast<long long>(c + 1) * pos) / S);
}

__device__ __forceinline__ int attn_pp(const KParams &p) { return PAGE_BYTES / (4 * p.hd); }

// Lane-held input vector: element (j*32*ws + sw*32 + lane)*8 + e sits in xr[j*8+e]
// (the 256-element groups of the k-slices interleaved: measured 657.7 -> 652.7 us
// per 1B step against slice-contiguous groups).
// The RMSNorm gain of a normed instruction (QKV, gate/up, LM head), or null.
__device__ __forceinline__ const uint16_t *norm_gain(const KParams &p, const Smem &s, const Instr &ins) {
    switch (ins.op) {
        case OP_QKV: return layer_w(p, s, ins.layer).attn_norm;
        case OP_GATEUP: return layer_w(p, s, ins.layer).mlp_norm;
        case OP_LMHEAD: return p.final_norm;
        default: return nullptr;
    }
}

// Gains are weights: a lane's slice is fetched before the dependency wait.
template <int VPL>
__device__ __forceinline__ void load_gain(const KParams &p, const Smem &s, const Instr &ins, const MvShape &mv, uint4 (&gv)[VPL]) {
    const uint16_t *gain = norm_gain(p, s, ins);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int sw = mv.w_sw[warp];
#pragma unroll
    for (int j = 0; j < VPL; j++)
        gv[j] = gain ? __ldg(reinterpret_cast<const uint4 *>(gain) + j * 32 * mv.ws + sw * 32 + lane) : make_uint4(0, 0, 0, 0);
}

// The instruction's input vector into registers (layout above), RMS-normed for
// QKV, gate/up and the LM head. Inputs that fit s.xin are staged there first, so
// that each tagged word is read once per block whatever the number of teams;
// wider ones (the down projection's) are read straight into the lanes. Returns
// false, in every consumer thread alike, if a wait failed.
// kbase: where the instruction's (row, k-slice) partials start in s.kpart (which
// shares space with s.xin). Past the staged input when they fit there (one
// sequence): a warp may then write its partials while others still read their
// input, with no barrier between; else 0, behind a barrier.
template <int VPL, bool BAT = false>
__device__ bool load_input(const KParams &p, Smem &s, const Instr &ins, const MvShape &mv,
                           float (&xr)[VPL * 8], const uint4 (&gv)[VPL], int &kbase, int b = 0) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, tid = threadIdx.x;
    const int sw = mv.w_sw[warp];
    const bool normed = norm_gain(p, s, ins) != nullptr;
    const uint64_t *src = nullptr;
    uint32_t tag = 0;
    switch (ins.op) {
        case OP_QKV:
            if (ins.layer > 0) {
                src = p.t_xout;
                tag = tag_of(p, s, ins.layer - 1);
            }
            break;
        case OP_GATEUP: src = p.t_xmid; tag = tag_of(p, s, ins.layer); break;
        case OP_LMHEAD: src = p.t_xout; tag = tag_of(p, s, p.L - 1); break;
        case OP_DOWN: src = p.t_act; tag = tag_of(p, s, ins.layer); break;
        case OP_OPROJ: src = p.t_o; tag = tag_of(p, s, ins.layer); break;
        default: break;
    }
    if (BAT && src) src += size_t(b) * size_t(mv.K);  // sequence b's words (laid out sequence after sequence)
    const bool staged = src && mv.K <= XIN_FLOATS;
    const int need = (ins.op == OP_GATEUP ? 2 : 1) * (ins.r1 - ins.r0) * mv.ws;
    const bool apart = !BAT && staged && mv.K + need <= KPART_FLOATS;
    kbase = apart ? mv.K : 0;
    // per-warp sums of squares; a batch's sequences each have their own, so
    // that the next sequence's input may be taken in while this one's are read
    auto nred = [&](int w) -> float & { return BAT ? s.nredb[w][b] : s.nred[w]; };
    if (staged) {
        constexpr int PAIRS = XIN_FLOATS / (2 * NCT);
        uint64_t w[2 * PAIRS];
        const int K = mv.K;
        poll_words(p, s, w, tag, [&](uint64_t (&ww)[2 * PAIRS]) {
#pragma unroll
            for (int k = 0; k < PAIRS; k++) {
                const int i = (tid + k * NCT) * 2;
                if (i < K) ld_tag2(src + i, ww[2 * k], ww[2 * k + 1]);
                else ww[2 * k] = ww[2 * k + 1] = static_cast<uint64_t>(tag) << 32;
            }
        });
        // one sequence: a normed input's sum of squares is taken here, each
        // element once, so that the barrier publishing s.xin publishes the warps'
        // sums as well (a batch's sequences take theirs after it, measured faster
        // for two sequences: 772 against 750 us per step)
        float ss = 0.f;
#pragma unroll
        for (int k = 0; k < PAIRS; k++) {
            const int i = (tid + k * NCT) * 2;
            if (i < K) {
                const float a = tag_val(w[2 * k]), c = tag_val(w[2 * k + 1]);
                s.xin[i] = a;
                s.xin[i + 1] = c;
                if (!BAT) ss = fmaf(c, c, fmaf(a, a, ss));
            }
        }
        if (!BAT && normed) {
            ss = warp_sum(ss);
            if (lane == 0) nred(warp) = ss;
        }
    }
    if (staged && consumer_any(s.abort)) return false;  // also publishes s.xin (and the sums)
#pragma unroll
    for (int j = 0; j < VPL; j++) {
        const int v = j * 32 * mv.ws + sw * 32 + lane;
        if (!LL_OK_IDX(11, v * 8 + 8, mv.K + 1)) continue;
        if (staged) {
            const float4 a = *reinterpret_cast<const float4 *>(&s.xin[v * 8]);
            const float4 b = *reinterpret_cast<const float4 *>(&s.xin[v * 8 + 4]);
            xr[j * 8 + 0] = a.x; xr[j * 8 + 1] = a.y; xr[j * 8 + 2] = a.z; xr[j * 8 + 3] = a.w;
            xr[j * 8 + 4] = b.x; xr[j * 8 + 5] = b.y; xr[j * 8 + 6] = b.z; xr[j * 8 + 7] = b.w;
        } else if (!src) {  // layer 0: the token's embedding row
            const uint4 u = __ldg(reinterpret_cast<const uint4 *>(p.embed + size_t(BAT ? s.btoken[b] : s.token) * p.H) + v);
            xr[j * 8 + 0] = bf_lo(u.x); xr[j * 8 + 1] = bf_hi(u.x);
            xr[j * 8 + 2] = bf_lo(u.y); xr[j * 8 + 3] = bf_hi(u.y);
            xr[j * 8 + 4] = bf_lo(u.z); xr[j * 8 + 5] = bf_hi(u.z);
            xr[j * 8 + 6] = bf_lo(u.w); xr[j * 8 + 7] = bf_hi(u.w);
        } else {
            // wide input, one 256-element group per j: the warp reads it with
            // coalesced loads (lane l takes words 2l + 64r, r < 4) and turns it
            // into the lane layout through its own 256 floats of s.xin
            uint64_t w[8];
            const uint64_t *at = src + size_t(j * 32 * mv.ws + sw * 32) * 8;
            poll_words(p, s, w, tag, [&](uint64_t (&ww)[8]) {
#pragma unroll
                for (int r = 0; r < 4; r++) ld_tag2(at + 64 * r + 2 * lane, ww[2 * r], ww[2 * r + 1]);
            });
            float *tw = s.xin + warp * 256;
#pragma unroll
            for (int r = 0; r < 4; r++)
                *reinterpret_cast<float2 *>(tw + 64 * r + 2 * lane) = make_float2(tag_val(w[2 * r]), tag_val(w[2 * r + 1]));
            __syncwarp();
            const float4 a = *reinterpret_cast<const float4 *>(tw + 8 * lane);
            const float4 b = *reinterpret_cast<const float4 *>(tw + 8 * lane + 4);
            xr[j * 8 + 0] = a.x; xr[j * 8 + 1] = a.y; xr[j * 8 + 2] = a.z; xr[j * 8 + 3] = a.w;
            xr[j * 8 + 4] = b.x; xr[j * 8 + 5] = b.y; xr[j * 8 + 6] = b.z; xr[j * 8 + 7] = b.w;
            __syncwarp();
        }
    }
    // (wide inputs: also every warp is done with its part of s.xin, which
    // s.kpart overlaps, before any team writes partial sums)
    if (!staged && src && consumer_any(s.abort)) return false;
    // s.kpart shares space with s.xin: unless the partials go past the input,
    // every warp holds its input before any team writes partial sums (a batch's
    // normed input: the norm's own barrier below)
    if (staged && !apart && !(BAT && normed)) consumer_sync();
    if (!normed) return true;
    // RMSNorm. Staged (one sequence): the NCW warps' sums of their staged
    // elements. Else the warps w < ws together hold every element once in their
    // registers.
    float tot = 0.f;
    if (staged && !BAT) {
#pragma unroll
        for (int w = 0; w < NCW; w++) tot += nred(w);
    } else {
        float ss = 0.f;
#pragma unroll
        for (int e = 0; e < VPL * 8; e++) ss = fmaf(xr[e], xr[e], ss);
        ss = warp_sum(ss);
        if (lane == 0 && warp < mv.ws) nred(warp) = ss;
        consumer_sync();
        for (int w = 0; w < mv.ws; w++) tot += nred(w);
    }
    const float r = 1.0f / sqrtf(tot / static_cast<float>(mv.K) + p.eps);
#pragma unroll
    for (int j = 0; j < VPL; j++) {
        const uint32_t g[4] = {gv[j].x, gv[j].y, gv[j].z, gv[j].w};
#pragma unroll
        for (int q = 0; q < 4; q++) {
            xr[j * 8 + 2 * q] = xr[j * 8 + 2 * q] * r * bf_lo(g[q]);
            xr[j * 8 + 2 * q + 1] = xr[j * 8 + 2 * q + 1] * r * bf_hi(g[q]);
        }
    }
    return true;
}

// Sum R per-lane values across the warp so that the lanes of group
// q = lane / (32 / R) end up holding the full sum of value q.
template <int R>
__device__ __forceinline__ float transpose_reduce(float (&v)[R]) {
    const int lane = threadIdx.x & 31;
    int n = R;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        if (n > 1) {
            const bool upper = (lane & off) != 0;
            const int half = n / 2;
#pragma unroll
            for (int i = 0; i < R / 2; i++) {
                if (i < half) {
                    const float send = upper ? v[i] : v[i + half];
                    const float keep = upper ? v[i + half] : v[i];
                    v[i] = keep + __shfl_xor_sync(0xffffffffu, send, off);
                }
            }
            n = half;
        } else {
            v[0] += __shfl_xor_sync(0xffffffffu, v[0], off);
        }
    }
    return v[0];
}

// The epilogue of a matrix-vector instruction, once every (row, k-slice)
// partial is in s.kpart: each row's sum of its ws k-slices, stored as q/k/v, the
// residual stream, silu(gate) * up, or the logits and each thread's running
// argmax. Inlined: as a called function it made the 1B step ~7 % slower (measured).
__device__ __forceinline__ void mv_store(const KParams &p, Smem &s, const Instr &ins, int ii, int ws, int kbase,
                                         float &best, int &best_idx) {
    const int tid = threadIdx.x;
    const int nrows = ins.r1 - ins.r0;
    const int r0 = ins.r0;
    const uint32_t wtag = write_tag(p, s, ins);
    struct RowSum {  // the row's k-slices, summed in k-slice order
        const float *kp;
        int ws, kbase;
        __device__ float operator[](int t) const {
            float y = 0.f;
            for (int w = 0; w < ws; w++)
                if (LL_OK_IDX(3, kbase + t * ws + w, KPART_FLOATS)) y += kp[kbase + t * ws + w];
            return y;
        }
    } acc{s.kpart, ws, kbase};
    switch (ins.op) {
        case OP_QKV:
            for (int t = tid; t < nrows; t += NCT)
                if (LL_OK_IDX(5, r0 + t, (p.nq + 2 * p.nkv) * p.hd) && LL_OK_IDX(6, t, ACC_FLOATS))
                    st_tag(p.t_qkv + r0 + t, acc[t], wtag);
            break;
        case OP_OPROJ:
        case OP_DOWN: {
            // this SM owns rows [r0, r1) of the residual stream in both projections
            // (same row split), so it keeps them in shared memory across layers
            const bool from_embed = ins.op == OP_OPROJ && ins.layer == 0;
            for (int t = tid; t < nrows; t += NCT) {
                const int row = r0 + t;
                if (!LL_OK_IDX(7, row, p.H) || !LL_OK_IDX(20, t, XOWN_MAX)) continue;
                const float base = from_embed ? bf16_to_f(p.embed[size_t(s.token) * p.H + row]) : s.xown[t];
                const float v = base + acc[t];
                s.xown[t] = v;
                st_tag((ins.op == OP_OPROJ ? p.t_xmid : p.t_xout) + row, v, wtag);
            }
            break;
        }
        case OP_GATEUP:
            for (int t = tid; t < nrows; t += NCT) {
                const float g = acc[t];
                if (LL_OK_IDX(8, r0 + t, p.I) && LL_OK_IDX(9, nrows + t, ACC_FLOATS))
                    st_tag(p.t_act + r0 + t, g / (1.0f + expf(-g)) * acc[nrows + t], wtag);
            }
            break;
        default:  // OP_LMHEAD: logits out, running argmax per thread (rows ascend per thread)
            for (int t = tid; t < nrows; t += NCT) {
                const float y = acc[t];
                if (s.c_logits && LL_OK_IDX(10, r0 + t, p.V)) s.c_logits[r0 + t] = y;
                if (y > best) {
                    best = y;
                    best_idx = r0 + t;
                }
            }
            break;
    }
    if (threadIdx.x == 0) trace_put(p, ii, 2);
}


template <int VPL, int RW>
__device__ bool mv_instr(const KParams &p, Smem &s, uint8_t *pages, const Instr &ins, int ii, uint32_t &cpage,
                         float &best, int &best_idx) {
    const MvShape &mv = mv_of(p, ins.op);
    Seg seg[3];
    const int nseg = mv_segments(p, s, ins, seg);
    if (nseg == 0) return true;  // no rows here: nothing to read or wait for
    uint4 gv[VPL];
    load_gain<VPL>(p, s, ins, mv, gv);
    float xr[VPL * 8];
    int kbase;
    if (!load_input<VPL>(p, s, ins, mv, xr, gv, kbase)) return false;
    if (threadIdx.x == 0) trace_put(p, ii, 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, tid = threadIdx.x;
    const int team = mv.w_team[warp], sw = mv.w_sw[warp], rgi = mv.w_rgi[warp];
    // a page is released by the NCW arrivals its team's working warps make in all
    const uint32_t my_arrivals = mv.w_arrive[warp];  // 0: no work in this warp
    const uint32_t row_bytes = uint32_t(mv.K) * 2;
    const int nrows = ins.r1 - ins.r0;
    constexpr int GROUP = 32 / RW;  // lanes that end up holding one row's sum
    constexpr int QB = (RW < 4 / VPL) ? RW : (4 / VPL > 0 ? 4 / VPL : 1);  // rows loaded together
    bool bad = false;  // a page wait failed: walk on without work, leave together below

    for (int si = 0; si < nseg; si++) {
        const Seg sg = seg[si];
        // where the segment's rows land among the instruction's rows (s.kpart)
        const int acc0 = sg.kind == OUT_QKV ? sg.out0 + sg.row0 - ins.r0 : (sg.kind == OUT_UP ? nrows : 0);
        for (int pr = 0; pr < sg.nrows; pr += mv.rpp) {
            const int nr = min(mv.rpp, sg.nrows - pr);
            const uint32_t slot = cpage % NPAGES;
            const uint32_t this_page = cpage++;
            if (int(this_page & uint32_t(mv.teams - 1)) != team || my_arrivals == 0) continue;
            if (bad || !wait_page(p, s, this_page)) {
                bad = true;
                continue;
            }
            if ((sw | rgi) == 0 && lane == 0) {  // the team's first warp
                ptrace_put(p, this_page, 1);
                if (si == 0 && pr == 0) trace_put(p, ii, 6);
            }
            const uint32_t page = smem_addr(pages) + slot * PAGE_BYTES + (sw * 32 + lane) * 16;
            float v[RW];
#pragma unroll
            for (int q0 = 0; q0 < RW; q0 += QB) {
                // rows past nr hold stale bytes; their sums are never used
                uint4 wv[QB][VPL];
#pragma unroll
                for (int qq = 0; qq < QB; qq++) {
                    const uint32_t wrow = page + uint32_t(rgi + (q0 + qq) * mv.rg) * row_bytes;
#pragma unroll
                    for (int j = 0; j < VPL; j++) {
                        const uint32_t at = wrow + uint32_t(j * 32 * mv.ws) * 16u;
                        if (LL_OK_IDX(1, (at + 16) - smem_addr(pages), NPAGES * PAGE_BYTES + 1))
                            wv[qq][j] = lds128(at);
                        else
                            wv[qq][j] = make_uint4(0, 0, 0, 0);
                    }
                }
#pragma unroll
                for (int qq = 0; qq < QB; qq++) {
                    float a0 = 0.f, a1 = 0.f;
#pragma unroll
                    for (int j = 0; j < VPL; j++) {
                        const uint4 w = wv[qq][j];
                        a0 = fmaf(bf_lo(w.x), xr[j * 8 + 0], a0);
                        a1 = fmaf(bf_hi(w.x), xr[j * 8 + 1], a1);
                        a0 = fmaf(bf_lo(w.y), xr[j * 8 + 2], a0);
                        a1 = fmaf(bf_hi(w.y), xr[j * 8 + 3], a1);
                        a0 = fmaf(bf_lo(w.z), xr[j * 8 + 4], a0);
                        a1 = fmaf(bf_hi(w.z), xr[j * 8 + 5], a1);
                        a0 = fmaf(bf_lo(w.w), xr[j * 8 + 6], a0);
                        a1 = fmaf(bf_hi(w.w), xr[j * 8 + 7], a1);
                    }
                    v[q0 + qq] = a0 + a1;
                }
            }
            const float sum = transpose_reduce<RW>(v);
            // this warp's k-slice of its rows; the page goes back to the producer
            // as soon as every active warp has read it (the k-slices are summed
            // once per instruction, below)
            const int r = rgi + (lane / GROUP) * mv.rg;
            if ((lane % GROUP) == 0 && r < nr && LL_OK_IDX(2, kbase + (acc0 + pr + r) * mv.ws + sw, KPART_FLOATS))
                s.kpart[kbase + (acc0 + pr + r) * mv.ws + sw] = sum;
            __syncwarp();
            if (lane == 0) {
                ptrace_put(p, this_page, 2);
                mbar_arrive_cnt(&s.empty[slot], my_arrivals);
            }
        }
    }
    if (tid == 0) trace_put(p, ii, 7);
    if (consumer_any(bad)) return false;  // else every k-slice of every row is in s.kpart
    mv_store(p, s, ins, ii, mv.ws, kbase, best, best_idx);
    return true;
}

// ---------------------------------------------------------------------------------
// Two sequences on CUDA-core pages (batched handles whose input widths allow it,
// see mv_shape_bc): every page is read once and multiplied with both sequences'
// inputs, each lane holding 2 x VPL x 8 input floats. The (row, k-slice,
// sequence) partials go to s.kpart; the epilogue sums them per (row, sequence)
// and stores each sequence's outputs as the batched kernel lays them out.
constexpr int NBC = 2;  // sequences of the batched CUDA-core kernel

__device__ __forceinline__ void mv_store_bc(const KParams &p, Smem &s, const Instr &ins, int ii, int ws, float &best,
                                            int &best_idx) {
    const int tid = threadIdx.x;
    const int nrows = ins.r1 - ins.r0, r0 = ins.r0;
    const uint32_t wtag = write_tag(p, s, ins);
    auto sum = [&](int t, int b) {  // row t's k-slices of sequence b, in k-slice order
        float y = 0.f;
        for (int w = 0; w < ws; w++)
            if (LL_OK_IDX(3, (t * ws + w) * NBC + b, KPART_FLOATS)) y += s.kpart[(t * ws + w) * NBC + b];
        return y;
    };
    const int qkvd = (p.nq + 2 * p.nkv) * p.hd;
    // idx % NBC == tid % NBC: each thread keeps to one sequence (lm_finish_b's argmax)
    for (int idx = tid; idx < nrows * NBC; idx += NCT) {
        const int t = idx / NBC, b = idx % NBC;
        const float y = sum(t, b);
        switch (ins.op) {
            case OP_QKV:
                if (LL_OK_IDX(5, r0 + t, qkvd)) st_tag(p.t_qkv + size_t(b) * qkvd + r0 + t, y, wtag);
                break;
            case OP_OPROJ:
            case OP_DOWN: {
                const int row = r0 + t;
                if (!LL_OK_IDX(7, row, p.H) || !LL_OK_IDX(20, t, XOWN_MAX)) break;
                const float base = ins.op == OP_OPROJ && ins.layer == 0
                                       ? bf16_to_f(p.embed[size_t(s.btoken[b]) * p.H + row])
                                       : s.bxown[b][t];
                const float v = base + y;
                s.bxown[b][t] = v;
                st_tag((ins.op == OP_OPROJ ? p.t_xmid : p.t_xout) + size_t(b) * p.H + row, v, wtag);
                break;
            }
            case OP_GATEUP: {
                const float u = sum(nrows + t, b);
                if (LL_OK_IDX(8, r0 + t, p.I)) st_tag(p.t_act + size_t(b) * p.I + r0 + t, y / (1.0f + expf(-y)) * u, wtag);
                break;
            }
            default:  // OP_LMHEAD: rows ascend per thread
                if (s.c_logits && LL_OK_IDX(10, r0 + t, p.V)) s.c_logits[size_t(b) * p.V + r0 + t] = y;
                if (y > best) {
                    best = y;
                    best_idx = r0 + t;
                }
                break;
        }
    }
}

template <int VPL, int RW>
__device__ bool mv_instr_bc(const KParams &p, Smem &s, uint8_t *pages, const Instr &ins, int ii, uint32_t &cpage,
                            float &best, int &best_idx) {
    const MvShape &mv = mv_of(p, ins.op);
    Seg seg[3];
    const int nseg = mv_segments(p, s, ins, seg);
    if (nseg == 0) return true;
    float xr[NBC][VPL * 8];
#pragma unroll
    for (int b = 0; b < NBC; b++) {
        uint4 gv[VPL];
        load_gain<VPL>(p, s, ins, mv, gv);
        int kbase;  // (0: a batched input is always behind a barrier)
        if (!load_input<VPL, true>(p, s, ins, mv, xr[b], gv, kbase, b)) return false;
    }
    if (threadIdx.x == 0) trace_put(p, ii, 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, tid = threadIdx.x;
    const int team = mv.w_team[warp], sw = mv.w_sw[warp], rgi = mv.w_rgi[warp];
    const uint32_t my_arrivals = mv.w_arrive[warp];
    const uint32_t row_bytes = uint32_t(mv.K) * 2;
    const int nrows = ins.r1 - ins.r0;
    constexpr int GROUP = 32 / RW;
    constexpr int QB = (RW < 4 / VPL) ? RW : (4 / VPL > 0 ? 4 / VPL : 1);
    bool bad = false;
    for (int si = 0; si < nseg; si++) {
        const Seg sg = seg[si];
        const int acc0 = sg.kind == OUT_QKV ? sg.out0 + sg.row0 - ins.r0 : (sg.kind == OUT_UP ? nrows : 0);
        for (int pr = 0; pr < sg.nrows; pr += mv.rpp) {
            const int nr = min(mv.rpp, sg.nrows - pr);
            const uint32_t slot = cpage % NPAGES;
            const uint32_t this_page = cpage++;
            if (int(this_page & uint32_t(mv.teams - 1)) != team || my_arrivals == 0) continue;
            if (bad || !wait_page(p, s, this_page)) {
                bad = true;
                continue;
            }
            if ((sw | rgi) == 0 && lane == 0) {
                ptrace_put(p, this_page, 1);
                if (si == 0 && pr == 0) trace_put(p, ii, 6);
            }
            const uint32_t page = smem_addr(pages) + slot * PAGE_BYTES + (sw * 32 + lane) * 16;
            float v[NBC][RW];
#pragma unroll
            for (int q0 = 0; q0 < RW; q0 += QB) {
                uint4 wv[QB][VPL];
#pragma unroll
                for (int qq = 0; qq < QB; qq++) {
                    const uint32_t wrow = page + uint32_t(rgi + (q0 + qq) * mv.rg) * row_bytes;
#pragma unroll
                    for (int j = 0; j < VPL; j++) {
                        const uint32_t at = wrow + uint32_t(j * 32 * mv.ws) * 16u;
                        if (LL_OK_IDX(1, (at + 16) - smem_addr(pages), NPAGES * PAGE_BYTES + 1))
                            wv[qq][j] = lds128(at);
                        else
                            wv[qq][j] = make_uint4(0, 0, 0, 0);
                    }
                }
#pragma unroll
                for (int b = 0; b < NBC; b++)
#pragma unroll
                    for (int qq = 0; qq < QB; qq++) {
                        float a0 = 0.f, a1 = 0.f;
#pragma unroll
                        for (int j = 0; j < VPL; j++) {
                            const uint4 w = wv[qq][j];
                            a0 = fmaf(bf_lo(w.x), xr[b][j * 8 + 0], a0);
                            a1 = fmaf(bf_hi(w.x), xr[b][j * 8 + 1], a1);
                            a0 = fmaf(bf_lo(w.y), xr[b][j * 8 + 2], a0);
                            a1 = fmaf(bf_hi(w.y), xr[b][j * 8 + 3], a1);
                            a0 = fmaf(bf_lo(w.z), xr[b][j * 8 + 4], a0);
                            a1 = fmaf(bf_hi(w.z), xr[b][j * 8 + 5], a1);
                            a0 = fmaf(bf_lo(w.w), xr[b][j * 8 + 6], a0);
                            a1 = fmaf(bf_hi(w.w), xr[b][j * 8 + 7], a1);
                        }
                        v[b][q0 + qq] = a0 + a1;
                    }
            }
            const int r = rgi + (lane / GROUP) * mv.rg;
#pragma unroll
            for (int b = 0; b < NBC; b++) {
                const float sum = transpose_reduce<RW>(v[b]);
                const int k = ((acc0 + pr + r) * mv.ws + sw) * NBC + b;
                if ((lane % GROUP) == 0 && r < nr && LL_OK_IDX(2, k, KPART_FLOATS)) s.kpart[k] = sum;
            }
            __syncwarp();
            if (lane == 0) {
                ptrace_put(p, this_page, 2);
                mbar_arrive_cnt(&s.empty[slot], my_arrivals);
            }
        }
    }
    if (tid == 0) trace_put(p, ii, 7);
    if (consumer_any(bad)) return false;
    mv_store_bc(p, s, ins, ii, mv.ws, best, best_idx);
    return true;
}

// Greedy argmax across the grid: every SM publishes its best key, the last SM to
// arrive reduces them and writes the token.
__device__ void lm_finish(const KParams &p, Smem &s, float best, int best_idx) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, tid = threadIdx.x;
    unsigned long long key = best_idx >= 0 ? argmax_key(best, best_idx) : 0ull;
    key = warp_max_u64(key);
    if (lane == 0) s.kred[warp] = key;
    consumer_sync();
    if (tid == 0) {
        unsigned long long k = 0;
        for (int w = 0; w < NCW; w++) k = s.kred[w] > k ? s.kred[w] : k;
        p.lm_keys[blockIdx.x] = k;
        __threadfence();
        const uint32_t old = atomicAdd(p.ctr + size_t(CtrLayout::lm_ticket(p.L)) * CTR_STRIDE, 1u);
        s.flag = (old + 1u == s.c_epoch * static_cast<uint32_t>(p.nsm)) ? 1 : 0;
        __threadfence();
    }
    consumer_sync();
    if (!s.flag) return;
    unsigned long long k = 0;
    for (int i = tid; i < p.nsm; i += NCT) {
        unsigned long long v = __ldcg(p.lm_keys + i);
        k = v > k ? v : k;
    }
    k = warp_max_u64(k);
    if (lane == 0) s.kred[warp] = k;
    consumer_sync();
    if (tid == 0) {
        unsigned long long m = 0;
        for (int w = 0; w < NCW; w++) m = s.kred[w] > m ? s.kred[w] : m;
        // no SM found an orderable logit (all NaN): there is no greedy token
        if (m == 0) atomicCAS(p.status, 0, LL_ERR_NUMERIC);
        const int32_t tok = static_cast<int32_t>(0xffffffffu - static_cast<uint32_t>(m & 0xffffffffu));
        p.token_out[0] = tok;
        if (p.tokens_dev) p.tokens_dev[s.c_epoch - p.epoch] = tok;
        else if (p.next_token_dev) *p.next_token_dev = tok;
        if (p.n_steps > 1) {
            // the next step of this launch waits for this word (its tag is this step's epoch)
            __threadfence();
            const uint64_t w = (static_cast<uint64_t>(s.c_epoch) << 32) | static_cast<uint32_t>(tok);
            asm volatile("st.relaxed.gpu.global.b64 [%0], %1;" ::"l"(p.t_token), "l"(w) : "memory");
        }
    }
}

// ---------------------------------------------------------------------------------
// Attention instruction: one KV head g, one split c of the cached positions
// 0..pos-1; the split that owns position pos also takes in the new k, v and
// writes them to the cache. Its unnormalised partial (o, m, l) per query head
// goes to global memory, and the O projection merges the splits when it loads
// its input, so no instruction waits for a separate merge.

// DL consecutive bf16 from shared memory, widened.
template <int DL>
__device__ __forceinline__ void lds_bf16(uint32_t addr, float (&out)[DL]) {
    if constexpr (DL == 2) {
        uint32_t u;
        asm volatile("ld.shared.u32 %0, [%1];" : "=r"(u) : "r"(addr));
        out[0] = bf_lo(u);
        out[1] = bf_hi(u);
    } else {
        static_assert(DL == 4, "head_dim 64 or 128");
        uint32_t u0, u1;
        asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(u0), "=r"(u1) : "r"(addr));
        out[0] = bf_lo(u0);
        out[1] = bf_hi(u0);
        out[2] = bf_lo(u1);
        out[3] = bf_hi(u1);
    }
}

// Attention over one page. Lane l of a warp owns dims [l*DL, l*DL + DL) of the
// query heads, taken four at a time from the rotated queries in shared memory; a
// position's K or V row is then one 128/256-byte conflict-free access per warp.
// Scores: warp w takes positions w, w + NCW, ... and reduces its per-head partial
// dots across lanes. Softmax statistics: warp h for head h. P.V: ATT_WARPS warps
// split the positions, each reading a position's probabilities with one
// broadcast load, and their partial sums are added through shared memory by one
// thread per (head, dim).
template <int DL>
__device__ void attn_block(const KParams &p, Smem &s, const uint16_t *K, const uint16_t *Vv, int n,
                           bool with_new, float &oacc, int G, int ii) {
    constexpr int hd = DL * 32, GP = 4;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int nt = n + (with_new ? 1 : 0);
    const uint32_t kbase = K ? smem_addr(K) : 0u, vbase = Vv ? smem_addr(Vv) : 0u;
    const uint32_t knew = smem_addr(s.knew), vnew = smem_addr(s.vnew);
    // scores
    for (int h0 = 0; h0 < G; h0 += GP) {
        float q[GP][DL];
#pragma unroll
        for (int h = 0; h < GP; h++)
#pragma unroll
            for (int e = 0; e < DL; e++) q[h][e] = h0 + h < G ? s.qr[h0 + h][lane * DL + e] : 0.f;
        for (int j = warp; j < nt; j += NCW) {
            const uint32_t kr = (j < n ? kbase + uint32_t(j) * (hd * 2) : knew) + lane * (DL * 2);
            float k[DL];
            lds_bf16<DL>(kr, k);
            float v[GP];
#pragma unroll
            for (int h = 0; h < GP; h++) {
                float a = 0.f;
#pragma unroll
                for (int e = 0; e < DL; e++) a = fmaf(q[h][e], k[e], a);
                v[h] = a;
            }
            const float sum = transpose_reduce<GP>(v);
            const int h = h0 + lane / (32 / GP);
            if ((lane % (32 / GP)) == 0 && h < G && LL_OK_IDX(14, j, 132)) s.sc[h][j] = sum;
        }
    }
    consumer_sync();
    if (tid == 0) trace_put(p, ii, 8);
    // online softmax statistics: warp h handles head h; probabilities go out position-major
    if (warp < G) {
        const int h = warp;
        float mx = -INFINITY;
        for (int j = lane; j < nt; j += 32) mx = fmaxf(mx, s.sc[h][j]);
        mx = warp_max(mx);
        const float m_old = s.m_run[h];
        const float m_new = fmaxf(m_old, mx);
        float sum = 0.f;
        for (int j = lane; j < nt; j += 32) {
            const float e = expf(s.sc[h][j] - m_new);
            s.pt[j][h] = e;
            sum += e;
        }
        sum = warp_sum(sum);
        if (lane == 0) {
            const float a = (m_old == -INFINITY) ? 0.f : expf(m_old - m_new);
            s.alpha[h] = a;
            s.l_run[h] = s.l_run[h] * a + sum;
            s.m_run[h] = m_new;
        }
    }
    consumer_sync();
    if (tid == 0) trace_put(p, ii, 9);
    // P.V partial sums of ATT_WARPS warps, four heads at a time. The partials of a
    // group use ATT_WARPS*4*hd floats from the start of the union: with 64-dim heads
    // that ends below sc/pt (up to eight heads, two groups); with 128-dim heads
    // (at most four, one group) it overlaps them, read by then.
    float *ared = s.xin;
    for (int h0 = 0; h0 < G; h0 += GP) {
        float o[GP][DL];
#pragma unroll
        for (int h = 0; h < GP; h++)
#pragma unroll
            for (int e = 0; e < DL; e++) o[h][e] = 0.f;
        if (warp < ATT_WARPS) {
            for (int j = warp; j < nt; j += ATT_WARPS) {
                const uint32_t vr = (j < n ? vbase + uint32_t(j) * (hd * 2) : vnew) + lane * (DL * 2);
                float v[DL];
                lds_bf16<DL>(vr, v);
                const float4 t4 = lds_f4(smem_addr(&s.pt[j][h0]));
                const float pj[GP] = {t4.x, t4.y, t4.z, t4.w};
#pragma unroll
                for (int h = 0; h < GP; h++)
#pragma unroll
                    for (int e = 0; e < DL; e++) o[h][e] = fmaf(pj[h], v[e], o[h][e]);
            }
        }
        consumer_sync();  // s.pt read (128-dim heads) and the previous group's partials summed
        if (warp < ATT_WARPS) {
#pragma unroll
            for (int h = 0; h < GP; h++)
                if (h0 + h < G)
#pragma unroll
                    for (int e = 0; e < DL; e++) ared[(warp * GP + h) * hd + lane * DL + e] = o[h][e];
        }
        consumer_sync();
        const int t = tid - h0 * hd;
        if (t >= 0 && t < GP * hd && tid < G * hd) {
            float a = 0.f;
#pragma unroll
            for (int w = 0; w < ATT_WARPS; w++) a += ared[w * GP * hd + t];
            oacc = oacc * s.alpha[h0 + t / hd] + a;
        }
    }
    if (tid == 0) trace_put(p, ii, 10);
}

// The S splits of KV head g merge their partials between them: split c takes
// outputs [c*G*hd/S, (c+1)*G*hd/S) of the group's G*hd, for each
//   o = sum_c' exp(m_c' - M) o_c' / sum_c' exp(m_c' - M) l_c',  M = max_c' m_c',
// and stores them, tagged, to t_o. The threads of one output split the S partials
// between them (a running maximum each), then one thread combines theirs through
// shared memory.
// (b: the sequence of a batched handle, whose partials and outputs lie b whole
// buffers further on)
__device__ bool merge_splits(const KParams &p, Smem &s, int g, int c, int G, int hd, uint32_t tag, uint32_t wtag,
                             int b = 0) {
    const int S = p.attn_splits, GH = G * hd, stride = hd + 4, tid = threadIdx.x;
    const int v0 = static_cast<int>(static_cast<long long>(c) * GH / S);
    const int nv = static_cast<int>(static_cast<long long>(c + 1) * GH / S) - v0;
    if (nv <= 0) return true;  // uniform: no outputs for this split
    const int T = NCT / nv;    // threads per output (nv <= 512)
    const int v = tid % nv, j = tid / nv;
    float M = -INFINITY, L = 0.f, O = 0.f;
    if (j < T) {
        const int h = (v0 + v) / hd, d = (v0 + v) % hd;
        const uint64_t *base = p.t_part + size_t(b) * p.nq * S * stride + size_t(g * G + h) * S * stride;
        for (int cb = j; cb < S; cb += 4 * T) {
            uint64_t w[12];  // per split: m, l, o[d]
            poll_words(p, s, w, tag, [&](uint64_t (&ww)[12]) {
#pragma unroll
                for (int k = 0; k < 4; k++) {
                    const int c2 = cb + k * T;
                    if (c2 < S) {
                        const uint64_t *pc = base + size_t(c2) * stride;
                        ld_tag2(pc + hd, ww[3 * k], ww[3 * k + 1]);
                        ww[3 * k + 2] = ld_tag(pc + d);
                    } else {
                        ww[3 * k] = ww[3 * k + 1] = ww[3 * k + 2] = static_cast<uint64_t>(tag) << 32;
                    }
                }
            });
#pragma unroll
            for (int k = 0; k < 4; k++) {
                if (cb + k * T >= S) break;
                const float m = tag_val(w[3 * k]);
                if (m == -INFINITY) continue;  // a split with no positions
                const float Mn = fmaxf(M, m);
                const float a = (M == -INFINITY) ? 0.f : expf(M - Mn), b = expf(m - Mn);
                L = L * a + tag_val(w[3 * k + 1]) * b;
                O = O * a + tag_val(w[3 * k + 2]) * b;
                M = Mn;
            }
        }
        s.xin[(j * nv + v) * 3 + 0] = M;
        s.xin[(j * nv + v) * 3 + 1] = L;
        s.xin[(j * nv + v) * 3 + 2] = O;
    }
    if (consumer_any(s.abort)) return false;
    if (tid < nv) {
        float Mx = -INFINITY;
        for (int jj = 0; jj < T; jj++) Mx = fmaxf(Mx, s.xin[(jj * nv + tid) * 3]);
        float Ls = 0.f, Os = 0.f;
        for (int jj = 0; jj < T; jj++) {
            const float m = s.xin[(jj * nv + tid) * 3];
            if (m == -INFINITY) continue;
            const float b = expf(m - Mx);
            Ls = fmaf(s.xin[(jj * nv + tid) * 3 + 1], b, Ls);
            Os = fmaf(s.xin[(jj * nv + tid) * 3 + 2], b, Os);
        }
        st_tag(p.t_o + size_t(b) * p.nq * hd + size_t(g) * GH + v0 + tid, Os / Ls, wtag);
    }
    return true;
}

// BATCH: the item belongs to sequence ins.sub of a batched handle (its q/k/v,
// position, caches, partials and output); otherwise to the one sequence.
template <int DL, bool BATCH = false>
__device__ bool attn_item(const KParams &p, Smem &s, uint8_t *pages, const Instr &ins, int ii, uint32_t &cpage) {
    const int g = ins.r0, c = ins.r1, S = p.attn_splits, l = ins.layer;
    constexpr int hd = DL * 32, half = hd / 2;
    const int G = p.nq / p.nkv, tid = threadIdx.x;
    const int qd = p.nq * hd, kd = p.nkv * hd;
    const bool owner = c == S - 1;  // this split owns position pos
    const float scale = 1.0f / sqrtf(static_cast<float>(hd));
    const int b = BATCH ? int(ins.sub) : 0;
    const int pos = BATCH ? s.bpos[b] : s.c_pos;
    const float2 *cs = p.rope_cs + size_t(pos) * half;
    const uint64_t *qkv_b = p.t_qkv + size_t(b) * (qd + 2 * kd);
    const uint32_t tag = tag_of(p, s, l);
    // the group's query heads with RoPE ("rotate half") applied, pre-scaled by
    // 1/sqrt(hd); the owner also rotates the new key and takes the new value
    {
        const uint64_t *qh = qkv_b + size_t(g * G) * hd;
        const uint64_t *kh = qkv_b + qd + size_t(g) * hd;
        const uint64_t *vh = qkv_b + qd + kd + size_t(g) * hd;
        const bool has_q = tid < G * hd, has_k = owner && tid < half, has_v = owner && tid < hd;
        const int h = tid / hd, d = tid % hd, i = d < half ? d : d - half;
        uint64_t w[5];
        poll_words(p, s, w, tag, [&](uint64_t (&ww)[5]) {
            const uint64_t ok = static_cast<uint64_t>(tag) << 32;
            ww[0] = has_q ? ld_tag(qh + size_t(h) * hd + i) : ok;
            ww[1] = has_q ? ld_tag(qh + size_t(h) * hd + i + half) : ok;
            ww[2] = has_k ? ld_tag(kh + tid) : ok;
            ww[3] = has_k ? ld_tag(kh + tid + half) : ok;
            ww[4] = has_v ? ld_tag(vh + tid) : ok;
        });
        if (has_q) {
            const float a = tag_val(w[0]), b = tag_val(w[1]);
            const float2 r = cs[i];
            s.qr[h][d] = (d < half ? a * r.x - b * r.y : a * r.y + b * r.x) * scale;
        }
        if (has_k) {
            const float a = tag_val(w[2]), b = tag_val(w[3]);
            const float2 r = cs[tid];
            s.knew[tid] = f_to_bf16(a * r.x - b * r.y);
            s.knew[tid + half] = f_to_bf16(a * r.y + b * r.x);
        }
        if (has_v) s.vnew[tid] = f_to_bf16(tag_val(w[4]));
    }
    if (tid < G) {
        s.m_run[tid] = -INFINITY;
        s.l_run[tid] = 0.f;
    }
    if (consumer_any(s.abort)) return false;
    if (tid == 0) trace_put(p, ii, 1);
    if (owner) {
        const size_t at = ((size_t(l) * p.nkv + g) * size_t(p.max_seq) + pos) * hd;
        uint16_t *kc = BATCH ? p.kc_b[b] : p.k_cache, *vc = BATCH ? p.vc_b[b] : p.v_cache;
        if (LL_OK_IDX(16, at + hd, size_t(p.L) * p.nkv * p.max_seq * hd + 1))
            for (int d = tid; d < hd; d += NCT) {
                kc[at + d] = s.knew[d];
                vc[at + d] = s.vnew[d];
            }
    }
    float oacc = 0.f;
    int c0, c1;
    attn_range(p, pos, c, c0, c1);
    const int PP = attn_pp(p);
    for (int p0 = c0; p0 < c1; p0 += PP) {
        const int n = min(PP, c1 - p0);
        const bool with_new = owner && p0 + PP >= c1;  // fold the new token into the last page
        const uint32_t slot = cpage % NPAGES;
        if (consumer_any(!wait_page(p, s, cpage))) return false;
        if (tid == 0) {
            ptrace_put(p, cpage, 1);
            trace_put(p, ii, 6);
        }
        const uint16_t *pg = reinterpret_cast<const uint16_t *>(pages + size_t(slot) * PAGE_BYTES);
        attn_block<DL>(p, s, pg, pg + PAGE_BYTES / 4, n, with_new, oacc, G, ii);  // V at half a page
        if (tid == 0) {
            ptrace_put(p, cpage, 2);
            mbar_arrive_cnt(&s.empty[slot], NCW);
        }
        ++cpage;
    }
    if (owner && c0 == c1) attn_block<DL>(p, s, nullptr, nullptr, 0, true, oacc, G, ii);
    if (tid == 0) trace_put(p, ii, 7);

    // partials: part[(qhead * S + c) * (hd + 4) + {d, hd: m, hd+1: l}]
    const int stride = hd + 4;
    uint64_t *part_b = p.t_part + size_t(b) * p.nq * S * stride;
    const uint32_t wtag = write_tag(p, s, ins);
    if (tid < G * hd) {
        const int h = tid / hd, d = tid % hd;
        st_tag(part_b + (size_t(g * G + h) * S + c) * stride + d, oacc, wtag);
    }
    if (tid < G && LL_OK_IDX(17, (size_t(g * G + tid) * S + c) * stride + hd + 1, size_t(p.nq) * S * stride)) {
        st_tag(part_b + (size_t(g * G + tid) * S + c) * stride + hd, s.m_run[tid], wtag);
        st_tag(part_b + (size_t(g * G + tid) * S + c) * stride + hd + 1, s.l_run[tid], wtag);
    }
    if (tid == 0) trace_put(p, ii, 2);
    return merge_splits(p, s, g, c, G, hd, tag, wtag, b);
}

// D += A * B, m16n8k16, all four A registers: a0 = (row g, cols 2t, 2t + 1),
// a1 = (row g + 8, same cols), a2 = (row g, cols 2t + 8, 2t + 9), a3 = (row g + 8,
// those cols); D: d0, d1 = row g, d2, d3 = row g + 8, at cols 2t, 2t + 1.
__device__ __forceinline__ void mma_16816(float (&d)[4], const uint4 &a, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a.x), "r"(a.y), "r"(a.z), "r"(a.w), "r"(b0), "r"(b1));
}

// Four 8 x 8 bf16 matrices from shared memory: lanes 8i .. 8i + 7 give the row
// addresses of matrix i; lane (g, t) receives row g, elements 2t, 2t + 1 of each
// (trans: element rows 2t, 2t + 1 of column g).
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t (&r)[4]) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}

__device__ __forceinline__ uint4 lds_v4(uint32_t addr) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
    return v;
}

// x as the sum of two bf16 terms (hi, lo), so that a bf16 tensor-core product of
// x with a bf16 operand keeps ~16 bits of x.
__device__ __forceinline__ void split_bf16(float x, uint16_t &hi, uint16_t &lo) {
    hi = f_to_bf16(x);
    lo = f_to_bf16(x - bf16_to_f(hi));
}

// Attention over one page of n cached positions plus, if with_new, the new token
// (s.knew, s.vnew) at index n, for the group's G query heads, as flash decoding:
// the calling warp takes the 16-position tiles tile0, tile0 + tstride, ... for the
// 64 dims of its dim group dg, keeping its own running softmax across tiles and
// pages. The page holds K at kbase and V at vbase, each as [dim half][position]
// [64 dims] with PP positions per half and 128-byte rows in the TMA 128-byte
// swizzle (16-byte chunk c of row r at chunk c ^ (r % 8)), so that the eight rows
// of an ldmatrix fall in eight different bank groups.
//
// The query heads' fp32 values enter as two bf16 terms, hi in rows 0..7 of the
// A operand and lo in rows 8..15 (a KV head has at most 8 query heads), so one
// m16n8k16 product yields both and their sum is exact to ~16 bits. Per tile:
// S = Q K^T (K^T as B, 8 positions per product, two products per k-step); the
// tile's maximum and sum over the 4 lanes of each head; P = exp(S - m), split the
// same way into hi (rows g) and lo (rows g + 8), which in the m16n8k16 layouts
// is already the A fragment of O += P V (V as B, 16 positions by 8 dims per
// product). Positions past the page's end read s.zrow (zero K and V), the new
// token's position reads s.knew / s.vnew. Lane (g, t) keeps head g's running m
// and l and its O at dims 64 dg + 8d + 2t, +1 for d < 8.
template <int HD>
__device__ __forceinline__ void attn_tiles(const Smem &s, uint32_t kbase, uint32_t vbase, int n, bool with_new,
                                           float &m_run, float &l_run, float (&o)[8][2], int dg, int tile0,
                                           int tstride, int PP) {
    constexpr int KS = HD / 16;  // k-steps
    const int lane = threadIdx.x & 31, t = lane & 3, mi = lane >> 3, r = lane & 7;
    const int nt = n + (with_new ? 1 : 0);
    const uint32_t half_bytes = uint32_t(PP) * 128u;
    for (int tile = tile0; tile * ATT_TILE < nt; tile += tstride) {
        const int j0 = tile * ATT_TILE;
        // this lane's ldmatrix row for K: position jk, 16-byte chunk 2 (ks % 4) + (mi & 1)
        // of dim half ks / 4; for V: position jv, chunk 2 dd + (mi >> 1) of half dg
        uint32_t krow, kh, kx, vrow, vx;
        {
            const int jk = j0 + 8 * (mi >> 1) + r;
            if (jk < n) {
                krow = kbase + uint32_t(jk) * 128u, kh = half_bytes, kx = uint32_t(jk & 7);
            } else if (with_new && jk == n) {
                krow = smem_addr(s.knew), kh = 128u, kx = 0u;
            } else {
                krow = smem_addr(s.zrow), kh = 0u, kx = 0u;
            }
            const int jv = j0 + 8 * (mi & 1) + r;
            if (jv < n) {
                vrow = vbase + uint32_t(dg) * half_bytes + uint32_t(jv) * 128u, vx = uint32_t(jv & 7);
            } else if (with_new && jv == n) {
                vrow = smem_addr(s.vnew) + uint32_t(dg) * 128u, vx = 0u;
            } else {
                vrow = smem_addr(s.zrow), vx = 0u;
            }
        }
        // scores: c[nb] covers positions j0 + 8 nb .. + 7 (columns), hi / lo rows
        float c[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
        const uint4 *qa = &s.qf[0][lane];
#pragma unroll
        for (int ks = 0; ks < KS; ks++) {
            uint32_t b[4];
            const uint32_t ch = uint32_t(2 * (ks & 3) + (mi & 1));
            ldsm_x4(krow + uint32_t(ks >> 2) * kh + ((ch ^ kx) << 4), b);
            const uint4 a = lds_v4(smem_addr(qa + ks * 32));  // (volatile: not kept across tiles)
            mma_16816(c[0], a, b[0], b[1]);
            mma_16816(c[1], a, b[2], b[3]);
        }
        // this lane: head g at positions j0 + 2t, +1 (c[0]) and j0 + 8 + 2t, +1 (c[1])
        float sc[4];
#pragma unroll
        for (int nb = 0; nb < 2; nb++)
#pragma unroll
            for (int e = 0; e < 2; e++) {
                const int j = j0 + 8 * nb + 2 * t + e;
                sc[2 * nb + e] = j < nt ? c[nb][e] + c[nb][e + 2] : -INFINITY;
            }
        float mt = fmaxf(fmaxf(sc[0], sc[1]), fmaxf(sc[2], sc[3]));
        mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, 1));
        mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, 2));
        const float m_new = fmaxf(m_run, mt);  // finite: position j0 exists
        const float alpha = m_run == -INFINITY ? 0.f : expf(m_run - m_new);
        float pr[4], ps = 0.f;
#pragma unroll
        for (int e = 0; e < 4; e++) {
            pr[e] = sc[e] == -INFINITY ? 0.f : expf(sc[e] - m_new);
            ps += pr[e];
        }
        ps += __shfl_xor_sync(0xffffffffu, ps, 1);
        ps += __shfl_xor_sync(0xffffffffu, ps, 2);
        l_run = l_run * alpha + ps;
        m_run = m_new;
        uint16_t h[4], lo[4];
#pragma unroll
        for (int e = 0; e < 4; e++) split_bf16(pr[e], h[e], lo[e]);
        const uint4 pa = make_uint4(uint32_t(h[0]) | (uint32_t(h[1]) << 16), uint32_t(lo[0]) | (uint32_t(lo[1]) << 16),
                                    uint32_t(h[2]) | (uint32_t(h[3]) << 16), uint32_t(lo[2]) | (uint32_t(lo[3]) << 16));
        // P.V: 8 dims per product, two products per ldmatrix
#pragma unroll
        for (int dd = 0; dd < 4; dd++) {
            uint32_t b[4];
            const uint32_t ch = uint32_t(2 * dd + (mi >> 1));
            ldsm_x4_t(vrow + ((ch ^ vx) << 4), b);
#pragma unroll
            for (int u = 0; u < 2; u++) {
                const int d = 2 * dd + u;
                float acc[4] = {o[d][0] * alpha, o[d][1] * alpha, 0.f, 0.f};
                mma_16816(acc, pa, b[2 * u], b[2 * u + 1]);
                o[d][0] = acc[0] + acc[2];
                o[d][1] = acc[1] + acc[3];
            }
        }
    }
}

template <int DL, bool BATCH = false>
__device__ bool attn_item_flash(const KParams &p, Smem &s, uint8_t *pages, const Instr &ins, int ii, uint32_t &cpage) {
    const int g = ins.r0, c = ins.r1, S = p.attn_splits, l = ins.layer;
    constexpr int hd = DL * 32, half = hd / 2;
    const int G = p.nq / p.nkv, tid = threadIdx.x;
    const int qd = p.nq * hd, kd = p.nkv * hd;
    const bool owner = c == S - 1;  // this split owns position pos
    const float scale = 1.0f / sqrtf(static_cast<float>(hd));
    const int b = BATCH ? int(ins.sub) : 0;
    const int pos = BATCH ? s.bpos[b] : s.c_pos;
    const float2 *cs = p.rope_cs + size_t(pos) * half;
    const uint64_t *qkv_b = p.t_qkv + size_t(b) * (qd + 2 * kd);
    const uint32_t tag = tag_of(p, s, l);
    // the group's query heads with RoPE ("rotate half") applied, pre-scaled by
    // 1/sqrt(hd); the owner also rotates the new key and takes the new value
    {
        const uint64_t *qh = qkv_b + size_t(g * G) * hd;
        const uint64_t *kh = qkv_b + qd + size_t(g) * hd;
        const uint64_t *vh = qkv_b + qd + kd + size_t(g) * hd;
        const bool has_q = tid < G * hd, has_k = owner && tid < half, has_v = owner && tid < hd;
        const int h = tid / hd, d = tid % hd, i = d < half ? d : d - half;
        uint64_t w[5];
        poll_words(p, s, w, tag, [&](uint64_t (&ww)[5]) {
            const uint64_t ok = static_cast<uint64_t>(tag) << 32;
            ww[0] = has_q ? ld_tag(qh + size_t(h) * hd + i) : ok;
            ww[1] = has_q ? ld_tag(qh + size_t(h) * hd + i + half) : ok;
            ww[2] = has_k ? ld_tag(kh + tid) : ok;
            ww[3] = has_k ? ld_tag(kh + tid + half) : ok;
            ww[4] = has_v ? ld_tag(vh + tid) : ok;
        });
        if (has_q) {
            const float a = tag_val(w[0]), b = tag_val(w[1]);
            const float2 r = cs[i];
            s.qr[h][d] = (d < half ? a * r.x - b * r.y : a * r.y + b * r.x) * scale;
        }
        if (has_k) {
            const float a = tag_val(w[2]), b = tag_val(w[3]);
            const float2 r = cs[tid];
            s.knew[tid] = f_to_bf16(a * r.x - b * r.y);
            s.knew[tid + half] = f_to_bf16(a * r.y + b * r.x);
        }
        if (has_v) s.vnew[tid] = f_to_bf16(tag_val(w[4]));
    }
    if (tid < G) {
        s.m_run[tid] = -INFINITY;
        s.l_run[tid] = 0.f;
    }
    if (consumer_any(s.abort)) return false;
    // the queries as tensor-core A fragments: lane (g, t) of k-step ks holds head g
    // at dims 16ks + 2t, +1 (x: bf16 hi, y: lo) and 16ks + 2t + 8, +9 (z: hi, w: lo),
    // zero past G heads
    for (int i = tid; i < (hd / 16) * 32; i += NCT) {
        const int ks = i / 32, ln = i % 32, g = ln >> 2, t = ln & 3;
        uint16_t h[4] = {0, 0, 0, 0}, lo[4] = {0, 0, 0, 0};
        if (g < G) {
            const int d[4] = {16 * ks + 2 * t, 16 * ks + 2 * t + 1, 16 * ks + 2 * t + 8, 16 * ks + 2 * t + 9};
#pragma unroll
            for (int e = 0; e < 4; e++) split_bf16(s.qr[g][d[e]], h[e], lo[e]);
        }
        s.qf[ks][ln] = make_uint4(uint32_t(h[0]) | (uint32_t(h[1]) << 16), uint32_t(lo[0]) | (uint32_t(lo[1]) << 16),
                                  uint32_t(h[2]) | (uint32_t(h[3]) << 16), uint32_t(lo[2]) | (uint32_t(lo[3]) << 16));
    }
    consumer_sync();
    if (tid == 0) trace_put(p, ii, 1);
    if (owner) {
        const size_t at = ((size_t(l) * p.nkv + g) * size_t(p.max_seq) + pos) * hd;
        uint16_t *kc = BATCH ? p.kc_b[b] : p.k_cache, *vc = BATCH ? p.vc_b[b] : p.v_cache;
        if (LL_OK_IDX(16, at + hd, size_t(p.L) * p.nkv * p.max_seq * hd + 1))
            for (int d = tid; d < hd; d += NCT) {
                kc[at + d] = s.knew[d];
                vc[at + d] = s.vnew[d];
            }
    }
    // this lane's share of the running softmax and output (see attn_tiles)
    float m_run = -INFINITY, l_run = 0.f, o[8][2];
#pragma unroll
    for (int d = 0; d < 8; d++) o[d][0] = o[d][1] = 0.f;
    int c0, c1;
    attn_range(p, pos, c, c0, c1);
    const int PP = attn_pp(p);
    // The warps form DG dim groups (64 dims each); within a dim group, NGR page
    // groups of W warps each take every NGR-th page of the item, W warps sharing a
    // page's tiles. So NGR pages are worked on at once and a warp's chain of tiles
    // per page stays short; the last of a page's DG * W warps releases it.
    constexpr int DG = hd / 64, GWD = NCW / DG, NGR = 4, W = GWD / NGR;
    const int warp_i = tid >> 5, lane_i = tid & 31;
    const int dgi = warp_i / GWD, pgq = (warp_i % GWD) / W, wi = warp_i % W;
    bool bad = false;
    int npg = 0;
    for (int p0 = c0; p0 < c1; p0 += PP, npg++) {
        const uint32_t page = cpage + uint32_t(npg), slot = page % NPAGES;
        if (npg % NGR != pgq) continue;
        const int n = min(PP, c1 - p0);
        const bool with_new = owner && p0 + PP >= c1;  // fold the new token into the last page
        bool okp = !bad;
        if (lane_i == 0 && okp) okp = wait_page(p, s, page);
        okp = __shfl_sync(0xffffffffu, okp, 0);
        if (!okp) {
            bad = true;
            continue;
        }
        const uint32_t pg = smem_addr(pages + size_t(slot) * PAGE_BYTES);
        attn_tiles<hd>(s, pg, pg + PAGE_BYTES / 2, n, with_new, m_run, l_run, o, dgi, wi, W, PP);  // V at half a page
        __syncwarp();
        if (lane_i == 0) {
            __threadfence_block();
            if (atomicAdd(&s.pcnt[slot], 1) == DG * W - 1) {
                s.pcnt[slot] = 0;
                ptrace_put(p, page, 2);
                mbar_arrive_cnt(&s.empty[slot], NCW);
            }
        }
    }
    cpage += uint32_t(npg);
    if (consumer_any(bad)) return false;
    if (owner && c0 == c1 && pgq == 0) attn_tiles<hd>(s, 0u, 0u, 0, true, m_run, l_run, o, dgi, wi, W, PP);
    consumer_sync();  // s.qf is read up to here; the merge below reuses its space
    if (tid == 0) trace_put(p, ii, 7);

    // merge the warps of each dim group pairwise, halving their number each round
    constexpr int GW = NCW * 64 / hd;
    const int warp = tid >> 5, dg = warp / GW, tw = warp % GW, gq = (tid & 31) >> 2, tq = tid & 3;
    for (int half = GW / 2; half >= 1; half /= 2) {
        if (tw >= half && tw < 2 * half && gq < G) {
            float *sl = s.ared[dg * (GW / 2) + tw - half];
#pragma unroll
            for (int d = 0; d < 8; d++) {
                sl[gq * 64 + 8 * d + 2 * tq] = o[d][0];
                sl[gq * 64 + 8 * d + 2 * tq + 1] = o[d][1];
            }
            if (tq == 0) {
                sl[512 + gq] = m_run;
                sl[512 + MAX_GQA + gq] = l_run;
            }
        }
        consumer_sync();
        if (tw < half && gq < G) {
            const float *sl = s.ared[dg * (GW / 2) + tw];
            const float mo = sl[512 + gq], lo = sl[512 + MAX_GQA + gq];
            const float M = fmaxf(m_run, mo);
            const float wa = m_run == -INFINITY ? 0.f : expf(m_run - M), wb = mo == -INFINITY ? 0.f : expf(mo - M);
            l_run = l_run * wa + lo * wb;
            m_run = M;
#pragma unroll
            for (int d = 0; d < 8; d++) {
                o[d][0] = o[d][0] * wa + sl[gq * 64 + 8 * d + 2 * tq] * wb;
                o[d][1] = o[d][1] * wa + sl[gq * 64 + 8 * d + 2 * tq + 1] * wb;
            }
        }
        consumer_sync();
    }

    // partials: part[(qhead * S + c) * (hd + 4) + {d, hd: m, hd+1: l}], from the
    // first warp of every dim group
    const int stride = hd + 4;
    const uint32_t wtag = write_tag(p, s, ins);
    if (tw == 0 && gq < G) {
        uint64_t *dst = p.t_part + size_t(b) * p.nq * S * stride + (size_t(g * G + gq) * S + c) * stride;
#pragma unroll
        for (int d = 0; d < 8; d++) {
            st_tag(dst + 64 * dg + 8 * d + 2 * tq, o[d][0], wtag);
            st_tag(dst + 64 * dg + 8 * d + 2 * tq + 1, o[d][1], wtag);
        }
        if (dg == 0 && tq == 0) {
            st_tag(dst + hd, m_run, wtag);
            st_tag(dst + hd + 1, l_run, wtag);
        }
    }
    if (tid == 0) trace_put(p, ii, 2);
    return merge_splits(p, s, g, c, G, hd, tag, wtag, b);
}


// ---------------------------------------------------------------------------------
// The tensor-core kernel: matrix-vector instructions on tensor-core pages for nb
// sequences at once (a batched handle; a single-sequence handle is a batch of
// one). The columns of width K are cut into nch chunks of kc (2048, or 1024); a
// page holds nr <= TC_ROWS rows of one chunk, loaded by one TMA copy of a 3-D
// view of the matrix (64 columns, rows, K / 64 column blocks) in the 128-byte
// swizzle: column block o of row r is the 128-byte line o * nr + r of the page,
// its 16-byte chunk c at chunk c ^ ((o * nr + r) % 8). So the eight rows an
// ldmatrix reads at one column block fall in eight different bank groups.
//
// The product is m16n8k16 with the inputs as the A operand and the page's rows
// as B (n = 8 rows). Each sequence's input enters as T bf16 terms, x = t0 + t1
// (+ t2): T = 3 (to the 24 bits of an fp32 value) for up to 4 sequences, T = 2 (~16
// bits) for 5..8; one term misses the logits' bar, and with two the bf16 roundings
// of stored K/V flip measurably more often than with fp32 products. A row r of A
// is (sequence, term): rows 0..7 hold the first 8 / T * T of them, rows 8..15 the
// next. All NCW warps work on every page, warp w on its own KS / 4 64-column
// blocks of the chunk, so a page costs the same products for one sequence or
// eight. The RMSNorm gain multiplies the input before the split and the norm's
// 1 / rms, one number per sequence, multiplies the sums after.
//
// A warp's partial sums of a page go into that page's own lines of the warp's
// columns (read by no other warp, and done with once its products are issued):
// shared memory has no room for NCW x 8 sequences x 8 rows per ring slot. The last
// warp to finish the page adds the NCW partials into s.bacc and releases it.

// The epilogue of a tensor-core instruction, once s.bacc holds every (row,
// sequence) sum: per sequence b, q/k/v, the residual stream, silu(gate) * up, or
// the logits and this thread's running argmax, stored as the instruction's
// outputs; sums of a normed input are scaled by b's 1 / rms here. Thread tid
// handles sequence tid % nb (nb divides NCT), so its best/best_idx belong to one
// sequence.
__device__ __forceinline__ void mv_store_b(const KParams &p, Smem &s, const Instr &ins, int ii, bool normed,
                                           float &best, int &best_idx) {
    const int tid = threadIdx.x, nb = p.nb;
    const int nrows = ins.r1 - ins.r0, r0 = ins.r0;
    const uint32_t wtag = write_tag(p, s, ins);
    const int b = tid % nb;
    float rn = 1.0f;
    if (normed) {
        float tot = 0.f;
#pragma unroll
        for (int w = 0; w < NCW; w++) tot += s.nredb[w][b];
        rn = 1.0f / sqrtf(tot / static_cast<float>(mv_of(p, ins.op).K) + p.eps);
    }
    const int qkvd = (p.nq + 2 * p.nkv) * p.hd;
    for (int idx = tid; idx < nrows * nb; idx += NCT) {
        const int t = idx / nb;  // idx % nb == b
        const float y = s.bacc[idx] * rn;
        switch (ins.op) {
            case OP_QKV:
                if (LL_OK_IDX(5, r0 + t, qkvd)) st_tag(p.t_qkv + size_t(b) * qkvd + r0 + t, y, wtag);
                break;
            case OP_OPROJ:
            case OP_DOWN: {
                const int row = r0 + t;
                if (!LL_OK_IDX(7, row, p.H) || !LL_OK_IDX(20, t, XOWN_MAX)) break;
                const float base = ins.op == OP_OPROJ && ins.layer == 0
                                       ? bf16_to_f(p.embed[size_t(s.btoken[b]) * p.H + row])
                                       : s.bxown[b][t];
                const float v = base + y;
                s.bxown[b][t] = v;
                st_tag((ins.op == OP_OPROJ ? p.t_xmid : p.t_xout) + size_t(b) * p.H + row, v, wtag);
                break;
            }
            case OP_GATEUP: {
                const float u = s.bacc[(nrows + t) * nb + b] * rn;
                if (LL_OK_IDX(8, r0 + t, p.I)) st_tag(p.t_act + size_t(b) * p.I + r0 + t, y / (1.0f + expf(-y)) * u, wtag);
                break;
            }
            default:  // OP_LMHEAD: rows ascend per thread
                if (s.c_logits && LL_OK_IDX(10, r0 + t, p.V)) s.c_logits[size_t(b) * p.V + r0 + t] = y;
                if (y > best) {
                    best = y;
                    best_idx = r0 + t;
                }
                break;
        }
    }
    if (threadIdx.x == 0) trace_put(p, ii, 2);
}

// Greedy argmax of every sequence across the grid (batched handles): each SM
// publishes its best key per sequence, the last SM to arrive reduces them and
// writes the tokens. Thread tid's best is for sequence tid % nb.
__device__ void lm_finish_b(const KParams &p, Smem &s, float best, int best_idx) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, tid = threadIdx.x, nb = p.nb;
    unsigned long long key = best_idx >= 0 ? argmax_key(best, best_idx) : 0ull;
    for (int o = 16; o >= nb; o >>= 1) {
        const unsigned long long w = __shfl_xor_sync(0xffffffffu, key, o);
        key = w > key ? w : key;
    }
    unsigned long long *kr = reinterpret_cast<unsigned long long *>(s.xin);  // [NCW][MAX_B]
    if (lane < nb) kr[warp * MAX_B + lane] = key;
    consumer_sync();
    if (tid < nb) {
        unsigned long long k = 0;
        for (int w = 0; w < NCW; w++) k = kr[w * MAX_B + tid] > k ? kr[w * MAX_B + tid] : k;
        p.lm_keys[size_t(blockIdx.x) * nb + tid] = k;
        __threadfence();
    }
    consumer_sync();
    if (tid == 0) {
        const uint32_t old = atomicAdd(p.ctr + size_t(CtrLayout::lm_ticket(p.L)) * CTR_STRIDE, 1u);
        s.flag = (old + 1u == s.c_epoch * static_cast<uint32_t>(p.nsm)) ? 1 : 0;
        __threadfence();
    }
    consumer_sync();
    if (!s.flag || warp >= nb) return;
    // warp b reduces sequence b
    const int b = warp;
    unsigned long long k = 0;
    for (int i = lane; i < p.nsm; i += 32) {
        const unsigned long long v = __ldcg(p.lm_keys + size_t(i) * nb + b);
        k = v > k ? v : k;
    }
    k = warp_max_u64(k);
    if (lane == 0) {
        if (k == 0) atomicCAS(p.status, 0, LL_ERR_NUMERIC);  // every logit NaN: no greedy token
        const int32_t tok = static_cast<int32_t>(0xffffffffu - static_cast<uint32_t>(k & 0xffffffffu));
        p.token_out[b] = tok;
        if (p.tokens_dev) p.tokens_dev[size_t(s.c_epoch - p.epoch) * nb + b] = tok;
        else if (p.next_token_dev) p.next_token_dev[b] = tok;
        if (p.n_steps > 1) {
            __threadfence();
            const uint64_t w = (static_cast<uint64_t>(s.c_epoch) << 32) | static_cast<uint32_t>(tok);
            asm volatile("st.relaxed.gpu.global.b64 [%0], %1;" ::"l"(p.t_token + b), "l"(w) : "memory");
        }
    }
}

// The step the consumers of the tensor-core kernel start: as consumer_step_begin,
// for each of the nb sequences (its position, and after a launch's first step the
// token the previous step chose for it).
__device__ bool consumer_step_begin_b(const KParams &p, Smem &s, int st) {
    if (threadIdx.x == 0) {
        s.c_epoch = p.epoch + static_cast<uint32_t>(st);
        s.c_pos = p.pos_b[0] + st;
        s.c_logits = p.logits ? p.logits + size_t(st) * size_t(p.nb) * size_t(p.V) : nullptr;
    }
    if (threadIdx.x < p.nb) {
        const int b = threadIdx.x;
        s.bpos[b] = p.pos_b[b] + st;
        if (st > 0) {
            const uint32_t prev = p.epoch + static_cast<uint32_t>(st - 1);
            uint64_t w = 0, t0 = 0;
            for (uint32_t it = 0;; ++it) {
                w = ld_tag(p.t_token + b);
                if (tag_ok(w, prev) || poll_give_up(p, s, it, t0)) break;
            }
            asm volatile("fence.acq_rel.gpu;" ::: "memory");
            s.btoken[b] = static_cast<int32_t>(static_cast<uint32_t>(w));
            // a step without a greedy token (no orderable logit) hands on -1:
            // stop here rather than index the embedding with it
            if (s.btoken[b] < 0 || s.btoken[b] >= p.V) raise_status(p, s, LL_ERR_NUMERIC);
        }
    }
    if (consumer_any(s.abort)) return false;
    if (threadIdx.x == 0) {
        s.token = s.btoken[0];
        if (st > 0) {
            // what the sequences' threads acquired, released to the producer's gate
            asm volatile("fence.acq_rel.gpu;" ::: "memory");
            s.tok_step = st;
        }
    }
    return !consumer_any(s.abort);
}

// Sequence and term of A row r (0..15), or -1.
__device__ __forceinline__ int tc_seq(int r, int nb, int T, int &term) {
    const int half = r >> 3, rr = r & 7, spb = 8 / T;
    term = rr % T;
    if (rr >= spb * T) return -1;
    const int b = half * spb + rr / T;
    return b < nb ? b : -1;
}

// Term `term` (0, 1, 2) of the pair (v0, v1) as packed bf16x2: term k is the
// bf16 nearest (round to nearest even, the cvt instruction) to what terms
// 0..k-1 leave of each value.
__device__ __forceinline__ uint32_t cvt_bf16x2(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}
__device__ __forceinline__ uint32_t bf16x2_term(float v0, float v1, int term) {
    uint32_t h = cvt_bf16x2(v0, v1);
    if (term == 0) return h;
    v0 -= bf_lo(h);
    v1 -= bf_hi(h);
    h = cvt_bf16x2(v0, v1);
    if (term == 1) return h;
    v0 -= bf_lo(h);
    v1 -= bf_hi(h);
    return cvt_bf16x2(v0, v1);
}

// A fragments of column chunk c for this lane's two A rows (g and g + 8):
// a[j] = {a0, a1, a2, a3} of k-step j of the warp (rows g / g + 8 at columns 2t,
// 2t + 1 and 2t + 8, 2t + 9 of the k-step). The inputs are staged in s.xin as
// fp32, XIN_FLOATS / kc sequences at a time, from the previous instruction's
// tagged words (or the tokens' embedding rows for layer 0). With count_ss, this
// lane adds the squares of the values of its term-0 rows to ssl[h].
template <int KS>
__device__ bool tc_fragments(const KParams &p, Smem &s, const Instr &ins, const MvShape &mv, int c, const uint64_t *src,
                             uint32_t tag, const uint16_t *gain, int b_lo, int t_lo, int b_hi, int t_hi, bool count_ss,
                             float (&ssl)[2], uint32_t (&a)[KS][4]) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, tid = threadIdx.x, t = lane & 3;
    const int nb = p.nb, K = mv.K, Kc = mv.kc, NSR = XIN_FLOATS / Kc;
#pragma unroll
    for (int j = 0; j < KS; j++) a[j][0] = a[j][1] = a[j][2] = a[j][3] = 0u;
    for (int b0 = 0; b0 < nb; b0 += NSR) {
        const int nsr = min(NSR, nb - b0), total = nsr * Kc;
        consumer_sync();  // s.xin is free
        if (src) {
            constexpr int PAIRS = XIN_FLOATS / (2 * NCT);
            uint64_t w[2 * PAIRS];
            poll_words(p, s, w, tag, [&](uint64_t (&ww)[2 * PAIRS]) {
#pragma unroll
                for (int k = 0; k < PAIRS; k++) {
                    const int i = (tid + k * NCT) * 2;
                    if (i < total) {
                        const int sq = b0 + i / Kc, kk = i % Kc;
                        ld_tag2(src + size_t(sq) * K + size_t(c) * Kc + kk, ww[2 * k], ww[2 * k + 1]);
                    } else {
                        ww[2 * k] = ww[2 * k + 1] = static_cast<uint64_t>(tag) << 32;
                    }
                }
            });
#pragma unroll
            for (int k = 0; k < PAIRS; k++) {
                const int i = (tid + k * NCT) * 2;
                if (i < total) {
                    s.xin[i] = tag_val(w[2 * k]);
                    s.xin[i + 1] = tag_val(w[2 * k + 1]);
                }
            }
        } else {
            for (int i = tid; i < total; i += NCT) {
                const int sq = b0 + i / Kc, kk = i % Kc;
                s.xin[i] = bf16_to_f(p.embed[size_t(s.btoken[sq]) * p.H + size_t(c) * Kc + kk]);
            }
        }
        if (consumer_any(s.abort)) return false;  // also publishes s.xin
#pragma unroll
        for (int h = 0; h < 2; h++) {
            const int b = h ? b_hi : b_lo, term = h ? t_hi : t_lo;
            if (b < b0 || b >= b0 + nsr) continue;
            const float *xs = s.xin + (b - b0) * Kc;
#pragma unroll
            for (int j = 0; j < KS; j++) {
                const int k = (warp * KS + j) * 16 + 2 * t;  // within the chunk
#pragma unroll
                for (int q = 0; q < 2; q++) {
                    const float2 x = *reinterpret_cast<const float2 *>(xs + k + 8 * q);
                    float v0 = x.x, v1 = x.y;
                    if (count_ss && term == 0) ssl[h] = fmaf(v0, v0, fmaf(v1, v1, ssl[h]));
                    if (gain) {
                        const uint32_t gw = __ldg(reinterpret_cast<const uint32_t *>(gain + size_t(c) * Kc + k + 8 * q));
                        v0 *= bf_lo(gw);
                        v1 *= bf_hi(gw);
                    }
                    a[j][h + 2 * q] = bf16x2_term(v0, v1, term);
                }
            }
        }
    }
    return true;
}

template <int KS>
__device__ bool mv_instr_tc(const KParams &p, Smem &s, uint8_t *pages, const Instr &ins, int ii, uint32_t &cpage,
                            float &best, int &best_idx) {
    static_assert(KS == 4 || KS == 8, "a warp works on whole 64-column blocks");
    const MvShape &mv = mv_of(p, ins.op);
    Seg seg[3];
    const int nseg = mv_segments(p, s, ins, seg);
    if (nseg == 0) return true;  // no rows here: nothing to read or wait for
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, tid = threadIdx.x;
    const int g = lane >> 2, t = lane & 3, q = lane >> 3, rr = lane & 7;
    const int nb = p.nb, T = nb <= 4 ? 3 : 2;
    int t_lo, t_hi;
    const int b_lo = tc_seq(g, nb, T, t_lo), b_hi = tc_seq(g + 8, nb, T, t_hi);
    const uint16_t *gain = norm_gain(p, s, ins);
    const uint64_t *src = nullptr;
    uint32_t tag = 0;
    switch (ins.op) {
        case OP_QKV:
            if (ins.layer > 0) {
                src = p.t_xout;
                tag = tag_of(p, s, ins.layer - 1);
            }
            break;
        case OP_GATEUP: src = p.t_xmid; tag = tag_of(p, s, ins.layer); break;
        case OP_LMHEAD: src = p.t_xout; tag = tag_of(p, s, p.L - 1); break;
        case OP_DOWN: src = p.t_act; tag = tag_of(p, s, ins.layer); break;
        default: src = p.t_o; tag = tag_of(p, s, ins.layer); break;  // OP_OPROJ
    }
    const int nrows = ins.r1 - ins.r0;
    const int ntot = (ins.op == OP_GATEUP ? 2 : 1) * nrows;
    for (int i = tid; i < ntot * nb; i += NCT)
        if (LL_OK_IDX(30, i, BACC_FLOATS)) s.bacc[i] = 0.f;
    const uint32_t zrow = smem_addr(s.zrow);
    float ssl[2] = {0.f, 0.f};
    uint32_t a[KS][4];
    int have = -1;  // the chunk whose fragments a[] holds
    bool bad = false;
    for (int si = 0; si < nseg; si++) {
        const Seg sg = seg[si];
        const int acc0 = sg.kind == OUT_QKV ? sg.out0 + sg.row0 - ins.r0 : (sg.kind == OUT_UP ? nrows : 0);
        for (int c = 0; c < mv.nch; c++) {
            if (c != have) {
                if (!tc_fragments<KS>(p, s, ins, mv, c, src, tag, gain, b_lo, t_lo, b_hi, t_hi, si == 0, ssl, a))
                    return false;
                if (tid == 0 && si == 0 && c == 0) trace_put(p, ii, 1);
                have = c;
            }
            for (int pr = 0; pr < sg.nrows; pr += TC_ROWS) {
                const int nr = min(TC_ROWS, sg.nrows - pr);
                const uint32_t slot = cpage % NPAGES;
                const uint32_t this_page = cpage++;
                if (bad || !wait_page(p, s, this_page)) {
                    bad = true;
                    continue;
                }
                if (warp == 0 && lane == 0) {
                    ptrace_put(p, this_page, 1);
                    if (si == 0 && c == 0 && pr == 0) trace_put(p, ii, 6);
                }
                uint8_t *pg = pages + size_t(slot) * PAGE_BYTES;
                const uint32_t base = smem_addr(pg);
                float d[4] = {0.f, 0.f, 0.f, 0.f}, e[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int j = 0; j < KS; j += 2) {
                    const int ks = warp * KS + j;  // k-steps ks, ks + 1: columns 16 ks .. 16 ks + 31 of the chunk
                    const int line = (ks >> 2) * nr + rr;
                    const uint32_t chunk = uint32_t((ks & 3) * 2 + q);
                    const uint32_t at =
                        rr < nr ? base + uint32_t(line) * 128u + ((chunk ^ uint32_t(line & 7)) << 4) : zrow;
                    uint32_t bm[4] = {0u, 0u, 0u, 0u};
                    if (at == zrow || LL_OK_IDX(21, at + 16 - smem_addr(pages), NPAGES * PAGE_BYTES + 1)) ldsm_x4(at, bm);
                    mma_16816(d, make_uint4(a[j][0], a[j][1], a[j][2], a[j][3]), bm[0], bm[1]);
                    mma_16816(e, make_uint4(a[j + 1][0], a[j + 1][1], a[j + 1][2], a[j + 1][3]), bm[2], bm[3]);
                }
                // D: lane (g, t) holds A rows g (d0, d1) and g + 8 (d2, d3) at page rows
                // 2t, 2t + 1; a sequence's terms are the rows below its term 0, 4 lanes apart
                float v[4] = {d[0] + e[0], d[1] + e[1], d[2] + e[2], d[3] + e[3]};
                if (T == 3) {
#pragma unroll
                    for (int i = 0; i < 4; i++) {
                        const float u4 = __shfl_down_sync(0xffffffffu, v[i], 4);
                        const float u8 = __shfl_down_sync(0xffffffffu, v[i], 8);
                        v[i] += u4 + u8;
                    }
                } else {
#pragma unroll
                    for (int i = 0; i < 4; i++) v[i] += __shfl_down_sync(0xffffffffu, v[i], 4);
                }
                // partials [row][sequence] into the page lines of this warp's columns
                float *own = reinterpret_cast<float *>(pg + size_t((warp * KS) >> 2) * nr * 128);
#pragma unroll
                for (int h = 0; h < 2; h++) {
                    const int b = h ? b_hi : b_lo, term = h ? t_hi : t_lo;
                    if (b < 0 || term != 0) continue;
#pragma unroll
                    for (int e2 = 0; e2 < 2; e2++) {
                        const int r = 2 * t + e2;
                        if (r < nr && LL_OK_IDX(31, r * nb + b, nr * 32)) own[r * nb + b] = v[2 * h + e2];
                    }
                }
                // these generic writes precede the producer's next TMA write of the slot
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                __syncwarp();
                int last = 0;
                if (lane == 0) {
                    __threadfence_block();
                    last = atomicAdd(&s.pcnt[slot], 1) == NCW - 1;
                }
                last = __shfl_sync(0xffffffffu, last, 0);
                if (last) {  // this warp finishes the page: the NCW partials of every (row, sequence)
                    __threadfence_block();
                    for (int idx = lane; idx < nr * nb; idx += 32) {
                        float y = 0.f;
#pragma unroll
                        for (int w = 0; w < NCW; w++)
                            y += reinterpret_cast<const float *>(pg + size_t((w * KS) >> 2) * nr * 128)[idx];
                        const int r = idx / nb, b = idx % nb;
                        if (LL_OK_IDX(4, (acc0 + pr + r) * nb + b, BACC_FLOATS)) s.bacc[(acc0 + pr + r) * nb + b] += y;
                    }
                    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                    __syncwarp();
                    if (lane == 0) {
                        s.pcnt[slot] = 0;
                        ptrace_put(p, this_page, 2);
                        mbar_arrive_cnt(&s.empty[slot], NCW);
                    }
                }
            }
        }
    }
    if (tid == 0) trace_put(p, ii, 7);
    if (consumer_any(bad)) return false;  // else every page is reduced into s.bacc
    // each warp's share of every sequence's sum of squares (normed inputs)
    if (gain) {
#pragma unroll
        for (int h = 0; h < 2; h++) {
            float v2 = ssl[h];
            v2 += __shfl_xor_sync(0xffffffffu, v2, 1);
            v2 += __shfl_xor_sync(0xffffffffu, v2, 2);
            const int b = h ? b_hi : b_lo, term = h ? t_hi : t_lo;
            if (t == 0 && b >= 0 && term == 0) s.nredb[warp][b] = v2;
        }
        consumer_sync();
    }
    mv_store_b(p, s, ins, ii, gain != nullptr, best, best_idx);
    return true;
}
// FLASH: the kernel variant for long attention items (see attn_tiles); the other
// variant keeps a block-wide softmax per page, cheaper when an item spans a page
// or two. The host picks the variant by the longest item at max_seq.
// (TC: the tensor-core kernel, whose items carry their sequence)
template <bool FLASH, bool TC = false>
__device__ bool attn_instr(const KParams &p, Smem &s, uint8_t *pages, const Instr &ins, int ii, uint32_t &cpage) {
    if constexpr (FLASH)
        return p.hd == 64 ? attn_item_flash<2, TC>(p, s, pages, ins, ii, cpage)
                          : attn_item_flash<4, TC>(p, s, pages, ins, ii, cpage);
    else
        return p.hd == 64 ? attn_item<2, TC>(p, s, pages, ins, ii, cpage) : attn_item<4, TC>(p, s, pages, ins, ii, cpage);
}

// ---------------------------------------------------------------------------------
// Producer: walks the same instruction list and streams every page in order.
// While the ring is full and the consumers are held up by a dependency, it keeps
// HBM busy by prefetching the pages that come next into L2
// (cp.async.bulk.prefetch.L2), up to p.l2_prefetch pages ahead of the ring, so
// that the ring refills from L2 once the dependency is met.

__device__ __forceinline__ void bulk_prefetch_l2(const void *src, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

__device__ __forceinline__ void bulk_load_hint(void *dst, const void *src, uint32_t bytes, uint64_t *bar,
                                               uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], "
        "%4;" ::"r"(smem_addr(dst)),
        "l"(src), "r"(bytes), "r"(smem_addr(bar)), "l"(policy)
        : "memory");
}

// TMA tensor copy of one box of a 2-D tensor map (coordinates: x the inner
// element index, a multiple of 64 here; y the row) into shared memory.
__device__ __forceinline__ void tma_load_2d(void *dst, const TensorMap *map, int x, int y, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], "
        "[%4];" ::"r"(smem_addr(dst)),
        "l"(reinterpret_cast<unsigned long long>(map)), "r"(x), "r"(y), "r"(smem_addr(bar))
        : "memory");
}

// TMA tensor copy of one box of a 3-D tensor map (x, y, z coordinates) into
// shared memory, with an L2 cache policy.
__device__ __forceinline__ void tma_load_3d_hint(void *dst, const TensorMap *map, int x, int y, int z, uint64_t *bar,
                                                 uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1, "
        "{%2, %3, %4}], [%5], %6;" ::"r"(smem_addr(dst)),
        "l"(reinterpret_cast<unsigned long long>(map)), "r"(x), "r"(y), "r"(z), "r"(smem_addr(bar)), "l"(policy)
        : "memory");
}

// The producer thread walks its SM's host-built page list (weight pages with
// their addresses, attention items expanded from pos here), so that issuing a
// page costs it only a few instructions: it shares its scheduler with consumer
// warps and gets a small share of the issue slots.
template <bool FLASH, bool TC>
__device__ void producer(const KParams &p, Smem &s, uint8_t *pages) {
    const PDesc *dl = p.pdesc + p.pdesc_off[blockIdx.x];
    const int nd = p.pdesc_off[blockIdx.x + 1] - p.pdesc_off[blockIdx.x];
    uint64_t evict_first;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(evict_first));
    uint32_t ppage = 0;
    int pfi = 0;  // next list entry the L2 prefetch may touch
    int last_instr = -1;
    bool ok = true;
    const int PP = attn_pp(p);
    const uint32_t l2_ahead = p.l2_prefetch;
    const uint32_t lim = p.max_inflight >= 1 && p.max_inflight < NPAGES ? p.max_inflight : NPAGES;
    // the list once per step of the launch: weight pages run ahead into the next
    // step freely, K/V pages of a later step wait until the consumers hold that
    // step's input token (everything the previous steps wrote is then visible)
    int gate = 0;  // steps whose K/V pages may be fetched
    for (int st = 0; st < p.n_steps && ok; st++) {
        const int pos = p.pos + st;
        pfi = 0;
        for (int di = 0; di < nd && ok; di++) {
            const PDesc e = dl[di];
            int a_c0 = 0, a_c1 = 1, a_p0 = 0, a_n = 0;
            size_t head_row = 0;
            const uint16_t *a_kc = p.k_cache, *a_vc = p.v_cache;  // the item's sequence's caches
            const TensorMap *a_maps = p.kv_maps;                 // and KV tensor maps
            if (e.kind == PD_ATTN && st > gate) {
                const uint64_t t0 = gtimer();
                for (uint32_t it = 1; s.tok_step < st; ++it) {
                    if ((it & 15u) == 0) {
                        if (s.abort) { ok = false; break; }
                        if (gtimer() - t0 > p.timeout_ns) {
                            raise_status(p, s, LL_ERR_DEP_TIMEOUT);
                            ok = false;
                            break;
                        }
                    }
                }
                if (!ok) break;
                // acquire what the consumers acquired, and order it before this
                // thread's bulk-copy (async proxy) reads of the cache
                asm volatile("fence.acq_rel.gpu;" ::: "memory");
                asm volatile("fence.proxy.async.global;" ::: "memory");
                gate = st;
            }
            if (e.kind == PD_ATTN) {
                const int layer = int((e.src >> 32) & 0xffffu), g = int((e.src >> 16) & 0xffffu), c = int(e.src & 0xffffu);
                int a_pos = pos;
                if (TC) {  // batched handles: the item's sequence
                    const int b = int(e.src >> 48);
                    a_pos = p.pos_b[b] + st;
                    a_kc = p.kc_b[b];
                    a_vc = p.vc_b[b];
                    a_maps = p.kvmaps_b + size_t(b) * TM_COUNT;
                }
                attn_range(p, a_pos, c, a_c0, a_c1);
                a_p0 = a_c0;
                head_row = (size_t(layer) * p.nkv + g) * size_t(p.max_seq);
                if (a_c0 >= a_c1) continue;  // empty split: no pages
            }
            // weight entries are one page; attention entries one page per PP positions
            while (ok) {
                const void *src0, *src1 = nullptr;
                uint32_t b0, b1 = 0;
                int a_row = 0;
                if (e.kind == PD_ATTN) {
                    if (a_p0 >= a_c1) break;
                    a_n = min(PP, a_c1 - a_p0);
                    a_row = int(head_row) + a_p0;
                    if (FLASH) {
                        // K and V through the tensor maps: whole page, or 16-row tiles
                        const uint32_t tiles = uint32_t(a_n + ATT_TILE - 1) / ATT_TILE;
                        b0 = b1 = a_n == PP ? uint32_t(PAGE_BYTES / 2) : tiles * uint32_t(p.hd / 64) * ATT_TILE * 128u;
                        src0 = src1 = nullptr;
                    } else {
                        b0 = b1 = uint32_t(a_n) * p.hd * 2;
                        src0 = a_kc + (head_row + size_t(a_p0)) * p.hd;
                        src1 = a_vc + (head_row + size_t(a_p0)) * p.hd;
                    }
                    a_p0 += a_n;
                } else if (TC && e.kind == PD_TMA_W) {
                    src0 = nullptr;  // the tensor map and row are in e.src
                    b0 = e.bytes;
                } else {
                    src0 = reinterpret_cast<const void *>(e.src);
                    b0 = e.bytes;
                }
                const uint32_t slot = ppage % NPAGES;
                // a page goes out once its slot is free and fewer than p.max_inflight
                // earlier pages are still landing
                auto can_issue = [&]() -> bool {
                    if (ppage >= NPAGES && !mbar_test(&s.empty[slot], ((ppage / NPAGES) - 1u) & 1u)) return false;
                    if (ppage >= lim) {
                        const uint32_t q = ppage - lim;
                        if (!mbar_test(&s.full[q % NPAGES], (q / NPAGES) & 1u)) return false;
                    }
                    return true;
                };
                if (!can_issue()) {
                    if (pfi < di) pfi = di;  // from the page that is waiting
                    const uint64_t t0 = gtimer();
                    for (uint32_t it = 1;; ++it) {
                        if (can_issue()) break;
                        // while held up, pull the weight pages that come next into L2
                        if (pfi < nd && uint32_t(pfi - di) < l2_ahead) {
                            const PDesc f = dl[pfi++];
                            if (f.kind == PD_WEIGHTS) bulk_prefetch_l2(reinterpret_cast<const void *>(f.src), f.bytes);
                            continue;
                        }
                        __nanosleep(p.producer_sleep_ns);
                        if ((it & 15u) == 0) {
                            if (s.abort) { ok = false; break; }
                            if (gtimer() - t0 > p.timeout_ns) {
                                raise_status(p, s, LL_ERR_DEP_TIMEOUT);
                                ok = false;
                                break;
                            }
                        }
                    }
                    if (!ok) break;
                }
                uint8_t *dst = pages + size_t(slot) * PAGE_BYTES;
                ptrace_put(p, ppage, 0);
                s.slot_page[slot] = ppage;
                mbar_expect_tx(&s.full[slot], b0 + b1);
                if (FLASH && e.kind == PD_ATTN) {
                    // [K | V] x [dim half] x [positions] x 64 dims, swizzled (see attn_tiles)
                    const int dh = p.hd / 64;
                    for (int kv = 0; kv < 2; kv++)
                        for (int h = 0; h < dh; h++) {
                            uint8_t *d = dst + kv * (PAGE_BYTES / 2) + h * PP * 128;
                            if (a_n == PP) {
                                tma_load_2d(d, &a_maps[kv ? TM_V_PAGE : TM_K_PAGE], 64 * h, a_row, &s.full[slot]);
                            } else {
                                for (int j = 0; j < a_n; j += ATT_TILE)
                                    tma_load_2d(d + j * 128, &a_maps[kv ? TM_V_TILE : TM_K_TILE], 64 * h, a_row + j,
                                                &s.full[slot]);
                            }
                        }
                } else if (TC && e.kind == PD_TMA_W) {
                    // a tensor-core page: rows [row, row + nr) of one column chunk of a
                    // matrix, swizzled (see mv_instr_tc)
                    const TensorMap *map = p.wmaps + (e.src >> 40);
                    const int z = int((e.src >> 32) & 0xffu), row = int(uint32_t(e.src & 0xffffffffu));
                    tma_load_3d_hint(dst, map, 0, row, z, &s.full[slot], evict_first);
                } else {
                    if (e.kind == PD_WEIGHTS && p.evict_first) bulk_load_hint(dst, src0, b0, &s.full[slot], evict_first);
                    else bulk_load(dst, src0, b0, &s.full[slot]);
                    if (b1) bulk_load(dst + PAGE_BYTES / 2, src1, b1, &s.full[slot]);
                }
                if (int(e.instr) != last_instr) {
                    trace_put(p, e.instr, 4);
                    last_instr = e.instr;
                }
                trace_put(p, e.instr, 5);
                ++ppage;
                if (e.kind != PD_ATTN) break;
            }
        }
    }
    // Never leave with copies in flight into this block's shared memory: wait for
    // the newest page of every slot (older ones completed before their slot was
    // reused). In a normal step the consumers wait for the same pages.
    const uint32_t first = ppage > NPAGES ? ppage - NPAGES : 0;
    for (uint32_t qi = first; qi < ppage; qi++) {
        uint64_t *bar = &s.full[qi % NPAGES];
        const uint32_t par = (qi / NPAGES) & 1u;
        const uint64_t t0 = gtimer();
        while (!mbar_test(bar, par)) {
            if (gtimer() - t0 > p.timeout_ns) {
                raise_status(p, s, LL_ERR_DEP_TIMEOUT);
                break;
            }
        }
    }
}


// The step the consumers start: its epoch, position and logits, and for every
// step after the first of a launch the token the previous step chose, read from
// its tagged word with acquire order, so that everything the previous step wrote
// (the K/V rows of its position among them) is visible here. The producer may
// only fetch this step's K/V pages after that (s.tok_step).
__device__ bool consumer_step_begin(const KParams &p, Smem &s, int st) {
    if (threadIdx.x == 0) {
        s.c_epoch = p.epoch + static_cast<uint32_t>(st);
        s.c_pos = p.pos + st;
        s.c_logits = p.logits ? p.logits + size_t(st) * size_t(p.V) : nullptr;
        if (st > 0) {
            const uint32_t prev = p.epoch + static_cast<uint32_t>(st - 1);
            uint64_t w = 0, t0 = 0;
            for (uint32_t it = 0;; ++it) {
                w = ld_tag(p.t_token);
                if (tag_ok(w, prev) || poll_give_up(p, s, it, t0)) break;
            }
            asm volatile("fence.acq_rel.gpu;" ::: "memory");
            s.token = static_cast<int32_t>(static_cast<uint32_t>(w));
            // a step without a greedy token (no orderable logit) hands on -1:
            // stop here rather than index the embedding with it
            if (s.token < 0 || s.token >= p.V) raise_status(p, s, LL_ERR_NUMERIC);
            s.tok_step = st;
        }
    }
    return !consumer_any(s.abort);
}

// The (vpl, rw) matrix-vector geometries a kernel carries: all of them (GEO 0), or
// only those of one model family (the host picks such a kernel when a model's
// three input widths all fall in it): the per-warp attention kernel ran 1.5-2.4 %
// faster without the geometries it does not use.
__host__ __device__ constexpr bool geo_has(int geo, int vpl, int rw) {
    return geo == 0 || (geo == GEO_2048 && ((vpl == 2 && rw == 8) || (vpl == 4 && rw == 2))) ||
           (geo == GEO_4096 && ((vpl == 4 && rw == 4) || (vpl == 4 && rw == 1)));
}

template <bool FLASH, bool TC, int GEO>
__device__ bool consumer_step(const KParams &p, Smem &s, uint8_t *pages, const Instr *list, int n, uint32_t &cpage) {
    float best = -INFINITY;
    int best_idx = -1;
    for (int i = 0; i < n; i++) {
        const Instr ins = list[i];
        if (threadIdx.x == 0) trace_put(p, i, 0);
        bool ok;
        if (ins.op == OP_ATTN) {
            ok = attn_instr<FLASH, TC>(p, s, pages, ins, i, cpage);
        } else if constexpr (TC && GEO == GEO_BCC) {
            // two sequences on CUDA-core pages (the host launches this kernel only
            // for the geometries mv_shape_bc gives)
            const MvShape &mv = mv_of(p, ins.op);
            switch (mv.vpl * 16 + mv.rw) {
                case 2 * 16 + 8: ok = mv_instr_bc<2, 8>(p, s, pages, ins, i, cpage, best, best_idx); break;
                case 2 * 16 + 2: ok = mv_instr_bc<2, 2>(p, s, pages, ins, i, cpage, best, best_idx); break;
                default: ok = false; raise_status(p, s, LL_ERR_SHAPE); break;
            }
            if (ok && ins.op == OP_LMHEAD && ins.sub) {
                // lm_finish_b's scratch (s.xin) overlaps the partials the epilogue
                // was reading: every thread is past them first
                consumer_sync();
                lm_finish_b(p, s, best, best_idx);
            }
        } else if constexpr (TC) {
            // every width has tensor-core geometry here (the host launches this
            // kernel only then)
            switch (mv_of(p, ins.op).kc) {
                case 1024: ok = mv_instr_tc<4>(p, s, pages, ins, i, cpage, best, best_idx); break;
                case 2048: ok = mv_instr_tc<8>(p, s, pages, ins, i, cpage, best, best_idx); break;
                default: ok = false; raise_status(p, s, LL_ERR_SHAPE); break;
            }
            if (ok && ins.op == OP_LMHEAD && ins.sub) lm_finish_b(p, s, best, best_idx);
        } else {
            const MvShape &mv = mv_of(p, ins.op);
            switch (mv.vpl * 16 + mv.rw) {
#define LL_MV_CASE(V, R)                                                                     \
    case V * 16 + R:                                                                         \
        if constexpr (geo_has(GEO, V, R)) {                                                  \
            ok = mv_instr<V, R>(p, s, pages, ins, i, cpage, best, best_idx);                 \
        } else {                                                                             \
            ok = false;                                                                      \
            raise_status(p, s, LL_ERR_SHAPE);                                                \
        }                                                                                    \
        break;
                // the (vpl, rw) pairs mv_shape can choose (see mv_combo_ok)
                LL_MV_CASE(1, 8) LL_MV_CASE(2, 8) LL_MV_CASE(3, 1) LL_MV_CASE(3, 2)
                LL_MV_CASE(3, 4) LL_MV_CASE(4, 1) LL_MV_CASE(4, 2) LL_MV_CASE(4, 4)
#undef LL_MV_CASE
                default: ok = false; raise_status(p, s, LL_ERR_SHAPE); break;
            }
            // (an SM's vocabulary rows may come in several pieces: the last one finishes)
            if (ok && ins.op == OP_LMHEAD && ins.sub) lm_finish(p, s, best, best_idx);
        }
        if (ok) ok = instr_sync(s);
        if (!ok) return false;
        if (threadIdx.x == 0) trace_put(p, i, 3);
    }
    return true;
}

template <bool FLASH, bool TC, int GEO>
__device__ void consumer(const KParams &p, Smem &s, uint8_t *pages) {
    const Instr *list = p.instrs + size_t(blockIdx.x) * p.max_instr;
    const int n = p.n_instr[blockIdx.x];
    uint32_t cpage = 0;
    for (int st = 0; st < p.n_steps; st++) {
        if (!(TC ? consumer_step_begin_b(p, s, st) : consumer_step_begin(p, s, st))) return;
        if (!consumer_step<FLASH, TC, GEO>(p, s, pages, list, n, cpage)) return;
    }
}

// FLASH: the attention variant (see attn_instr). TC: the kernel takes the widths
// whose mv.tc is set on tensor-core pages; without it those widths never reach
// it (the host launches the TC kernel exactly when a width has mv.tc), so the
// CUDA-core kernel carries none of that code: its size matters, the step being
// sensitive to instruction-cache misses when the instruction kind changes.
template <bool FLASH, bool TC, int GEO>
__device__ __forceinline__ void megakernel_body(const KParams &p) {
    extern __shared__ __align__(1024) uint8_t smem[];
    uint8_t *pages = smem;
    Smem &s = *reinterpret_cast<Smem *>(smem + NPAGES * PAGE_BYTES);
    if (threadIdx.x == 0) {
        for (int i = 0; i < NPAGES; i++) {
            mbar_init(&s.full[i], 1);
            mbar_init(&s.empty[i], NCW);
            s.pcnt[i] = 0;
            s.slot_page[i] = 0xffffffffu;
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        s.abort = 0;
        s.flag = 0;
        s.token = p.token_dev ? *p.token_dev : p.token;
        s.tok_step = 0;
        s.start_status = ld_relaxed(p.status);
        // swizzled pages (the per-warp attention's KV, tensor-core weight pages) need
        // 1024-byte aligned slots
        if ((FLASH || p.wmaps) && (smem_addr(pages) & 1023u) != 0) {
            atomicCAS(p.status, 0, LL_ERR_DEVICE);
            s.start_status = LL_ERR_DEVICE;
        }
    }
    if (threadIdx.x < 32) reinterpret_cast<uint32_t *>(s.zrow)[threadIdx.x] = 0u;
    {
        const int nl = p.L < SMEM_LAYERS ? p.L : SMEM_LAYERS;
        constexpr int WORDS = sizeof(LayerW) / 8;
        const unsigned long long *src = reinterpret_cast<const unsigned long long *>(p.layers);
        unsigned long long *dst = reinterpret_cast<unsigned long long *>(s.lw);
        for (int i = threadIdx.x; i < nl * WORDS; i += NTHREADS) dst[i] = __ldg(src + i);
    }
    __syncthreads();
    if (s.start_status != 0) return;  // an earlier step failed: do nothing
    if (TC) {  // every sequence's first token (a batch of one: the one token)
        if (threadIdx.x < p.nb) {
            const int t = p.token_dev ? p.token_dev[threadIdx.x] : p.token;
            s.btoken[threadIdx.x] = t;
            if (t < 0 || t >= p.V) s.flag = 1;
        }
        __syncthreads();
        if (s.flag) {
            if (threadIdx.x == 0) atomicCAS(p.status, 0, LL_ERR_ARG);
            return;
        }
    }
    if (s.token < 0 || s.token >= p.V) {
        if (threadIdx.x == 0) atomicCAS(p.status, 0, LL_ERR_ARG);
        return;
    }
    if (threadIdx.x >= NCT) {
        if (threadIdx.x == NCT) producer<FLASH, TC>(p, s, pages);
    } else {
        consumer<FLASH, TC, GEO>(p, s, pages);
    }
}

// One block of NTHREADS per SM: ptxas gives each thread 96 registers (17 warps
// on 4 schedulers: 5 warps share one scheduler's 16K registers).
template <bool FLASH, bool TC, int GEO = 0>
__global__ void __launch_bounds__(NTHREADS, 1) decode_megakernel(const __grid_constant__ KParams p) {
    megakernel_body<FLASH, TC, GEO>(p);
}


}  // namespace
}  // namespace ll
