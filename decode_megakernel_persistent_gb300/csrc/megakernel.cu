// megakernel.cu -- the persistent decode megakernel for sm_103a.
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
//   * counters: instead of kernel boundaries, each finished instruction bumps a
//     global-memory integer and a dependent instruction waits until that
//     integer reaches its target (paragraph on the counter system).
//
// GB300 choices (not from the page): pages are filled with one-dimensional
// bulk async copies (cp.async.bulk) completing on mbarriers; matrix-vector
// products run on CUDA cores with the input vector held in registers; the
// split-KV attention merge is done by the last split to finish (an atomic
// ticket), so no instruction waits for it; the greedy argmax is reduced the
// same way. Every wait is bounded by a time limit.
#include <cuda_runtime.h>
#include <stdint.h>

#include "ll_internal.h"

namespace ll {

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

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
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

__device__ __forceinline__ uint32_t ld_acquire(const uint32_t *p) {
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ int32_t ld_relaxed(const int32_t *p) {
    int32_t v;
    asm volatile("ld.relaxed.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void consumer_sync() {
    asm volatile("bar.sync 1, %0;" ::"n"(NCT) : "memory");
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

struct alignas(16) Smem {
    uint64_t full[NPAGES];   // page filled (tx bytes landed)
    uint64_t empty[NPAGES];  // page released by the consumers
    float red[2][MAX_RPP][NCW];
    float gbuf[GBUF_FLOATS];
    alignas(16) float qs[MAX_GQA][MAX_HD];
    alignas(16) float sc[MAX_GQA][128];
    alignas(16) uint16_t knew[MAX_HD];
    alignas(16) uint16_t vnew[MAX_HD];
    float m_run[MAX_GQA], l_run[MAX_GQA], alpha[MAX_GQA];
    float nred[NCW];
    unsigned long long kred[NCW];
    int32_t token;
    int32_t start_status;
    volatile int32_t flag;
    volatile int32_t abort;
};

constexpr int SMEM_BYTES = NPAGES * PAGE_BYTES + static_cast<int>(sizeof(Smem));

// ---------------------------------------------------------------------------------
// Bounded waits. A wait that runs past p.timeout_ns records LL_ERR_DEP_TIMEOUT in
// the status word; any wait that sees a nonzero status gives up as well.

__device__ __forceinline__ void raise_status(const KParams &p, Smem &s, int32_t code) {
    atomicCAS(p.status, 0, code);
    s.abort = 1;
}

__device__ bool wait_counter(const KParams &p, Smem &s, const uint32_t *ctr, uint32_t target) {
    if (static_cast<int32_t>(ld_acquire(ctr) - target) >= 0) return true;
    const uint64_t t0 = gtimer();
    for (uint32_t it = 1;; ++it) {
        if (static_cast<int32_t>(ld_acquire(ctr) - target) >= 0) return true;
        if ((it & 31u) == 0) {
            if (s.abort) return false;
            if (ld_relaxed(p.status) != 0) {
                s.abort = 1;
                return false;
            }
            if (gtimer() - t0 > p.timeout_ns) {
                raise_status(p, s, LL_ERR_DEP_TIMEOUT);
                return false;
            }
        }
    }
}

__device__ bool wait_page(const KParams &p, Smem &s, uint64_t *bar, uint32_t parity) {
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

// Consumer-side dependency wait: thread 0 polls, everyone learns the outcome.
__device__ bool dep_wait(const KParams &p, Smem &s, const Instr &ins) {
    if (ins.wait_ctr >= 0 && threadIdx.x == 0) {
        wait_counter(p, s, p.ctr + size_t(ins.wait_ctr) * CTR_STRIDE, p.epoch * ins.wait_count);
    }
    consumer_sync();
    return !s.abort;
}

__device__ void signal_done(const KParams &p, const Instr &ins) {
    consumer_sync();
    if (threadIdx.x == 0 && ins.sig_ctr >= 0) {
        __threadfence();
        atomicAdd(p.ctr + size_t(ins.sig_ctr) * CTR_STRIDE, 1u);
    }
}

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

__device__ int mv_segments(const KParams &p, const Instr &ins, Seg *seg) {
    const LayerW *lw = ins.op == OP_LMHEAD ? nullptr : &p.layers[ins.layer];
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
__device__ __forceinline__ void attn_range(const KParams &p, int c, int &c0, int &c1) {
    const long long S = p.attn_splits;
    c0 = static_cast<int>((static_cast<long long>(c) * p.pos) / S);
    c1 = static_cast<int>((static_cast<long long>(c + 1) * p.pos) / S);
}

__device__ __forceinline__ int attn_pp(const KParams &p) { return PAGE_BYTES / (4 * p.hd); }

// Lane-held input vector: element (sw*32*VPL + j*32 + lane)*8 + e sits in xr[j*8+e].
template <int VPL>
__device__ void load_input(const KParams &p, Smem &s, const Instr &ins, const MvShape &mv,
                           float (&xr)[VPL * 8]) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int sw = warp % mv.ws;
    const uint16_t *gain = nullptr;
    const float *src = nullptr;
    const uint16_t *src16 = nullptr;
    switch (ins.op) {
        case OP_QKV:
            gain = p.layers[ins.layer].attn_norm;
            if (ins.layer == 0) src16 = p.embed + size_t(s.token) * p.H;
            else src = p.x;
            break;
        case OP_GATEUP: gain = p.layers[ins.layer].mlp_norm; src = p.x; break;
        case OP_LMHEAD: gain = p.final_norm; src = p.x; break;
        case OP_OPROJ: src = p.o; break;
        default: src = p.act; break;
    }
#pragma unroll
    for (int j = 0; j < VPL; j++) {
        const int v = sw * 32 * VPL + j * 32 + lane;
        if (src16) {
            uint4 u = __ldg(reinterpret_cast<const uint4 *>(src16) + v);
            xr[j * 8 + 0] = bf_lo(u.x); xr[j * 8 + 1] = bf_hi(u.x);
            xr[j * 8 + 2] = bf_lo(u.y); xr[j * 8 + 3] = bf_hi(u.y);
            xr[j * 8 + 4] = bf_lo(u.z); xr[j * 8 + 5] = bf_hi(u.z);
            xr[j * 8 + 6] = bf_lo(u.w); xr[j * 8 + 7] = bf_hi(u.w);
        } else {
            float4 a = __ldcg(reinterpret_cast<const float4 *>(src) + 2 * v);
            float4 b = __ldcg(reinterpret_cast<const float4 *>(src) + 2 * v + 1);
            xr[j * 8 + 0] = a.x; xr[j * 8 + 1] = a.y; xr[j * 8 + 2] = a.z; xr[j * 8 + 3] = a.w;
            xr[j * 8 + 4] = b.x; xr[j * 8 + 5] = b.y; xr[j * 8 + 6] = b.z; xr[j * 8 + 7] = b.w;
        }
    }
    if (!gain) return;
    // RMSNorm: the warps w < ws together hold every element once.
    float ss = 0.f;
#pragma unroll
    for (int e = 0; e < VPL * 8; e++) ss = fmaf(xr[e], xr[e], ss);
    ss = warp_sum(ss);
    if (lane == 0 && warp < mv.ws) s.nred[warp] = ss;
    consumer_sync();
    float tot = 0.f;
    for (int w = 0; w < mv.ws; w++) tot += s.nred[w];
    const float r = 1.0f / sqrtf(tot / static_cast<float>(mv.K) + p.eps);
#pragma unroll
    for (int j = 0; j < VPL; j++) {
        const int v = sw * 32 * VPL + j * 32 + lane;
        uint4 u = __ldg(reinterpret_cast<const uint4 *>(gain) + v);
        const uint32_t g[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int q = 0; q < 4; q++) {
            xr[j * 8 + 2 * q] = xr[j * 8 + 2 * q] * r * bf_lo(g[q]);
            xr[j * 8 + 2 * q + 1] = xr[j * 8 + 2 * q + 1] * r * bf_hi(g[q]);
        }
    }
}

template <int VPL>
__device__ bool mv_instr(const KParams &p, Smem &s, uint8_t *pages, const Instr &ins, uint32_t &cpage,
                         float &best, int &best_idx) {
    const MvShape &mv = mv_of(p, ins.op);
    Seg seg[3];
    const int nseg = mv_segments(p, ins, seg);
    if (nseg == 0) return true;  // no rows here: nothing to read or wait for
    if (!dep_wait(p, s, ins)) return false;

    float xr[VPL * 8];
    load_input<VPL>(p, s, ins, mv, xr);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, tid = threadIdx.x;
    const int sw = warp % mv.ws, rg = warp / mv.ws, ngroups = NCW / mv.ws;
    const size_t row_bytes = size_t(mv.K) * 2;

    for (int si = 0; si < nseg; si++) {
        const Seg sg = seg[si];
        for (int pr = 0; pr < sg.nrows; pr += mv.rpp) {
            const int nr = min(mv.rpp, sg.nrows - pr);
            const uint32_t slot = cpage % NPAGES, par = (cpage / NPAGES) & 1u;
            if (!wait_page(p, s, &s.full[slot], par)) return false;
            const uint8_t *page = pages + size_t(slot) * PAGE_BYTES;
            float(*red)[NCW] = s.red[cpage & 1u];
            for (int rl = rg; rl < nr; rl += ngroups) {
                const uint4 *wrow = reinterpret_cast<const uint4 *>(page + size_t(rl) * row_bytes);
                uint4 wv[VPL];
#pragma unroll
                for (int j = 0; j < VPL; j++) wv[j] = wrow[sw * 32 * VPL + j * 32 + lane];
                float a0 = 0.f, a1 = 0.f;
#pragma unroll
                for (int j = 0; j < VPL; j++) {
                    a0 = fmaf(bf_lo(wv[j].x), xr[j * 8 + 0], a0);
                    a1 = fmaf(bf_hi(wv[j].x), xr[j * 8 + 1], a1);
                    a0 = fmaf(bf_lo(wv[j].y), xr[j * 8 + 2], a0);
                    a1 = fmaf(bf_hi(wv[j].y), xr[j * 8 + 3], a1);
                    a0 = fmaf(bf_lo(wv[j].z), xr[j * 8 + 4], a0);
                    a1 = fmaf(bf_hi(wv[j].z), xr[j * 8 + 5], a1);
                    a0 = fmaf(bf_lo(wv[j].w), xr[j * 8 + 6], a0);
                    a1 = fmaf(bf_hi(wv[j].w), xr[j * 8 + 7], a1);
                }
                const float acc = warp_sum(a0 + a1);
                if (lane == 0) red[rl][sw] = acc;
            }
            consumer_sync();
            if (tid == 0) mbar_arrive(&s.empty[slot]);  // page bytes no longer needed
            ++cpage;
            if (tid < nr) {
                float y = 0.f;
                for (int w = 0; w < mv.ws; w++) y += red[tid][w];
                const int row = sg.row0 + pr + tid;  // row within the matrix
                switch (sg.kind) {
                    case OUT_QKV: p.qkv[sg.out0 + row] = y; break;
                    case OUT_RESID: {
                        float base = (ins.op == OP_OPROJ && ins.layer == 0)
                                         ? bf16_to_f(p.embed[size_t(s.token) * p.H + row])
                                         : __ldcg(p.x + row);
                        p.x[row] = base + y;
                        break;
                    }
                    case OUT_GATE: s.gbuf[row - ins.r0] = y; break;
                    case OUT_UP: {
                        const float g = s.gbuf[row - ins.r0];
                        p.act[row] = g / (1.0f + expf(-g)) * y;
                        break;
                    }
                    default:  // OUT_LOGITS
                        if (p.logits) p.logits[row] = y;
                        if (y > best) { best = y; best_idx = row; }
                        break;
                }
            }
        }
    }
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
        s.flag = (old + 1u == p.epoch * static_cast<uint32_t>(p.nsm)) ? 1 : 0;
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
        const int32_t tok = static_cast<int32_t>(0xffffffffu - static_cast<uint32_t>(m & 0xffffffffu));
        p.token_out[0] = tok;
        if (p.next_token_dev) *p.next_token_dev = tok;
    }
}

// ---------------------------------------------------------------------------------
// Attention instruction: one KV head g, one split c of the cached positions; the
// split that owns position pos also folds in the new k, v and writes them to the
// cache. Partial (o, m, l) go to global memory; the last split of the head merges.

__device__ void attn_block(const KParams &p, Smem &s, const uint16_t *K, const uint16_t *Vv, int n,
                           float (&oacc)[4], int G) {
    const int hd = p.hd, tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int nch = hd / 8;
    // scores: one position per thread, all G heads; chunk order rotated by position
    // so that the 16-byte reads of a warp spread over all banks
    if (tid < n) {
        const uint4 *krow = reinterpret_cast<const uint4 *>(K + size_t(tid) * hd);
        float acc[MAX_GQA];
#pragma unroll
        for (int h = 0; h < MAX_GQA; h++) acc[h] = 0.f;
        for (int i = 0; i < nch; i++) {
            const int c = (i + tid) % nch;
            const uint4 u = krow[c];
            const float k8[8] = {bf_lo(u.x), bf_hi(u.x), bf_lo(u.y), bf_hi(u.y),
                                 bf_lo(u.z), bf_hi(u.z), bf_lo(u.w), bf_hi(u.w)};
#pragma unroll
            for (int h = 0; h < MAX_GQA; h++) {
                if (h < G) {
                    const float4 qa = *reinterpret_cast<const float4 *>(&s.qs[h][c * 8]);
                    const float4 qb = *reinterpret_cast<const float4 *>(&s.qs[h][c * 8 + 4]);
                    float a = acc[h];
                    a = fmaf(qa.x, k8[0], a); a = fmaf(qa.y, k8[1], a);
                    a = fmaf(qa.z, k8[2], a); a = fmaf(qa.w, k8[3], a);
                    a = fmaf(qb.x, k8[4], a); a = fmaf(qb.y, k8[5], a);
                    a = fmaf(qb.z, k8[6], a); a = fmaf(qb.w, k8[7], a);
                    acc[h] = a;
                }
            }
        }
#pragma unroll
        for (int h = 0; h < MAX_GQA; h++)
            if (h < G) s.sc[h][tid] = acc[h];
    }
    consumer_sync();
    // online softmax statistics: warp h handles head h
    if (warp < G) {
        const int h = warp;
        float mx = -INFINITY;
        for (int j = lane; j < n; j += 32) mx = fmaxf(mx, s.sc[h][j]);
        mx = warp_max(mx);
        const float m_old = s.m_run[h];
        const float m_new = fmaxf(m_old, mx);
        float sum = 0.f;
        for (int j = lane; j < n; j += 32) {
            const float e = expf(s.sc[h][j] - m_new);
            s.sc[h][j] = e;
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
    // P V: one (head, dim) pair per accumulator slot
#pragma unroll
    for (int k = 0; k < 4; k++) {
        const int pi = tid + k * NCT;
        if (pi < G * hd) {
            const int h = pi / hd, d = pi % hd;
            float a = oacc[k] * s.alpha[h];
            for (int j = 0; j < n; j++) a = fmaf(s.sc[h][j], bf16_to_f(Vv[size_t(j) * hd + d]), a);
            oacc[k] = a;
        }
    }
    consumer_sync();
}

__device__ bool attn_instr(const KParams &p, Smem &s, uint8_t *pages, const Instr &ins, uint32_t &cpage) {
    if (!dep_wait(p, s, ins)) return false;
    const int g = ins.r0, c = ins.r1, S = p.attn_splits, l = ins.layer;
    const int hd = p.hd, half = hd / 2, G = p.nq / p.nkv, tid = threadIdx.x;
    const int qd = p.nq * p.hd, kd = p.nkv * p.hd;
    const float scale = 1.0f / sqrtf(static_cast<float>(hd));
    const float2 *cs = p.rope_cs + size_t(p.pos) * half;
    // RoPE ("rotate half") on the group's queries and on the new key
    for (int t = tid; t < G * half; t += NCT) {
        const int h = t / half, i = t % half;
        const float *q = p.qkv + size_t(g * G + h) * hd;
        const float a = __ldcg(q + i), b = __ldcg(q + i + half);
        const float2 r = cs[i];
        s.qs[h][i] = (a * r.x - b * r.y) * scale;
        s.qs[h][i + half] = (a * r.y + b * r.x) * scale;
    }
    for (int i = tid; i < half; i += NCT) {
        const float *k = p.qkv + qd + size_t(g) * hd;
        const float a = __ldcg(k + i), b = __ldcg(k + i + half);
        const float2 r = cs[i];
        s.knew[i] = f_to_bf16(a * r.x - b * r.y);
        s.knew[i + half] = f_to_bf16(a * r.y + b * r.x);
    }
    for (int d = tid; d < hd; d += NCT) s.vnew[d] = f_to_bf16(__ldcg(p.qkv + qd + kd + size_t(g) * hd + d));
    if (tid < G) {
        s.m_run[tid] = -INFINITY;
        s.l_run[tid] = 0.f;
    }
    consumer_sync();
    const size_t head_base = (size_t(l) * p.nkv + g) * size_t(p.max_seq) * hd;
    if (c == S - 1) {  // this split owns position pos: write the new entry
        for (int d = tid; d < hd; d += NCT) {
            p.k_cache[head_base + size_t(p.pos) * hd + d] = s.knew[d];
            p.v_cache[head_base + size_t(p.pos) * hd + d] = s.vnew[d];
        }
    }
    float oacc[4] = {0.f, 0.f, 0.f, 0.f};
    int c0, c1;
    attn_range(p, c, c0, c1);
    const int PP = attn_pp(p);
    for (int p0 = c0; p0 < c1; p0 += PP) {
        const int n = min(PP, c1 - p0);
        const uint32_t slot = cpage % NPAGES, par = (cpage / NPAGES) & 1u;
        if (!wait_page(p, s, &s.full[slot], par)) return false;
        const uint16_t *pg = reinterpret_cast<const uint16_t *>(pages + size_t(slot) * PAGE_BYTES);
        attn_block(p, s, pg, pg + PAGE_BYTES / 4, n, oacc, G);  // V at half a page
        if (tid == 0) mbar_arrive(&s.empty[slot]);
        ++cpage;
    }
    if (c == S - 1) attn_block(p, s, s.knew, s.vnew, 1, oacc, G);

    // partials: part[(qhead * S + c) * (hd + 2) + {d, hd: m, hd+1: l}]
    const int stride = hd + 2;
#pragma unroll
    for (int k = 0; k < 4; k++) {
        const int pi = tid + k * NCT;
        if (pi < G * hd) {
            const int h = pi / hd, d = pi % hd;
            p.part[(size_t(g * G + h) * S + c) * stride + d] = oacc[k];
        }
    }
    if (tid < G) {
        p.part[(size_t(g * G + tid) * S + c) * stride + hd] = s.m_run[tid];
        p.part[(size_t(g * G + tid) * S + c) * stride + hd + 1] = s.l_run[tid];
    }
    consumer_sync();
    if (tid == 0) {
        __threadfence();
        const int tk = CtrLayout::attn_ticket(p.L, l, g, p.nkv);
        const uint32_t old = atomicAdd(p.ctr + size_t(tk) * CTR_STRIDE, 1u);
        s.flag = (old + 1u == p.epoch * static_cast<uint32_t>(S)) ? 1 : 0;
        __threadfence();
    }
    consumer_sync();
    if (s.flag) {  // last split of this KV head: merge all splits
        for (int pi = tid; pi < G * hd; pi += NCT) {
            const int h = pi / hd, d = pi % hd;
            const float *base = p.part + size_t(g * G + h) * S * stride;
            float M = -INFINITY;
            for (int j = 0; j < S; j++) M = fmaxf(M, __ldcg(base + size_t(j) * stride + hd));
            float L = 0.f, O = 0.f;
            for (int j = 0; j < S; j++) {
                const float mj = __ldcg(base + size_t(j) * stride + hd);
                if (mj == -INFINITY) continue;
                const float w = expf(mj - M);
                L = fmaf(__ldcg(base + size_t(j) * stride + hd + 1), w, L);
                O = fmaf(__ldcg(base + size_t(j) * stride + d), w, O);
            }
            p.o[size_t(g * G + h) * hd + d] = O / L;
        }
        signal_done(p, ins);
    }
    return true;
}

// ---------------------------------------------------------------------------------
// Producer: walks the same instruction list and streams every page in order.

__device__ bool issue_page(const KParams &p, Smem &s, uint8_t *pages, uint32_t &ppage, const void *src0,
                           uint32_t bytes0, const void *src1, uint32_t bytes1) {
    const uint32_t slot = ppage % NPAGES;
    if (ppage >= NPAGES) {
        if (!wait_page(p, s, &s.empty[slot], ((ppage / NPAGES) - 1u) & 1u)) return false;
    }
    uint8_t *dst = pages + size_t(slot) * PAGE_BYTES;
    mbar_expect_tx(&s.full[slot], bytes0 + bytes1);
    if (bytes0) bulk_load(dst, src0, bytes0, &s.full[slot]);
    if (bytes1) bulk_load(dst + PAGE_BYTES / 2, src1, bytes1, &s.full[slot]);
    ++ppage;
    return true;
}

__device__ void producer(const KParams &p, Smem &s, uint8_t *pages) {
    const Instr *list = p.instrs + size_t(blockIdx.x) * p.max_instr;
    const int n = p.n_instr[blockIdx.x];
    uint32_t ppage = 0;
    bool ok = true;
    for (int i = 0; i < n && ok; i++) {
        const Instr ins = list[i];
        if (ins.op == OP_ATTN) {
            int c0, c1;
            attn_range(p, ins.r1, c0, c1);
            const int PP = attn_pp(p), hd = p.hd;
            const size_t head_base = (size_t(ins.layer) * p.nkv + ins.r0) * size_t(p.max_seq) * hd;
            for (int p0 = c0; p0 < c1 && ok; p0 += PP) {
                const int nn = min(PP, c1 - p0);
                const uint32_t b = uint32_t(nn) * hd * 2;
                ok = issue_page(p, s, pages, ppage, p.k_cache + head_base + size_t(p0) * hd, b,
                                p.v_cache + head_base + size_t(p0) * hd, b);
            }
            continue;
        }
        const MvShape &mv = mv_of(p, ins.op);
        Seg seg[3];
        const int nseg = mv_segments(p, ins, seg);
        for (int si = 0; si < nseg && ok; si++) {
            for (int pr = 0; pr < seg[si].nrows && ok; pr += mv.rpp) {
                const int nr = min(mv.rpp, seg[si].nrows - pr);
                const uint16_t *src = seg[si].w + size_t(seg[si].row0 + pr) * mv.K;
                ok = issue_page(p, s, pages, ppage, src, uint32_t(nr) * mv.K * 2, nullptr, 0);
            }
        }
    }
    // Never leave with copies in flight into this block's shared memory: wait for
    // the newest page of every slot (older ones completed before their slot was
    // reused). In a normal step the consumers wait for the same pages.
    const uint32_t first = ppage > NPAGES ? ppage - NPAGES : 0;
    for (uint32_t q = first; q < ppage; q++) {
        uint64_t *bar = &s.full[q % NPAGES];
        const uint32_t par = (q / NPAGES) & 1u;
        const uint64_t t0 = gtimer();
        while (!mbar_test(bar, par)) {
            if (gtimer() - t0 > p.timeout_ns) {
                raise_status(p, s, LL_ERR_DEP_TIMEOUT);
                break;
            }
        }
    }
}

__device__ void consumer(const KParams &p, Smem &s, uint8_t *pages) {
    const Instr *list = p.instrs + size_t(blockIdx.x) * p.max_instr;
    const int n = p.n_instr[blockIdx.x];
    uint32_t cpage = 0;
    float best = -INFINITY;
    int best_idx = -1;
    for (int i = 0; i < n; i++) {
        const Instr ins = list[i];
        bool ok;
        if (ins.op == OP_ATTN) {
            ok = attn_instr(p, s, pages, ins, cpage);
        } else {
            switch (mv_of(p, ins.op).vpl) {
                case 1: ok = mv_instr<1>(p, s, pages, ins, cpage, best, best_idx); break;
                case 2: ok = mv_instr<2>(p, s, pages, ins, cpage, best, best_idx); break;
                case 3: ok = mv_instr<3>(p, s, pages, ins, cpage, best, best_idx); break;
                case 4: ok = mv_instr<4>(p, s, pages, ins, cpage, best, best_idx); break;
                case 5: ok = mv_instr<5>(p, s, pages, ins, cpage, best, best_idx); break;
                case 6: ok = mv_instr<6>(p, s, pages, ins, cpage, best, best_idx); break;
                case 7: ok = mv_instr<7>(p, s, pages, ins, cpage, best, best_idx); break;
                default: ok = mv_instr<8>(p, s, pages, ins, cpage, best, best_idx); break;
            }
            if (ok && ins.op == OP_LMHEAD) {
                lm_finish(p, s, best, best_idx);
            } else if (ok && ins.op != OP_ATTN) {
                signal_done(p, ins);
            }
        }
        if (!ok) return;
    }
}

__global__ void __launch_bounds__(NTHREADS, 1) decode_megakernel(const __grid_constant__ KParams p) {
    extern __shared__ __align__(1024) uint8_t smem[];
    uint8_t *pages = smem;
    Smem &s = *reinterpret_cast<Smem *>(smem + NPAGES * PAGE_BYTES);
    if (threadIdx.x == 0) {
        for (int i = 0; i < NPAGES; i++) {
            mbar_init(&s.full[i], 1);
            mbar_init(&s.empty[i], 1);
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        s.abort = 0;
        s.flag = 0;
        s.token = p.token_dev ? *p.token_dev : p.token;
        s.start_status = ld_relaxed(p.status);
    }
    __syncthreads();
    if (s.start_status != 0) return;  // an earlier step failed: do nothing
    if (s.token < 0 || s.token >= p.V) {
        if (threadIdx.x == 0) atomicCAS(p.status, 0, LL_ERR_ARG);
        return;
    }
    if (threadIdx.x >= NCT) {
        if (threadIdx.x == NCT) producer(p, s, pages);
    } else {
        consumer(p, s, pages);
    }
}

int megakernel_smem_bytes() { return SMEM_BYTES; }

int megakernel_prepare(int smem_bytes) {
    cudaError_t e = cudaFuncSetAttribute(decode_megakernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         smem_bytes);
    if (e != cudaSuccess) return LL_ERR_CUDA;
    int blocks = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&blocks, decode_megakernel, NTHREADS, smem_bytes);
    if (e != cudaSuccess) return LL_ERR_CUDA;
    return blocks >= 1 ? LL_OK : LL_ERR_DEVICE;
}

int launch_megakernel(const KParams &p, void *stream, int smem_bytes) {
    void *args[] = {const_cast<KParams *>(&p)};
    cudaError_t e = cudaLaunchCooperativeKernel(reinterpret_cast<const void *>(decode_megakernel),
                                                dim3(p.nsm), dim3(NTHREADS), args, size_t(smem_bytes),
                                                static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? LL_OK : LL_ERR_CUDA;
}

}  // namespace ll
