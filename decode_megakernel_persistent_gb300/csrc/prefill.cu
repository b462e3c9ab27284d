// prefill.cu -- a prompt's positions through the model at once (ll_prefill).
//
// The page "Hazy Research Llama-3.2-1B Megakernel" is about decode; a prompt is
// the step before it: every position of the prompt goes through every layer,
// which turns each projection into a matrix product of (positions x width) by
// the weight matrix, filling the KV cache for the decode steps that follow.
// Here every projection is a tcgen05 GEMM (the fifth-generation tensor cores):
// TMA brings 128 x 64 bf16 tiles of both operands into shared memory in the
// 128-byte swizzle through a 4-stage mbarrier pipeline, one thread issues
// tcgen05.mma (M = 128 positions, N = 128 outputs, K = 16 per instruction) into a
// tensor-memory accumulator, and the four warps read it back with tcgen05.ld for
// the epilogue. The decode path keeps activations in fp32; a bf16 product with
// one term of them misses the logits' bar (and with two, bf16 roundings of the
// K/V written to the cache flip measurably more often than in fp32), so each
// activation matrix enters as three bf16 terms (t0 = bf16(x), t1 = bf16(x - t0),
// t2 = bf16(x - t0 - t1): the 24 bits of an fp32 value) and all their products
// accumulate in the same tensor-memory tile: the GEMM runs its K loop three
// times.
//
// Per layer: RMSNorm into the two terms; Q, K, V GEMMs; RoPE with the K/V
// rounded to bf16 into the cache; causal attention over the cache (CUDA cores,
// one warp per query position and head); O GEMM added into the residual;
// RMSNorm; gate GEMM; up GEMM whose epilogue forms silu(gate) * up in two terms;
// down GEMM added into the residual. Then the last position's final norm, LM
// head and argmax.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <algorithm>
#include <cstring>

#include "ll_internal.h"

namespace ll {
namespace {

constexpr int GM = 128, GN = 128, GK = 64, GSTAGES = 4, GTHREADS = 128;
constexpr int NTERMS = 3;  // bf16 terms of an activation
constexpr uint32_t GTILE = GM * GK * 2;  // bytes of one 128 x 64 bf16 tile (A and B alike)
constexpr int GEMM_SMEM = GSTAGES * 2 * int(GTILE) + 1024;

__device__ __forceinline__ uint32_t saddr(const void *p) { return static_cast<uint32_t>(__cvta_generic_to_shared(p)); }

__device__ __forceinline__ uint64_t now_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ bool mbar_try(uint64_t *bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\tselp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(saddr(bar)), "r"(parity)
        : "memory");
    return done != 0;
}

// Bounded wait: false (and the status word set) once timeout_ns pass.
__device__ bool mbar_wait(uint64_t *bar, uint32_t parity, uint64_t timeout_ns, int32_t *status, volatile int *err) {
    if (mbar_try(bar, parity)) return true;
    const uint64_t t0 = now_ns();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try(bar, parity)) return true;
        if ((it & 63u) == 0) {
            if (*err) return false;
            if (now_ns() - t0 > timeout_ns) {
                atomicCAS(status, 0, LL_ERR_DEP_TIMEOUT);
                *err = 1;
                return false;
            }
        }
    }
}

// Shared-memory matrix descriptor of a K-major tile in the 128-byte swizzle: rows
// of 128 bytes (64 bf16), 8-row groups 1024 bytes apart; start address, leading
// byte offset (unused with this swizzle), stride byte offset, descriptor version
// 1, layout type 2 (128-byte swizzle). Advancing K by 16 elements adds 32 bytes
// (2 in the start-address field).
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t addr) {
    uint64_t d = 0;
    d |= uint64_t((addr >> 4) & 0x3fffu);
    d |= uint64_t(1u) << 16;             // leading byte offset (ignored for swizzled K-major)
    d |= uint64_t(1024u >> 4) << 32;     // stride byte offset: next 8-row group
    d |= uint64_t(1u) << 46;             // descriptor version
    d |= uint64_t(2u) << 61;             // 128-byte swizzle
    return d;
}

// Instruction descriptor of kind::f16: fp32 accumulator, bf16 A and B, both
// K-major, N and M as given.
__host__ __device__ constexpr uint32_t idesc_bf16(int m, int n) {
    return (1u << 4) | (1u << 7) | (1u << 10) | (uint32_t(n >> 3) << 17) | (uint32_t(m >> 4) << 24);
}

__device__ __forceinline__ void tma2d(uint32_t dst, const TensorMap *map, int x, int y, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
            dst),
        "l"(reinterpret_cast<unsigned long long>(map)), "r"(x), "r"(y), "r"(saddr(bar))
        : "memory");
}

enum : int { EPI_STORE = 0, EPI_ADD = 1, EPI_SILU_MUL = 2 };

struct GemmArgs {
    TensorMap a[NTERMS], b;   // A terms [rows][K] and B [N][K], bf16, K-major, boxes 64 x 128, 128-byte swizzle
    int M, N, K;              // positions, outputs, inner width (K a multiple of 64)
    float *c;                 // [M][ldc] fp32: EPI_STORE c = A B^T, EPI_ADD c += A B^T
    int ldc;
    const float *gate;        // EPI_SILU_MUL: gate [M][ldc]; act = silu(gate) * (A B^T) as NTERMS bf16 terms
    uint16_t *act[NTERMS];
    int32_t *status;
    uint64_t timeout_ns;
};

// One 128 x 128 tile of C per block: warp 0 lane 0 feeds the pipeline with TMA,
// warp 1 lane 0 issues the MMAs, all four warps run the epilogue (warp w owns
// tensor-memory lanes, i.e. tile rows, 32 w .. 32 w + 31).
template <int EPI>
__global__ void __launch_bounds__(GTHREADS, 1) k_gemm(const __grid_constant__ GemmArgs g) {
    extern __shared__ __align__(1024) uint8_t gsm[];
    uint8_t *tiles = gsm;
    uint64_t *full = reinterpret_cast<uint64_t *>(gsm + GSTAGES * 2 * GTILE);
    uint64_t *empty = full + GSTAGES;
    uint64_t *done = empty + GSTAGES;
    volatile uint32_t *tmem_slot = reinterpret_cast<volatile uint32_t *>(done + 1);
    volatile int *err = reinterpret_cast<volatile int *>(done + 2);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int m0 = blockIdx.y * GM, n0 = blockIdx.x * GN;
    const int nk = g.K / GK, iters = NTERMS * nk;  // the K loop of term 0, then of term 1, ...
    if (threadIdx.x == 0) {
        for (int s = 0; s < GSTAGES; s++) {
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(saddr(&full[s])) : "memory");
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(saddr(&empty[s])) : "memory");
        }
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(saddr(done)) : "memory");
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        *err = 0;
    }
    if (warp == 0) {  // 128 fp32 columns of tensor memory: the 128 x 128 accumulator
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 128;" ::"r"(
                         saddr(const_cast<uint32_t *>(tmem_slot)))
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    const uint32_t tmem = *tmem_slot;

    if (warp == 0 && lane == 0) {
        int sent = 0;
        for (int it = 0; it < iters; it++) {
            const int s = it % GSTAGES;
            if (it >= GSTAGES && !mbar_wait(&empty[s], ((it / GSTAGES) - 1) & 1, g.timeout_ns, g.status, err)) break;
            asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(saddr(&full[s])),
                         "r"(2 * GTILE)
                         : "memory");
            const int kc = (it % nk) * GK;
            const uint32_t a_dst = saddr(tiles + size_t(s) * 2 * GTILE);
            tma2d(a_dst, &g.a[it / nk], kc, m0, &full[s]);
            tma2d(a_dst + GTILE, &g.b, kc, n0, &full[s]);
            sent++;
        }
        // never leave with copies in flight into this block's shared memory (after
        // an error; normally the products have consumed every stage)
        for (int q = sent > GSTAGES ? sent - GSTAGES : 0; q < sent; q++) {
            const uint64_t t0 = now_ns();
            while (!mbar_try(&full[q % GSTAGES], (q / GSTAGES) & 1) && now_ns() - t0 < g.timeout_ns) {
            }
        }
    } else if (warp == 1 && lane == 0) {
        constexpr uint32_t idesc = idesc_bf16(GM, GN);
        int issued = 0;
        for (int it = 0; it < iters; it++) {
            const int s = it % GSTAGES;
            if (!mbar_wait(&full[s], (it / GSTAGES) & 1, g.timeout_ns, g.status, err)) break;
            asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
            const uint32_t a_addr = saddr(tiles + size_t(s) * 2 * GTILE);
            const uint64_t ad = smem_desc_sw128(a_addr), bd = smem_desc_sw128(a_addr + GTILE);
#pragma unroll
            for (int kk = 0; kk < GK / 16; kk++) {
                const uint32_t acc = (it | kk) != 0 ? 1u : 0u;
                asm volatile(
                    "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
                    "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem),
                    "l"(ad + uint64_t(2 * kk)), "l"(bd + uint64_t(2 * kk)), "r"(idesc), "r"(acc)
                    : "memory");
            }
            // the stage is free once these products have read it
            asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                             saddr(&empty[s]))
                         : "memory");
            issued++;
        }
        // the accumulator is complete once every product issued so far is
        asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(saddr(done))
                     : "memory");
        (void)issued;
    }
    __syncwarp();
    const bool ok = mbar_wait(done, 0, g.timeout_ns, g.status, err) && !*err;
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    const int row = m0 + warp * 32 + lane;
    if (ok) {
#pragma unroll 1
        for (int c0 = 0; c0 < GN; c0 += 16) {
            uint32_t r[16];
            const uint32_t taddr = tmem + (uint32_t(warp * 32) << 16) + uint32_t(c0);
            asm volatile(
                "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, "
                "%14, %15}, [%16];"
                : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
                  "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
                : "r"(taddr));
            asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
            if (row >= g.M) continue;
#pragma unroll
            for (int j = 0; j < 16; j++) {
                const int col = n0 + c0 + j;
                if (col >= g.N) break;
                const float y = __uint_as_float(r[j]);
                const size_t at = size_t(row) * g.ldc + col;
                if (EPI == EPI_STORE) {
                    g.c[at] = y;
                } else if (EPI == EPI_ADD) {
                    g.c[at] += y;
                } else {
                    const float z = g.gate[at];
                    float a = z / (1.0f + expf(-z)) * y;
#pragma unroll
                    for (int q = 0; q < NTERMS; q++) {
                        const __nv_bfloat16 tq = __float2bfloat16_rn(a);
                        g.act[q][at] = __bfloat16_as_ushort(tq);
                        a -= __bfloat162float(tq);
                    }
                }
            }
        }
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    if (warp == 0) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 128;" ::"r"(tmem) : "memory");
}

// x[t] = E[tokens[t]] (fp32), tokens checked.
__global__ void k_pf_embed(const uint16_t *E, const int32_t *tokens, int n, int H, int V, float *x, int32_t *status) {
    const int t = blockIdx.x;
    const int tok = tokens[t];
    if (tok < 0 || tok >= V) {
        if (threadIdx.x == 0) atomicCAS(status, 0, LL_ERR_ARG);
        return;
    }
    for (int i = threadIdx.x; i < H; i += blockDim.x)
        x[size_t(t) * H + i] = __uint_as_float(uint32_t(E[size_t(tok) * H + i]) << 16);
}

// The NTERMS bf16 terms of v into t[q][at].
__device__ __forceinline__ void put_terms(float v, uint16_t *const *t, size_t at) {
#pragma unroll
    for (int q = 0; q < NTERMS; q++) {
        const __nv_bfloat16 b = __float2bfloat16_rn(v);
        t[q][at] = __bfloat16_as_ushort(b);
        v -= __bfloat162float(b);
    }
}

struct Terms {
    uint16_t *t[NTERMS];
};

// One block per position: h = x / sqrt(mean(x^2) + eps) * g as NTERMS bf16 terms.
__global__ void k_pf_norm_split(const float *x, const uint16_t *g, int H, float eps, Terms h) {
    __shared__ float red[32];
    const float *xr = x + size_t(blockIdx.x) * H;
    float ss = 0.f;
    for (int i = threadIdx.x; i < H; i += blockDim.x) ss = fmaf(xr[i], xr[i], ss);
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = ss;
    __syncthreads();
    if (threadIdx.x < 32) {
        float v = threadIdx.x < (blockDim.x >> 5) ? red[threadIdx.x] : 0.f;
        for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
        if (threadIdx.x == 0) red[0] = v;
    }
    __syncthreads();
    const float r = 1.0f / sqrtf(red[0] / float(H) + eps);
    for (int i = threadIdx.x; i < H; i += blockDim.x)
        put_terms(xr[i] * r * __uint_as_float(uint32_t(g[i]) << 16), h.t, size_t(blockIdx.x) * H + i);
}

// One block per position t: RoPE ("rotate half") on its q heads in place and on
// its k heads, k and v rounded to bf16 (nearest even) into the cache at pos0 + t.
__global__ void k_pf_rope_kv(float *qkv, const float2 *rope, int pos0, int nq, int nkv, int hd, uint16_t *kc,
                             uint16_t *vc, size_t layer_base, int max_seq) {
    const int t = blockIdx.x, half = hd / 2, pos = pos0 + t;
    const int qd = nq * hd, kd = nkv * hd;
    float *row = qkv + size_t(t) * (qd + 2 * kd);
    const float2 *c = rope + size_t(pos) * half;
    for (int u = threadIdx.x; u < (nq + nkv) * half; u += blockDim.x) {
        const int h = u / half, i = u % half;
        float *v = row + size_t(h) * hd;  // heads 0..nq-1 are q, then k
        const float a = v[i], b = v[i + half];
        const float ra = a * c[i].x - b * c[i].y, rb = a * c[i].y + b * c[i].x;
        if (h < nq) {
            v[i] = ra;
            v[i + half] = rb;
        } else {
            const size_t dst = layer_base + (size_t(h - nq) * max_seq + pos) * hd;
            kc[dst + i] = __bfloat16_as_ushort(__float2bfloat16_rn(ra));
            kc[dst + i + half] = __bfloat16_as_ushort(__float2bfloat16_rn(rb));
        }
    }
    for (int u = threadIdx.x; u < kd; u += blockDim.x) {
        const int g = u / hd, d = u % hd;
        vc[layer_base + (size_t(g) * max_seq + pos) * hd + d] =
            __bfloat16_as_ushort(__float2bfloat16_rn(row[qd + kd + u]));
    }
}

// Causal attention of the prompt's positions: one warp per (position t, query
// head h) over cache entries 0..pos0 + t of KV head h / (nq / nkv). The warp's
// four groups of eight lanes take positions j, j + 1, j + 2, j + 3; each lane
// holds hd / 8 dimensions of q (scaled by 1/sqrt(hd)) and a running (m, l, o) of
// its group, merged across the groups at the end. Output: o as NTERMS bf16 terms.
template <int DPL>  // dimensions per lane: hd / 8
__global__ void k_pf_attention(const float *qkv, const uint16_t *kc, const uint16_t *vc, size_t layer_base, int pos0,
                               int n, int nq, int nkv, int max_seq, Terms o_t) {
    constexpr int HD = DPL * 8;
    const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
    if (warp >= n * nq) return;
    const int t = warp / nq, h = warp % nq, grp = lane >> 3, sub = lane & 7;
    const int g = h / (nq / nkv), qd = nq * HD, kd = nkv * HD;
    const float scale = 1.0f / sqrtf(float(HD));
    float q[DPL], o[DPL];
    const float *qr = qkv + size_t(t) * (qd + 2 * kd) + size_t(h) * HD + sub * DPL;
#pragma unroll
    for (int e = 0; e < DPL; e++) {
        q[e] = qr[e] * scale;
        o[e] = 0.f;
    }
    float m = -INFINITY, l = 0.f;
    const uint16_t *K = kc + layer_base + size_t(g) * max_seq * HD + sub * DPL;
    const uint16_t *Vv = vc + layer_base + size_t(g) * max_seq * HD + sub * DPL;
    const int last = pos0 + t;
    for (int j0 = 0; j0 <= last; j0 += 4) {
        const int j = j0 + grp;
        float s = -INFINITY;
        float v[DPL];
        if (j <= last) {
            float acc = 0.f;
#pragma unroll
            for (int e = 0; e < DPL; e += 2) {
                const uint32_t kw = *reinterpret_cast<const uint32_t *>(K + size_t(j) * HD + e);
                acc = fmaf(q[e], __uint_as_float(kw << 16), acc);
                acc = fmaf(q[e + 1], __uint_as_float(kw & 0xffff0000u), acc);
                const uint32_t vw = *reinterpret_cast<const uint32_t *>(Vv + size_t(j) * HD + e);
                v[e] = __uint_as_float(vw << 16);
                v[e + 1] = __uint_as_float(vw & 0xffff0000u);
            }
            s = acc;
        } else {
#pragma unroll
            for (int e = 0; e < DPL; e++) v[e] = 0.f;
        }
        s += __shfl_xor_sync(0xffffffffu, s, 1);
        s += __shfl_xor_sync(0xffffffffu, s, 2);
        s += __shfl_xor_sync(0xffffffffu, s, 4);
        if (j <= last) {
            const float mn = fmaxf(m, s);
            const float a = m == -INFINITY ? 0.f : expf(m - mn), pj = expf(s - mn);
            l = l * a + pj;
#pragma unroll
            for (int e = 0; e < DPL; e++) o[e] = fmaf(pj, v[e], o[e] * a);
            m = mn;
        }
    }
    // merge the four groups (lanes sub, sub + 8, sub + 16, sub + 24)
#pragma unroll
    for (int off = 8; off <= 16; off <<= 1) {
        const float mo = __shfl_xor_sync(0xffffffffu, m, off), lo = __shfl_xor_sync(0xffffffffu, l, off);
        const float M = fmaxf(m, mo);
        const float wa = m == -INFINITY ? 0.f : expf(m - M), wb = mo == -INFINITY ? 0.f : expf(mo - M);
#pragma unroll
        for (int e = 0; e < DPL; e++) {
            const float oo = __shfl_xor_sync(0xffffffffu, o[e], off);
            o[e] = o[e] * wa + oo * wb;
        }
        l = l * wa + lo * wb;
        m = M;
    }
    if (grp == 0) {
        const size_t at = size_t(t) * qd + size_t(h) * HD + sub * DPL;
#pragma unroll
        for (int e = 0; e < DPL; e++) put_terms(o[e] / l, o_t.t, at + e);
    }
}

using EncodeTiled = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                 const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                 CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiled encoder() {
    static EncodeTiled fn = nullptr;
    if (fn) return fn;
    void *f = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess || !f) {
        cudaGetLastError();
        return nullptr;
    }
    fn = reinterpret_cast<EncodeTiled>(f);
    return fn;
}

// A [rows][K] bf16 matrix as a GEMM operand: boxes of 64 columns x 128 rows in the
// 128-byte swizzle, rows past the end read as zeros.
bool encode_operand(const uint16_t *base, int64_t rows, int K, TensorMap &out) {
    EncodeTiled enc = encoder();
    if (!enc) return false;
    const cuuint64_t dims[2] = {cuuint64_t(K), cuuint64_t(rows)};
    const cuuint64_t strides[1] = {cuuint64_t(K) * 2};
    const cuuint32_t box[2] = {64, 128}, estr[2] = {1, 1};
    CUtensorMap m;
    if (enc(&m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t *>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return false;
    static_assert(sizeof(m) == sizeof(TensorMap), "tensor map size");
    std::memcpy(&out, &m, sizeof m);
    return true;
}

template <int EPI>
int gemm(const TensorMap *a, const TensorMap &b, int M, int N, int K, float *c, int ldc, const float *gate,
         const Terms *act, const KParams &p, cudaStream_t st) {
    GemmArgs g;
    for (int q = 0; q < NTERMS; q++) {
        g.a[q] = a[q];
        g.act[q] = act ? act->t[q] : nullptr;
    }
    g.b = b;
    g.M = M;
    g.N = N;
    g.K = K;
    g.c = c;
    g.ldc = ldc;
    g.gate = gate;
    g.status = p.status;
    g.timeout_ns = p.timeout_ns;
    static bool attr = false;
    if (!attr) {
        if (cudaFuncSetAttribute(k_gemm<EPI>, cudaFuncAttributeMaxDynamicSharedMemorySize, GEMM_SMEM) != cudaSuccess)
            return LL_ERR_CUDA;
        attr = true;
    }
    const dim3 grid((N + GN - 1) / GN, (M + GM - 1) / GM);
    k_gemm<EPI><<<grid, GTHREADS, GEMM_SMEM, st>>>(g);
    return cudaGetLastError() == cudaSuccess ? LL_OK : LL_ERR_CUDA;
}

}  // namespace

bool prefill_prepare(const KParams &p, const LayerW *host_layers, int n, PrefillBufs &b) {
    static_assert(PrefillBufs::T == NTERMS, "terms");
    if (b.mem && n <= b.n_alloc) return true;
    prefill_release(b);
    const size_t na = size_t((std::max(n, 128) + GM - 1) / GM * GM);
    const size_t H = p.H, qd = size_t(p.nq) * p.hd, kd = size_t(p.nkv) * p.hd, I = p.I;
    auto r256 = [](size_t x) { return (x + 255) / 256 * 256; };
    const size_t sz_x = r256(na * H * 4), sz_h = r256(na * H * 2), sz_qkv = r256(na * (qd + 2 * kd) * 4),
                 sz_o = r256(na * qd * 2), sz_g = r256(na * I * 4), sz_a = r256(na * I * 2), sz_hr = r256(H * 4),
                 sz_l = r256(size_t(p.V) * 4);
    const size_t total = sz_x + NTERMS * sz_h + sz_qkv + NTERMS * sz_o + sz_g + NTERMS * sz_a + sz_hr + sz_l;
    if (cudaMalloc(&b.mem, total) != cudaSuccess) {
        cudaGetLastError();
        b.mem = nullptr;
        return false;
    }
    if (cudaMemset(b.mem, 0, total) != cudaSuccess) {
        prefill_release(b);
        return false;
    }
    uint8_t *cur = static_cast<uint8_t *>(b.mem);
    auto take = [&](size_t bytes) {
        uint8_t *q = cur;
        cur += bytes;
        return q;
    };
    b.x = reinterpret_cast<float *>(take(sz_x));
    for (int q = 0; q < NTERMS; q++) b.h[q] = reinterpret_cast<uint16_t *>(take(sz_h));
    b.qkv = reinterpret_cast<float *>(take(sz_qkv));
    for (int q = 0; q < NTERMS; q++) b.o[q] = reinterpret_cast<uint16_t *>(take(sz_o));
    b.gate = reinterpret_cast<float *>(take(sz_g));
    for (int q = 0; q < NTERMS; q++) b.a[q] = reinterpret_cast<uint16_t *>(take(sz_a));
    b.hrow = reinterpret_cast<float *>(take(sz_hr));
    b.logits = reinterpret_cast<float *>(take(sz_l));
    b.n_alloc = int(na);
    bool ok = true;
    for (int q = 0; q < NTERMS && ok; q++)
        ok = encode_operand(b.h[q], int64_t(na), p.H, b.m_h[q]) && encode_operand(b.o[q], int64_t(na), int(qd), b.m_o[q]) &&
             encode_operand(b.a[q], int64_t(na), p.I, b.m_a[q]);
    b.m_w.assign(size_t(p.L) * 7, TensorMap{});
    for (int l = 0; l < p.L && ok; l++) {
        const LayerW &w = host_layers[l];
        TensorMap *m = &b.m_w[size_t(l) * 7];
        ok = encode_operand(w.wq, int64_t(qd), p.H, m[0]) && encode_operand(w.wk, int64_t(kd), p.H, m[1]) &&
             encode_operand(w.wv, int64_t(kd), p.H, m[2]) && encode_operand(w.wo, p.H, int(qd), m[3]) &&
             encode_operand(w.wg, p.I, p.H, m[4]) && encode_operand(w.wu, p.I, p.H, m[5]) &&
             encode_operand(w.wd, p.H, p.I, m[6]);
    }
    if (!ok) prefill_release(b);
    return ok;
}

void prefill_release(PrefillBufs &b) {
    if (b.mem) cudaFree(b.mem);
    b = PrefillBufs{};
}

int launch_prefill(const KParams &p, const LayerW *host_layers, PrefillBufs &b, const int32_t *tokens_dev, int n,
                   int pos0, float *logits, int32_t *next_dev, void *stream_) {
    cudaStream_t st = static_cast<cudaStream_t>(stream_);
    const int H = p.H, qd = p.nq * p.hd, kd = p.nkv * p.hd, I = p.I;
    const size_t per_layer = size_t(p.nkv) * p.max_seq * p.hd;
    Terms th, to, ta;
    for (int q = 0; q < NTERMS; q++) {
        th.t[q] = b.h[q];
        to.t[q] = b.o[q];
        ta.t[q] = b.a[q];
    }
    k_pf_embed<<<n, 256, 0, st>>>(p.embed, tokens_dev, n, H, p.V, b.x, p.status);
    int rc = cudaGetLastError() == cudaSuccess ? LL_OK : LL_ERR_CUDA;
    for (int l = 0; l < p.L && rc == LL_OK; l++) {
        const LayerW &w = host_layers[l];
        const TensorMap *m = &b.m_w[size_t(l) * 7];
        const size_t lb = size_t(l) * per_layer;
        const int ld = qd + 2 * kd;
        k_pf_norm_split<<<n, 256, 0, st>>>(b.x, w.attn_norm, H, p.eps, th);
        rc = gemm<EPI_STORE>(b.m_h, m[0], n, qd, H, b.qkv, ld, nullptr, nullptr, p, st);
        if (rc == LL_OK) rc = gemm<EPI_STORE>(b.m_h, m[1], n, kd, H, b.qkv + qd, ld, nullptr, nullptr, p, st);
        if (rc == LL_OK) rc = gemm<EPI_STORE>(b.m_h, m[2], n, kd, H, b.qkv + qd + kd, ld, nullptr, nullptr, p, st);
        if (rc != LL_OK) break;
        k_pf_rope_kv<<<n, 256, 0, st>>>(b.qkv, p.rope_cs, pos0, p.nq, p.nkv, p.hd, p.k_cache, p.v_cache, lb, p.max_seq);
        const int blocks = (n * p.nq * 32 + 255) / 256;
        if (p.hd == 64)
            k_pf_attention<8><<<blocks, 256, 0, st>>>(b.qkv, p.k_cache, p.v_cache, lb, pos0, n, p.nq, p.nkv, p.max_seq, to);
        else
            k_pf_attention<16><<<blocks, 256, 0, st>>>(b.qkv, p.k_cache, p.v_cache, lb, pos0, n, p.nq, p.nkv, p.max_seq, to);
        rc = gemm<EPI_ADD>(b.m_o, m[3], n, H, qd, b.x, H, nullptr, nullptr, p, st);
        if (rc != LL_OK) break;
        k_pf_norm_split<<<n, 256, 0, st>>>(b.x, w.mlp_norm, H, p.eps, th);
        rc = gemm<EPI_STORE>(b.m_h, m[4], n, I, H, b.gate, I, nullptr, nullptr, p, st);
        if (rc == LL_OK) rc = gemm<EPI_SILU_MUL>(b.m_h, m[5], n, I, H, nullptr, I, b.gate, &ta, p, st);
        if (rc == LL_OK) rc = gemm<EPI_ADD>(b.m_a, m[6], n, H, I, b.x, H, nullptr, nullptr, p, st);
    }
    if (rc != LL_OK) return rc;
    if (cudaGetLastError() != cudaSuccess) return LL_ERR_CUDA;
    return launch_chain_head(p, b.x + size_t(n - 1) * H, b.hrow, logits ? logits : b.logits, next_dev, stream_);
}

}  // namespace ll
