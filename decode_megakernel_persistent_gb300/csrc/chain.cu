// chain.cu -- the same decode step as one kernel per operation.
//
// This is the "one small kernel per operation" execution that the page "Hazy
// Research Llama-3.2-1B Megakernel" (Chinese write-up, section on why
// conventional inference is inefficient) argues against: every RMSNorm, every
// projection, RoPE, attention, its merge and the activation is its own launch
// on the stream, and each launch waits for the previous one to drain. It is
// kept as an internal comparison for the megakernel and as a second,
// independently written GPU path.
#include <cuda_runtime.h>
#include <stdint.h>

#include "ll_internal.h"

namespace ll {
namespace {

__device__ __forceinline__ float bf(uint16_t b) { return __uint_as_float(uint32_t(b) << 16); }

__device__ __forceinline__ uint16_t to_bf(float f) {
    uint32_t u = __float_as_uint(f);
    if ((u & 0x7f800000u) == 0x7f800000u && (u & 0x007fffffu)) return 0x7fc0;
    u += 0x7fffu + ((u >> 16) & 1u);
    return uint16_t(u >> 16);
}

__device__ __forceinline__ float wsum(float v) {
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

__device__ __forceinline__ float wmax(float v) {
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

__global__ void k_embed(const uint16_t *E, const int32_t *token_dev, int token, int H, int V, float *x,
                        int32_t *status) {
    const int t = token_dev ? *token_dev : token;
    if (t < 0 || t >= V) {
        if (blockIdx.x == 0 && threadIdx.x == 0) atomicCAS(status, 0, LL_ERR_ARG);
        return;
    }
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < H; i += gridDim.x * blockDim.x)
        x[i] = bf(E[size_t(t) * H + i]);
}

// One block: out = x / sqrt(mean(x^2) + eps) * g.
__global__ void k_rmsnorm(const float *x, const uint16_t *g, int n, float eps, float *out) {
    __shared__ float red[32];
    float ss = 0.f;
    for (int i = threadIdx.x; i < n; i += blockDim.x) ss += x[i] * x[i];
    ss = wsum(ss);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = ss;
    __syncthreads();
    if (threadIdx.x < 32) {
        float v = threadIdx.x < (blockDim.x >> 5) ? red[threadIdx.x] : 0.f;
        v = wsum(v);
        if (threadIdx.x == 0) red[0] = v;
    }
    __syncthreads();
    const float r = 1.0f / sqrtf(red[0] / float(n) + eps);
    for (int i = threadIdx.x; i < n; i += blockDim.x) out[i] = x[i] * r * bf(g[i]);
}

// 16 bytes of a weight row, streamed past L1 (no side effects: the compiler may
// batch these loads ahead of their uses).
__device__ __forceinline__ uint4 ld_stream(const uint4 *p) {
    uint4 u;
    asm("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
        : "=r"(u.x), "=r"(u.y), "=r"(u.z), "=r"(u.w)
        : "l"(p));
    return u;
}

// out[r] (+)= W[r] . in, one warp per row, 16-byte streaming loads of W: up to
// 8 per lane (a 2048-wide row) in flight before the first product.
__global__ void k_matvec(const uint16_t *__restrict__ W, const float *__restrict__ in, int rows, int K,
                         float *out, int accumulate) {
    constexpr int U = 8;
    const int lane = threadIdx.x & 31;
    const int warps = (gridDim.x * blockDim.x) >> 5;
    const int nvec = K / 8;
    for (int r = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; r < rows; r += warps) {
        const uint4 *w = reinterpret_cast<const uint4 *>(W + size_t(r) * K);
        float a0 = 0.f, a1 = 0.f;
        for (int v0 = lane; v0 < nvec; v0 += 32 * U) {
            uint4 u[U];
#pragma unroll
            for (int j = 0; j < U; j++) u[j] = v0 + 32 * j < nvec ? ld_stream(w + v0 + 32 * j) : make_uint4(0, 0, 0, 0);
#pragma unroll
            for (int j = 0; j < U; j++) {
                const int v = v0 + 32 * j;
                if (v >= nvec) break;
                const float4 xa = reinterpret_cast<const float4 *>(in)[2 * v];
                const float4 xb = reinterpret_cast<const float4 *>(in)[2 * v + 1];
                a0 = fmaf(__uint_as_float(u[j].x << 16), xa.x, a0);
                a1 = fmaf(__uint_as_float(u[j].x & 0xffff0000u), xa.y, a1);
                a0 = fmaf(__uint_as_float(u[j].y << 16), xa.z, a0);
                a1 = fmaf(__uint_as_float(u[j].y & 0xffff0000u), xa.w, a1);
                a0 = fmaf(__uint_as_float(u[j].z << 16), xb.x, a0);
                a1 = fmaf(__uint_as_float(u[j].z & 0xffff0000u), xb.y, a1);
                a0 = fmaf(__uint_as_float(u[j].w << 16), xb.z, a0);
                a1 = fmaf(__uint_as_float(u[j].w & 0xffff0000u), xb.w, a1);
            }
        }
        const float y = wsum(a0 + a1);
        if (lane == 0) out[r] = accumulate ? out[r] + y : y;
    }
}

// RoPE on q (in place) and k; k and v rounded to bf16 and stored at pos. c is
// the (cos, sin) row of position pos, hd / 2 entries.
__global__ void k_rope_kv(float *qkv, const float2 *c, int pos, int nq, int nkv, int hd,
                          uint16_t *kc, uint16_t *vc, size_t layer_base, int max_seq) {
    const int half = hd / 2;
    const int total = (nq + nkv) * half;
    for (int t = blockIdx.x * blockDim.x + threadIdx.x; t < total + nkv * hd; t += gridDim.x * blockDim.x) {
        if (t < total) {
            const int h = t / half, i = t % half;
            float *v = qkv + size_t(h) * hd;  // heads 0..nq-1 are q, nq.. are k
            const float a = v[i], b = v[i + half];
            const float2 r = c[i];
            const float ra = a * r.x - b * r.y, rb = a * r.y + b * r.x;
            if (h < nq) {
                v[i] = ra;
                v[i + half] = rb;
            } else {
                const size_t dst = layer_base + (size_t(h - nq) * max_seq + pos) * hd;
                kc[dst + i] = to_bf(ra);
                kc[dst + i + half] = to_bf(rb);
            }
        } else {
            const int u = t - total, g = u / hd, d = u % hd;
            const float val = qkv[size_t(nq + nkv) * hd + u];
            vc[layer_base + (size_t(g) * max_seq + pos) * hd + d] = to_bf(val);
        }
    }
}

// Split-KV attention, grid (nkv, splits): partial (o, m, l) per query head of the
// group over positions [c0, c1) of 0..pos (the new entry is already in the cache).
__global__ void k_attn_partial(const float *q, const uint16_t *kc, const uint16_t *vc, size_t layer_base,
                               int pos, int max_seq, int G, int hd, int splits, float *part) {
    __shared__ float qs[MAX_GQA][MAX_HD];
    __shared__ float sc[MAX_GQA][128];
    __shared__ float mrun[MAX_GQA], lrun[MAX_GQA], alpha[MAX_GQA];
    const int g = blockIdx.x, c = blockIdx.y, tid = threadIdx.x;
    const int n_all = pos + 1;
    const int c0 = int((long long)c * n_all / splits), c1 = int((long long)(c + 1) * n_all / splits);
    const float scale = 1.0f / sqrtf(float(hd));
    for (int t = tid; t < G * hd; t += blockDim.x) qs[t / hd][t % hd] = q[size_t(g * G) * hd + t] * scale;
    if (tid < G) {
        mrun[tid] = -INFINITY;
        lrun[tid] = 0.f;
    }
    float oacc[4] = {0.f, 0.f, 0.f, 0.f};
    __syncthreads();
    const uint16_t *K = kc + layer_base + size_t(g) * max_seq * hd;
    const uint16_t *V = vc + layer_base + size_t(g) * max_seq * hd;
    const int warp = tid >> 5, lane = tid & 31;
    for (int t0 = c0; t0 < c1; t0 += 128) {
        const int n = min(128, c1 - t0);
        for (int u = tid; u < G * n; u += blockDim.x) {
            const int h = u / n, j = u % n;
            const uint16_t *k = K + size_t(t0 + j) * hd;
            float a = 0.f;
            for (int d = 0; d < hd; d++) a = fmaf(qs[h][d], bf(k[d]), a);
            sc[h][j] = a;
        }
        __syncthreads();
        if (warp < G) {
            float mx = -INFINITY;
            for (int j = lane; j < n; j += 32) mx = fmaxf(mx, sc[warp][j]);
            mx = wmax(mx);
            const float mo = mrun[warp], mn = fmaxf(mo, mx);
            float sum = 0.f;
            for (int j = lane; j < n; j += 32) {
                const float e = expf(sc[warp][j] - mn);
                sc[warp][j] = e;
                sum += e;
            }
            sum = wsum(sum);
            if (lane == 0) {
                const float a = mo == -INFINITY ? 0.f : expf(mo - mn);
                alpha[warp] = a;
                lrun[warp] = lrun[warp] * a + sum;
                mrun[warp] = mn;
            }
        }
        __syncthreads();
        for (int k = 0; k < 4; k++) {
            const int pi = tid + k * blockDim.x;
            if (pi < G * hd) {
                const int h = pi / hd, d = pi % hd;
                float a = oacc[k] * alpha[h];
                for (int j = 0; j < n; j++) a = fmaf(sc[h][j], bf(V[size_t(t0 + j) * hd + d]), a);
                oacc[k] = a;
            }
        }
        __syncthreads();
    }
    const int stride = hd + 2;
    for (int k = 0; k < 4; k++) {
        const int pi = tid + k * blockDim.x;
        if (pi < G * hd) {
            const int h = pi / hd, d = pi % hd;
            part[(size_t(g * G + h) * splits + c) * stride + d] = oacc[k];
        }
    }
    if (tid < G) {
        part[(size_t(g * G + tid) * splits + c) * stride + hd] = mrun[tid];
        part[(size_t(g * G + tid) * splits + c) * stride + hd + 1] = lrun[tid];
    }
}

__global__ void k_attn_combine(const float *part, int nq, int hd, int splits, float *o) {
    const int stride = hd + 2;
    for (int t = blockIdx.x * blockDim.x + threadIdx.x; t < nq * hd; t += gridDim.x * blockDim.x) {
        const int h = t / hd, d = t % hd;
        const float *b = part + size_t(h) * splits * stride;
        float M = -INFINITY;
        for (int j = 0; j < splits; j++) M = fmaxf(M, b[j * stride + hd]);
        float L = 0.f, O = 0.f;
        for (int j = 0; j < splits; j++) {
            const float mj = b[j * stride + hd];
            if (mj == -INFINITY) continue;
            const float w = expf(mj - M);
            L = fmaf(b[j * stride + hd + 1], w, L);
            O = fmaf(b[j * stride + d], w, O);
        }
        o[t] = O / L;
    }
}

__global__ void k_silu_mul(const float *g, const float *u, float *a, int n) {
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x) {
        const float z = g[i];
        a[i] = z / (1.0f + expf(-z)) * u[i];
    }
}

// One block: greedy argmax, lowest index on ties. Logits that hold no orderable
// value (all NaN) have no greedy token: the status word records LL_ERR_NUMERIC.
// Greedy token: the smallest index holding the largest logit (NaNs never win;
// all NaN is an error). One block: each thread keeps U running (max, index)
// pairs over float4 groups i, i + 4 blockDim, ... so that U loads are in flight.
__device__ __forceinline__ void argmax_take(float v, int i, float &best, int &idx) {
    if (v > best || (v == best && best > -INFINITY && i < idx)) {
        best = v;
        idx = i;
    }
}

__global__ void k_argmax(const float *v, int n, int32_t *next_dev, int32_t *token_out, int32_t *status) {
    constexpr int U = 4;
    __shared__ float bv[32];
    __shared__ int bi[32];
    float best = -INFINITY;
    int idx = 0x7fffffff;
    const int n4 = n / 4, step = int(blockDim.x);
    const float4 *v4 = reinterpret_cast<const float4 *>(v);
    if ((reinterpret_cast<uintptr_t>(v) & 15u) != 0) {  // (unaligned: plain loads)
        for (int i = threadIdx.x; i < n; i += step) argmax_take(v[i], i, best, idx);
    } else {
        for (int g0 = threadIdx.x; g0 < n4; g0 += U * step) {
            float4 x[U];
#pragma unroll
            for (int u = 0; u < U; u++) x[u] = g0 + u * step < n4 ? v4[g0 + u * step] : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int u = 0; u < U; u++) {
                if (g0 + u * step >= n4) break;
                const int i = 4 * (g0 + u * step);
                argmax_take(x[u].x, i, best, idx);
                argmax_take(x[u].y, i + 1, best, idx);
                argmax_take(x[u].z, i + 2, best, idx);
                argmax_take(x[u].w, i + 3, best, idx);
            }
        }
        for (int i = 4 * n4 + int(threadIdx.x); i < n; i += step) argmax_take(v[i], i, best, idx);
    }
    for (int o = 16; o > 0; o >>= 1) {
        const float ob = __shfl_xor_sync(0xffffffffu, best, o);
        const int oi = __shfl_xor_sync(0xffffffffu, idx, o);
        if (ob > best || (ob == best && oi < idx)) {
            best = ob;
            idx = oi;
        }
    }
    if ((threadIdx.x & 31) == 0) {
        bv[threadIdx.x >> 5] = best;
        bi[threadIdx.x >> 5] = idx;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        for (int w = 1; w < int(blockDim.x >> 5); w++)
            if (bv[w] > best || (bv[w] == best && bi[w] < idx)) {
                best = bv[w];
                idx = bi[w];
            }
        if (idx == 0x7fffffff) atomicCAS(status, 0, LL_ERR_NUMERIC);
        token_out[0] = idx;
        if (next_dev) *next_dev = idx;
    }
}

int grid_for_rows(int rows, int nsm) {
    const int blocks = (rows + 7) / 8;  // 8 warps per block, one row each
    return blocks < nsm * 8 ? blocks : nsm * 8;
}

}  // namespace

int launch_chain_head(const KParams &p, const float *x, float *h, float *logits, int32_t *next_dev, void *stream_) {
    cudaStream_t st = static_cast<cudaStream_t>(stream_);
    k_rmsnorm<<<1, 1024, 0, st>>>(x, p.final_norm, p.H, p.eps, h);
    k_matvec<<<grid_for_rows(p.V, p.nsm), 256, 0, st>>>(p.lm_head, h, p.V, p.H, logits, 0);
    k_argmax<<<1, 1024, 0, st>>>(logits, p.V, next_dev, p.token_out, p.status);
    return cudaGetLastError() == cudaSuccess ? LL_OK : LL_ERR_CUDA;
}

int launch_chain_step(const KParams &p, const ChainBufs &b, void *stream_) {
    cudaStream_t st = static_cast<cudaStream_t>(stream_);
    const int H = p.H, qd = p.nq * p.hd, kd = p.nkv * p.hd, I = p.I, G = p.nq / p.nkv;
    const size_t per_layer = size_t(p.nkv) * p.max_seq * p.hd;
    const float2 *rope_row = b.rope_row ? b.rope_row : p.rope_cs + size_t(p.pos) * (p.hd / 2);
    auto mv = [&](const uint16_t *W, const float *in, int rows, int K, float *out, int acc) {
        k_matvec<<<grid_for_rows(rows, p.nsm), 256, 0, st>>>(W, in, rows, K, out, acc);
    };
    k_embed<<<(H + 255) / 256, 256, 0, st>>>(p.embed, p.token_dev, p.token, H, p.V, b.x, p.status);
    for (int l = 0; l < p.L; l++) {
        const LayerW &w = b.host_layers[l];
        const size_t lb = size_t(l) * per_layer;
        k_rmsnorm<<<1, 1024, 0, st>>>(b.x, w.attn_norm, H, p.eps, b.h);
        mv(w.wq, b.h, qd, H, b.qkv, 0);
        mv(w.wk, b.h, kd, H, b.qkv + qd, 0);
        mv(w.wv, b.h, kd, H, b.qkv + qd + kd, 0);
        k_rope_kv<<<((p.nq + p.nkv) * p.hd / 2 + kd + 255) / 256, 256, 0, st>>>(
            b.qkv, rope_row, p.pos, p.nq, p.nkv, p.hd, p.k_cache, p.v_cache, lb, p.max_seq);
        k_attn_partial<<<dim3(p.nkv, b.splits), 256, 0, st>>>(b.qkv, p.k_cache, p.v_cache, lb, p.pos,
                                                             p.max_seq, G, p.hd, b.splits, b.part);
        k_attn_combine<<<(qd + 255) / 256, 256, 0, st>>>(b.part, p.nq, p.hd, b.splits, b.o);
        mv(w.wo, b.o, H, qd, b.x, 1);
        k_rmsnorm<<<1, 1024, 0, st>>>(b.x, w.mlp_norm, H, p.eps, b.h);
        mv(w.wg, b.h, I, H, b.gate, 0);
        mv(w.wu, b.h, I, H, b.up, 0);
        k_silu_mul<<<(I + 255) / 256, 256, 0, st>>>(b.gate, b.up, b.act, I);
        mv(w.wd, b.act, H, I, b.x, 1);
    }
    k_rmsnorm<<<1, 1024, 0, st>>>(b.x, p.final_norm, H, p.eps, b.h);
    float *logits = p.logits ? p.logits : b.logits;
    mv(p.lm_head, b.h, p.V, H, logits, 0);
    k_argmax<<<1, 1024, 0, st>>>(logits, p.V, p.next_token_dev, p.token_out, p.status);
    return cudaGetLastError() == cudaSuccess ? LL_OK : LL_ERR_CUDA;
}

}  // namespace ll
