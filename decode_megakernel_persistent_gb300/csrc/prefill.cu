// prefill.cu -- a prompt's positions through the model at once (ll_prefill).
//
// The page "Hazy Research Llama-3.2-1B Megakernel" is about decode; a prompt is
// the step before it: every position of the prompt goes through every layer,
// which turns each projection into a matrix product of (positions x width) by
// the weight matrix, filling the KV cache for the decode steps that follow.
// Here every projection is a persistent tcgen05 GEMM (the fifth-generation
// tensor cores): one block per SM walks its share of the output tiles; TMA brings
// 128 x 64 bf16 tiles of the operands into shared memory in the 128-byte swizzle
// through a 3- or 4-stage mbarrier pipeline that runs across tile boundaries; one
// thread issues tcgen05.mma (K = 16 per instruction, N = 256: the positions by
// the gate and up tiles together, or, transposed, the weight tile by two stacked
// activation terms) into one of two tensor-memory accumulators; eight warps read
// the other back with tcgen05.ld for the epilogue meanwhile. The decode path
// keeps activations in fp32, and a bf16 product with one term of them misses the
// logits' bar, so each activation matrix enters as bf16 terms (t0 = bf16(x),
// t1 = bf16(x - t0), t2 = bf16(x - t0 - t1)): three for the Q/K/V GEMM, whose K/V
// go to the cache (the 24 bits of an fp32 value), two for the others (16 bits);
// a pipeline stage carries one K step of every term, so each weight tile is
// loaded once for all of them.
//
// Per layer: RMSNorm into the terms; Q, K, V in one GEMM; RoPE with the K/V
// rounded to bf16 into the cache; causal attention over the cache (mma.sync
// tiles, two query positions x the KV head's query heads per warp); O GEMM added
// into the residual; RMSNorm; one GEMM for gate and up whose epilogue forms
// silu(gate) * up in terms; down GEMM added into the residual. These kernels are
// launched as programmatic dependents (see pdl_wait). Then the last position's
// final norm, LM head and argmax.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <algorithm>
#include <cstring>

#include "ll_internal.h"

namespace ll {
namespace {

constexpr int GM = 128, GN = 128, GK = 64, GTHREADS = 320;
constexpr int NTERMS = 3;  // bf16 terms of an activation
constexpr uint32_t GTILE = GM * GK * 2;  // bytes of one 128 x 64 bf16 tile (A and B alike)
// A pipeline stage holds one K step of every A term and every B operand (each B
// tile is loaded once for all the terms): 16 KB per tile, 64 KB for Q/K/V (three
// terms) and gate/up (two terms, two B operands), 48 KB for O and down; as many
// stages as fit in 192 KB of the 227 KB a block may have.
__host__ __device__ constexpr int gstages(int tiles) { return 196608 / (tiles * int(GTILE)); }  // tiles per stage
// The A terms a GEMM takes: three for the Q, K, V projection (its K/V are the
// cache entries the decode steps read, rounded to bf16, so they follow the fp32
// input to its last bit), two for the others (16 of the 24 mantissa bits: their
// outputs feed the residual stream and the MLP, whose parity bar is 1e-2 of the
// logits; the two-term input is within 2^-17 of the fp32 one).
__host__ __device__ constexpr int gterms(int epi) { return epi == 0 ? 3 : 2; }

__device__ __forceinline__ uint32_t saddr(const void *p) { return static_cast<uint32_t>(__cvta_generic_to_shared(p)); }

__device__ __forceinline__ uint64_t now_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Programmatic dependent launch (the per-layer kernels of a prefill): a kernel
// lets the next one in the stream start its blocks as soon as it runs itself
// (their set-up then overlaps its tail), and waits, before it reads anything
// the previous kernel wrote, until that kernel has finished and its writes are
// visible. Both are no-ops for a launch without the attribute.
__device__ __forceinline__ void pdl_release() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, args...);
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

enum : int { EPI_STORE = 0, EPI_ADD = 1, EPI_GATEUP = 2 };

struct GemmArgs {
    TensorMap a[NTERMS];         // A terms [rows][K], bf16, K-major, boxes 64 x 128, 128-byte swizzle
    TensorMap b[3];              // B [N][K] alike. EPI_GATEUP: b[0] the gate, b[1] the up matrix. Otherwise
                                 // the output columns may stack up to three matrices: columns [0, bsplit1)
                                 // come from b[0], [bsplit1, bsplit2) from b[1], the rest from b[2]
    int bsplit1, bsplit2;        // multiples of GN (a tile never straddles two matrices)
    int M, N, K;                 // positions, outputs, inner width (K a multiple of 64)
    float *c;                    // [M][ldc] fp32: EPI_STORE c = A B^T, EPI_ADD c += A B^T
    int ldc;
    uint16_t *act[NTERMS];       // EPI_GATEUP: silu(A Bg^T) * (A Bu^T) as NTERMS bf16 terms, [M][ldc]
    int32_t *status;
    uint64_t timeout_ns;
};

// A persistent GEMM: block b takes the output tiles b, b + gridDim.x, ... (a tile:
// 128 rows by GN columns; EPI_GATEUP: the same columns of the gate and the up
// products, side by side in one 128 x 256 accumulator). Warp 0 lane 0 feeds the
// stages with TMA, through all of the block's tiles without a break; warp 1 lane
// 0 issues the MMAs of a tile into one of two tensor-memory accumulators (256
// columns each) and commits it to acc_full; warps 2..9 run the epilogue of that
// accumulator (warp w reads tensor-memory lanes 32 (w % 4) .. 32 (w % 4) + 31
// and half (w - 2) / 4 of the columns), then hand it back through acc_empty, so
// a tile's epilogue runs under the next tile's products.
template <int EPI>
__global__ void __launch_bounds__(GTHREADS, 1) k_gemm(const __grid_constant__ GemmArgs g) {
    constexpr int NB = EPI == EPI_GATEUP ? 2 : 1;  // B operands (accumulators)
    constexpr int NT = gterms(EPI);                 // A terms
    constexpr int GSTAGES = gstages(NT + NB);
    constexpr uint32_t STAGE = GTILE * (NT + NB);
    // EPI_STORE and EPI_ADD run transposed: the weight tile is the MMA's A (128
    // output columns as the accumulator's lanes) and terms 0 and 1, adjacent in
    // the stage, are one 256-row B (accumulator columns: term 0's 128 positions,
    // then term 1's); a third term is an N = 128 product of its own, added into
    // term 0's columns. The epilogue adds the two halves. Per K step of 16: one
    // N = 256 product (and one N = 128) instead of two (three) N = 128 ones.
    constexpr bool TRANS = EPI != EPI_GATEUP;
    static_assert(!TRANS || NT == 2 || NT == 3, "the transposed product takes two or three terms");
    constexpr uint32_t ACC_COLS = TRANS ? 2 * 128 : 128 * NB;  // one accumulator
    constexpr int ACC_BUFS = 2 * ACC_COLS <= 512 ? 2 : 1;
    constexpr uint32_t TCOLS = ACC_BUFS * ACC_COLS <= 256 ? 256 : 512;  // a power of two
    constexpr int EPI_WARPS = 8;
    static_assert(GTHREADS == 32 * (2 + EPI_WARPS), "producer, MMA and epilogue warps");
    extern __shared__ __align__(1024) uint8_t gsm[];
    uint8_t *tiles = gsm;
    uint64_t *full = reinterpret_cast<uint64_t *>(gsm + GSTAGES * STAGE);
    uint64_t *empty = full + GSTAGES;
    uint64_t *acc_full = empty + GSTAGES;
    uint64_t *acc_empty = acc_full + 2;
    volatile uint32_t *tmem_slot = reinterpret_cast<volatile uint32_t *>(acc_empty + 2);
    volatile int *err = reinterpret_cast<volatile int *>(acc_empty + 3);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int tiles_n = (g.N + GN - 1) / GN, tiles_m = (g.M + GM - 1) / GM, ntiles = tiles_n * tiles_m;
    // gate/up: row tiles vary fastest, so the blocks sharing a weight tile run
    // together and read it from HBM once; the others: column tiles fastest
    auto tile_m = [&](int t) { return EPI == EPI_GATEUP ? t % tiles_m : t / tiles_n; };
    auto tile_n = [&](int t) { return EPI == EPI_GATEUP ? t / tiles_m : t % tiles_n; };
    const int iters = g.K / GK;  // K steps; each stage carries every term
    pdl_release();
    if (threadIdx.x == 0) {
        for (int s = 0; s < GSTAGES; s++) {
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(saddr(&full[s])) : "memory");
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(saddr(&empty[s])) : "memory");
        }
        for (int b = 0; b < 2; b++) {
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(saddr(&acc_full[b])) : "memory");
            asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(saddr(&acc_empty[b])), "r"(EPI_WARPS)
                         : "memory");
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        *err = 0;
    }
    if (warp == 0) {  // fp32 columns of tensor memory: ACC_BUFS accumulators
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         saddr(const_cast<uint32_t *>(tmem_slot))),
                     "n"(TCOLS)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    const uint32_t tmem = *tmem_slot;
    pdl_wait();  // the operands (and, adding into it, C) as the previous kernel left them

    if (warp == 0) {
        if (lane == 0) {
            int sent = 0;  // stages filled, over all of this block's tiles
            bool ok = true;
            for (int t = blockIdx.x; t < ntiles && ok; t += gridDim.x) {
                const int m0 = tile_m(t) * GM, n0 = tile_n(t) * GN;
                // the B matrix of this tile's columns and the tile's first row in it
                const int bsel = NB == 2 ? 0 : (n0 >= g.bsplit2 ? 2 : n0 >= g.bsplit1 ? 1 : 0);
                const int brow = n0 - (bsel == 2 ? g.bsplit2 : bsel == 1 ? g.bsplit1 : 0);
                for (int it = 0; it < iters; it++) {
                    const int s = sent % GSTAGES;
                    if (sent >= GSTAGES &&
                        !mbar_wait(&empty[s], ((sent / GSTAGES) - 1) & 1, g.timeout_ns, g.status, err)) {
                        ok = false;
                        break;
                    }
                    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(saddr(&full[s])),
                                 "r"(STAGE)
                                 : "memory");
                    const int kc = it * GK;
                    const uint32_t dst = saddr(tiles + size_t(s) * STAGE);
#pragma unroll
                    for (int q = 0; q < NT; q++) tma2d(dst + q * GTILE, &g.a[q], kc, m0, &full[s]);
                    if (NB == 2) {
                        tma2d(dst + NT * GTILE, &g.b[0], kc, n0, &full[s]);
                        tma2d(dst + (NT + 1) * GTILE, &g.b[1], kc, n0, &full[s]);
                    } else {
                        tma2d(dst + NT * GTILE, &g.b[bsel], kc, brow, &full[s]);
                    }
                    sent++;
                }
            }
            // never leave with copies in flight into this block's shared memory (after
            // an error; normally the products have consumed every stage)
            for (int q = sent > GSTAGES ? sent - GSTAGES : 0; q < sent; q++) {
                const uint64_t t0 = now_ns();
                while (!mbar_try(&full[q % GSTAGES], (q / GSTAGES) & 1) && now_ns() - t0 < g.timeout_ns) {
                }
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // gate/up: the two B tiles sit one after the other in the stage, so one
            // N = 256 product covers both (rows 128.. of the operand are the up tile)
            constexpr uint32_t idesc = TRANS ? idesc_bf16(GN, 2 * GM) : idesc_bf16(GM, GN * NB);
            constexpr uint32_t idesc3 = idesc_bf16(GN, GM);  // TRANS: the third term (into term 0's columns)
            int used = 0, tl = 0;  // stages consumed, tiles done (this block)
            bool ok = true;
            for (int t = blockIdx.x; t < ntiles && ok; t += gridDim.x, tl++) {
                const int buf = tl % ACC_BUFS, round = tl / ACC_BUFS;
                // the accumulator is free once the epilogue of its previous tile read it
                if (round > 0 && !mbar_wait(&acc_empty[buf], (round - 1) & 1, g.timeout_ns, g.status, err)) break;
                asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
                const uint32_t acc_base = tmem + uint32_t(buf) * ACC_COLS;
                for (int it = 0; it < iters; it++) {
                    const int s = used % GSTAGES;
                    if (!mbar_wait(&full[s], (used / GSTAGES) & 1, g.timeout_ns, g.status, err)) {
                        ok = false;
                        break;
                    }
                    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
                    const uint32_t base = saddr(tiles + size_t(s) * STAGE);
#pragma unroll
                    for (int q = 0; q < (TRANS ? 1 : NT); q++) {
                        const uint64_t ad = smem_desc_sw128(TRANS ? base + GTILE * NT : base + q * GTILE);
                        const uint64_t bd = smem_desc_sw128(TRANS ? base : base + GTILE * NT);
#pragma unroll
                        for (int kk = 0; kk < GK / 16; kk++) {
                            const uint32_t acc = (it | q | kk) != 0 ? 1u : 0u;
                            asm volatile(
                                "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
                                "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(acc_base),
                                "l"(ad + uint64_t(2 * kk)), "l"(bd + uint64_t(2 * kk)), "r"(idesc), "r"(acc)
                                : "memory");
                            if (TRANS && NT == 3) {
                                const uint64_t b3 = smem_desc_sw128(base + 2 * GTILE);
                                asm volatile(
                                    "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
                                    "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(acc_base),
                                    "l"(ad + uint64_t(2 * kk)), "l"(b3 + uint64_t(2 * kk)), "r"(idesc3), "r"(1u)
                                    : "memory");
                            }
                        }
                    }
                    // the stage is free once these products have read it
                    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                                     saddr(&empty[s]))
                                 : "memory");
                    used++;
                }
                if (!ok) break;
                // the accumulator is complete once every product issued so far is
                asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                                 saddr(&acc_full[buf]))
                             : "memory");
            }
        }
    } else {
        const int quarter = warp & 3, half = (warp - 2) >> 2;
        int tl = 0;
        for (int t = blockIdx.x; t < ntiles; t += gridDim.x, tl++) {
            const int buf = tl % ACC_BUFS, round = tl / ACC_BUFS;
            if (!mbar_wait(&acc_full[buf], round & 1, g.timeout_ns, g.status, err) || *err) break;
            asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
            const int m0 = tile_m(t) * GM, n0 = tile_n(t) * GN;
            const uint32_t acc_base = tmem + uint32_t(buf) * ACC_COLS;
            // (the wait is in the same statement as the load, so no use of the
            // registers can be placed before it)
            auto ld16 = [&](uint32_t col, uint32_t (&r)[16]) {
                const uint32_t taddr = acc_base + (uint32_t(quarter * 32) << 16) + col;
                asm volatile(
                    "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, "
                    "%13, %14, %15}, [%16];\n\ttcgen05.wait::ld.sync.aligned;"
                    : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
                      "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
                      "=r"(r[15])
                    : "r"(taddr)
                    : "memory");
            };
            if (TRANS) {
                // lane: output column n0 + 32 quarter + lane; columns of the accumulator:
                // positions (terms 0 and 2 at c, term 1 at 128 + c), this warp's half
                // of them
                const int col = n0 + quarter * 32 + lane;
#pragma unroll 1
                for (int c0 = half * (GM / 2); c0 < (half + 1) * (GM / 2); c0 += 16) {
                    uint32_t r[16], u[16];
                    ld16(uint32_t(c0), r);
                    ld16(uint32_t(GM + c0), u);
                    if (col >= g.N) continue;
                    float *const cp = g.c + size_t(m0 + c0) * g.ldc + col;
                    float old[16];
                    if (EPI == EPI_ADD) {  // all 16 loads in flight before the first store
#pragma unroll
                        for (int e = 0; e < 16; e++) old[e] = m0 + c0 + e < g.M ? cp[size_t(e) * g.ldc] : 0.f;
                    }
#pragma unroll
                    for (int e = 0; e < 16; e++) {
                        float v = __uint_as_float(r[e]) + __uint_as_float(u[e]);
                        if (EPI == EPI_ADD) v += old[e];
                        if (m0 + c0 + e < g.M) cp[size_t(e) * g.ldc] = v;
                    }
                }
            } else {  // EPI_GATEUP: row m0 + 32 quarter + lane, gate at c, up at 128 + c
                const int row = m0 + quarter * 32 + lane;
#pragma unroll 1
                for (int c0 = half * (GN / 2); c0 < (half + 1) * (GN / 2); c0 += 16) {
                    uint32_t r[16], u[16];
                    ld16(uint32_t(c0), r);
                    ld16(uint32_t(128 + c0), u);
                    const int col0 = n0 + c0;
                    if (row >= g.M || col0 + 16 > g.N) continue;  // (N is a multiple of 16 here)
                    const size_t at = size_t(row) * g.ldc + col0;
                    constexpr int NW = gterms(EPI_ADD);  // the down GEMM's terms
                    uint32_t w[NW][8];
#pragma unroll
                    for (int j = 0; j < 16; j += 2) {
                        float a2[2];
#pragma unroll
                        for (int e = 0; e < 2; e++) {
                            const float z = __uint_as_float(r[j + e]);
                            a2[e] = z / (1.0f + expf(-z)) * __uint_as_float(u[j + e]);
                        }
#pragma unroll
                        for (int q = 0; q < NW; q++) {
                            const __nv_bfloat162 t2 = __floats2bfloat162_rn(a2[0], a2[1]);
                            w[q][j / 2] = *reinterpret_cast<const uint32_t *>(&t2);
                            a2[0] -= __low2float(t2);
                            a2[1] -= __high2float(t2);
                        }
                    }
#pragma unroll
                    for (int q = 0; q < NW; q++) {
                        uint4 *dst = reinterpret_cast<uint4 *>(g.act[q] + at);
                        dst[0] = make_uint4(w[q][0], w[q][1], w[q][2], w[q][3]);
                        dst[1] = make_uint4(w[q][4], w[q][5], w[q][6], w[q][7]);
                    }
                }
            }
            // this warp is done reading the accumulator: hand it back to the MMAs
            asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
            __syncwarp();
            if (lane == 0) asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(saddr(&acc_empty[buf])) : "memory");
        }
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    if (warp == 0) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "n"(TCOLS) : "memory");
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
// Thread j takes the 8-element groups j, j + blockDim, ... (H a multiple of 8):
// 32-byte reads of x, 16-byte writes of each term. A thread with one group (H
// <= 8 blockDim, the usual launch) keeps it in registers between the two passes.
__device__ __forceinline__ void load8(const float *p, float (&v)[8]) {
    const float4 a = *reinterpret_cast<const float4 *>(p), b = *reinterpret_cast<const float4 *>(p + 4);
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w; v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}

// the normed group of 8 at i0 (x values v, gain g) as NTERMS bf16 terms
__device__ __forceinline__ void norm_store8(const float (&v)[8], float r, const uint16_t *g, int i0, size_t at,
                                            const Terms &h) {
    const uint4 gw = *reinterpret_cast<const uint4 *>(g + i0);
    const uint32_t gg[4] = {gw.x, gw.y, gw.z, gw.w};
    float y[8];
#pragma unroll
    for (int e = 0; e < 8; e++) y[e] = v[e] * r * __uint_as_float(e & 1 ? gg[e / 2] & 0xffff0000u : gg[e / 2] << 16);
#pragma unroll
    for (int q = 0; q < NTERMS; q++) {
        uint32_t w[4];
#pragma unroll
        for (int e = 0; e < 8; e += 2) {
            const __nv_bfloat162 b2 = __floats2bfloat162_rn(y[e], y[e + 1]);
            w[e / 2] = *reinterpret_cast<const uint32_t *>(&b2);
            y[e] -= __low2float(b2);
            y[e + 1] -= __high2float(b2);
        }
        *reinterpret_cast<uint4 *>(h.t[q] + at) = make_uint4(w[0], w[1], w[2], w[3]);
    }
}

__global__ void k_pf_norm_split(const float *x, const uint16_t *g, int H, float eps, Terms h) {
    __shared__ float red[32];
    pdl_release();
    pdl_wait();
    const int groups = H / 8, step = int(blockDim.x), j = int(threadIdx.x);
    const bool single = groups <= step;
    const float *xr = x + size_t(blockIdx.x) * H;
    float v[8];
    float ss = 0.f;
    if (single) {
        if (j < groups) {
            load8(xr + 8 * j, v);
#pragma unroll
            for (int e = 0; e < 8; e++) ss = fmaf(v[e], v[e], ss);
        }
    } else {
        for (int gi = j; gi < groups; gi += step) {
            load8(xr + 8 * gi, v);
#pragma unroll
            for (int e = 0; e < 8; e++) ss = fmaf(v[e], v[e], ss);
        }
    }
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = ss;
    __syncthreads();
    if (threadIdx.x < 32) {
        float t = threadIdx.x < (blockDim.x >> 5) ? red[threadIdx.x] : 0.f;
        for (int o = 16; o > 0; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
        if (threadIdx.x == 0) red[0] = t;
    }
    __syncthreads();
    const float r = 1.0f / sqrtf(red[0] / float(H) + eps);
    const size_t row = size_t(blockIdx.x) * H;
    if (single) {
        if (j < groups) norm_store8(v, r, g, 8 * j, row + 8 * j, h);
    } else {
        for (int gi = j; gi < groups; gi += step) {
            load8(xr + 8 * gi, v);
            norm_store8(v, r, g, 8 * gi, row + 8 * gi, h);
        }
    }
}

// One block per position t: RoPE ("rotate half") on its q heads in place and on
// its k heads, k and v rounded to bf16 (nearest even) into the cache at pos0 + t.
// A thread takes four consecutive pairs (i, i + hd / 2) of a head: 16-byte loads
// and stores of q, 8-byte stores into the cache.
__device__ __forceinline__ uint2 bf16x4(float a, float b, float c, float d) {
    const __nv_bfloat162 lo = __floats2bfloat162_rn(a, b), hi = __floats2bfloat162_rn(c, d);
    return make_uint2(*reinterpret_cast<const uint32_t *>(&lo), *reinterpret_cast<const uint32_t *>(&hi));
}

__global__ void k_pf_rope_kv(float *qkv, const float2 *rope, int pos0, int nq, int nkv, int hd, uint16_t *kc,
                             uint16_t *vc, size_t layer_base, int max_seq) {
    pdl_release();
    pdl_wait();
    const int t = blockIdx.x, half = hd / 2, quads = half / 4, pos = pos0 + t;
    const int qd = nq * hd, kd = nkv * hd;
    float *row = qkv + size_t(t) * (qd + 2 * kd);
    const float4 *c = reinterpret_cast<const float4 *>(rope + size_t(pos) * half);  // two (cos, sin) per float4
    for (int u = threadIdx.x; u < (nq + nkv) * quads; u += blockDim.x) {
        const int h = u / quads, i = 4 * (u % quads);
        float *v = row + size_t(h) * hd;  // heads 0..nq-1 are q, then k
        const float4 a = *reinterpret_cast<const float4 *>(v + i), b = *reinterpret_cast<const float4 *>(v + i + half);
        const float4 c01 = c[i / 2], c23 = c[i / 2 + 1];
        const float4 ra = make_float4(a.x * c01.x - b.x * c01.y, a.y * c01.z - b.y * c01.w, a.z * c23.x - b.z * c23.y,
                                      a.w * c23.z - b.w * c23.w);
        const float4 rb = make_float4(a.x * c01.y + b.x * c01.x, a.y * c01.w + b.y * c01.z, a.z * c23.y + b.z * c23.x,
                                      a.w * c23.w + b.w * c23.z);
        if (h < nq) {
            *reinterpret_cast<float4 *>(v + i) = ra;
            *reinterpret_cast<float4 *>(v + i + half) = rb;
        } else {
            const size_t dst = layer_base + (size_t(h - nq) * max_seq + pos) * hd;
            *reinterpret_cast<uint2 *>(kc + dst + i) = bf16x4(ra.x, ra.y, ra.z, ra.w);
            *reinterpret_cast<uint2 *>(kc + dst + i + half) = bf16x4(rb.x, rb.y, rb.z, rb.w);
        }
    }
    for (int u = 4 * int(threadIdx.x); u < kd; u += 4 * int(blockDim.x)) {
        const int g = u / hd, d = u % hd;
        const float4 x = *reinterpret_cast<const float4 *>(row + qd + kd + u);
        *reinterpret_cast<uint2 *>(vc + layer_base + (size_t(g) * max_seq + pos) * hd + d) = bf16x4(x.x, x.y, x.z, x.w);
    }
}

// Tensor-core causal attention of the prompt's positions. Block (16 positions,
// KV head g), 8 consumer warps and a producer warp. A warp takes two positions
// (one when the group has more than 4 query heads) and the G query heads of KV
// head g as the rows of an m16n8k16 A operand: row r < 8 is position r / G, head
// r % G, its q (scaled by 1/sqrt(hd)) as the hi bf16 term, row r + 8 the lo term.
// The producer streams the cache entries 0..pos0 + the block's last position in
// tiles of 16 positions through a ring of shared-memory stages by TMA (the
// tensor maps' 128-byte swizzle puts 16-byte chunk c of row r at c ^ (r % 8), so
// ldmatrix rows fall in different bank groups), each landing on the stage's
// mbarrier and released by the consumer warps' arrivals. Per tile: S = Q K^T (K
// rows by ldmatrix as B), each row's running max and sum over the 4 lanes
// holding it, P = exp(S - m) as hi and lo bf16 rows (already the A operand of
// P V), O += P V (V by ldmatrix.trans). Positions past a row's own are masked;
// V rows past the block's last position are read as zeros (the cache there may
// hold anything, and 0 * Inf is NaN).
// Blocks with the most positions to walk come first. Output: o as NTERMS terms.
__device__ __forceinline__ void mma16816(float (&d)[4], const uint4 &a, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a.x), "r"(a.y), "r"(a.z), "r"(a.w), "r"(b0), "r"(b1));
}
__device__ __forceinline__ void ldsm4(uint32_t addr, uint32_t (&r)[4]) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}
__device__ __forceinline__ void ldsm4t(uint32_t addr, uint32_t (&r)[4]) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t *>(&v);
}

constexpr int AT_NW = 8;      // consumer warps of an attention block
constexpr int AT_STAGES = 4;  // tiles in flight
// The running max of a row moves only once some row of the warp has grown past
// it by more than this (log2 units): until then probabilities are taken against
// the held max (each at most 2^8, well inside bf16 and fp32), the output needs
// no rescaling, and o / l is the same quotient.
constexpr float HOLD_LOG2 = 8.f;

struct PfAttnArgs {
    TensorMap kmap, vmap;  // the caches, boxes of 16 rows x 64 columns, 128-byte swizzle
    const float *qkv;      // [n][qd + 2 kd]
    int row0;              // cache row of (layer, KV head 0, position 0)
    int pos0, n, nq, nkv, max_seq;
    Terms o_t;
    int32_t *status;
    uint64_t timeout_ns;
};

template <int HD>
__global__ void __launch_bounds__((AT_NW + 1) * 32) k_pf_attn_tc(const __grid_constant__ PfAttnArgs a) {
    constexpr int DH = HD / 64, KS = HD / 16;  // 64-dim halves, k-steps
    constexpr uint32_t TILE_BYTES = 2u * DH * 16 * 128;
    __shared__ __align__(1024) uint8_t tile[AT_STAGES][2][DH][16][128];  // [stage][K | V][half][position][128 bytes]
    __shared__ __align__(8) uint64_t full[AT_STAGES], empty[AT_STAGES];
    __shared__ __align__(16) uint32_t zrow[4];  // a zero 16-byte row for ldmatrix
    __shared__ int err;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int gq = lane >> 2, tq = lane & 3, mi = lane >> 3, r8 = lane & 7;
    const int g = blockIdx.y, G = a.nq / a.nkv, qd = a.nq * HD, kd = a.nkv * HD;
    const int qpw = G <= 4 ? 2 : 1, qpb = AT_NW * qpw;  // positions per warp, per block
    const int t_base = (gridDim.x - 1 - int(blockIdx.x)) * qpb;  // the longest walks first
    const int block_last = a.pos0 + min(t_base + qpb - 1, a.n - 1);
    const int ntiles = block_last / 16 + 1;
    pdl_release();
    if (threadIdx.x == 0) {
        for (int st = 0; st < AT_STAGES; st++) {
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(saddr(&full[st])) : "memory");
            asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(saddr(&empty[st])), "r"(AT_NW) : "memory");
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        err = 0;
    }
    if (threadIdx.x < 4) zrow[threadIdx.x] = 0u;
    __syncthreads();
    pdl_wait();  // q (and the cache entries) as the previous kernel left them
    volatile int *errp = &err;
    if (warp == AT_NW) {  // producer
        if (lane == 0) {
            const int row = a.row0 + g * a.max_seq;
            int sent = 0;
            for (int ti = 0; ti < ntiles; ti++) {
                const int st = ti % AT_STAGES;
                if (ti >= AT_STAGES &&
                    !mbar_wait(&empty[st], ((ti / AT_STAGES) - 1) & 1, a.timeout_ns, a.status, errp))
                    break;
                asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(saddr(&full[st])),
                             "r"(TILE_BYTES)
                             : "memory");
#pragma unroll
                for (int h = 0; h < DH; h++) {
                    tma2d(saddr(&tile[st][0][h][0][0]), &a.kmap, 64 * h, row + 16 * ti, &full[st]);
                    tma2d(saddr(&tile[st][1][h][0][0]), &a.vmap, 64 * h, row + 16 * ti, &full[st]);
                }
                sent++;
            }
            // never leave with copies in flight into this block's shared memory
            for (int q = sent > AT_STAGES ? sent - AT_STAGES : 0; q < sent; q++) {
                const uint64_t t0 = now_ns();
                while (!mbar_try(&full[q % AT_STAGES], (q / AT_STAGES) & 1) && now_ns() - t0 < a.timeout_ns) {
                }
            }
        }
        return;
    }
    // this lane's row: position pi of the warp, head h of the group
    const bool row_ok = gq < qpw * G;
    const int pi = row_ok ? gq / G : 0, hh = row_ok ? gq % G : 0;
    const int t = t_base + warp * qpw + pi;
    const int last = a.pos0 + min(t, a.n - 1);                                 // this row's last position
    const int warp_last = a.pos0 + min(t_base + warp * qpw + qpw - 1, a.n - 1);  // the warp's
    // scores in log2 units (q scaled by log2(e) / sqrt(hd)), probabilities by exp2
    const float scale = 1.4426950408889634f / sqrtf(float(HD));
    // q as A fragments: k-step ks, lane (gq, tq): its row at dims 16 ks + 2tq, +1 (hi in x, lo in y) and +8, +9 (z, w)
    uint4 qa[KS];
#pragma unroll
    for (int ks = 0; ks < KS; ks++) {
        float v[4] = {0.f, 0.f, 0.f, 0.f};
        if (row_ok && t < a.n) {
            const float *qr = a.qkv + size_t(t) * (qd + 2 * kd) + size_t(g * G + hh) * HD + 16 * ks + 2 * tq;
            v[0] = qr[0] * scale;
            v[1] = qr[1] * scale;
            v[2] = qr[8] * scale;
            v[3] = qr[9] * scale;
        }
        const uint32_t h01 = pack_bf16(v[0], v[1]), h89 = pack_bf16(v[2], v[3]);
        const __nv_bfloat162 b01 = *reinterpret_cast<const __nv_bfloat162 *>(&h01);
        const __nv_bfloat162 b89 = *reinterpret_cast<const __nv_bfloat162 *>(&h89);
        qa[ks] = make_uint4(h01, pack_bf16(v[0] - __low2float(b01), v[1] - __high2float(b01)), h89,
                            pack_bf16(v[2] - __low2float(b89), v[3] - __high2float(b89)));
    }
    float m_run = -INFINITY, l_run = 0.f, o[HD / 8][2];
#pragma unroll
    for (int d = 0; d < HD / 8; d++) o[d][0] = o[d][1] = 0.f;
    // 128-dim heads: two tiles (32 positions) per softmax round, one max, sum and
    // rescale for both (3B at 2048 positions 34.3 -> 32.7 ms, 8B at 8192 376 ->
    // 346 ms); 64-dim heads: one tile per round (two measured slower: 1B
    // attention 73 -> 86 us per layer)
    if constexpr (HD == 128) {
        constexpr int TPR = 2;
        static_assert(AT_STAGES % TPR == 0, "a round's tiles are consecutive stages");
        bool fail = false;
        for (int ti = 0; ti < ntiles && !fail; ti += TPR) {
            const int nt = min(TPR, ntiles - ti);  // tiles in this round
            int st[TPR];
            for (int u = 0; u < nt; u++) {
                st[u] = (ti + u) % AT_STAGES;
                if (!mbar_wait(&full[st[u]], ((ti + u) / AT_STAGES) & 1, a.timeout_ns, a.status, errp)) fail = true;
            }
            if (fail) break;
            if (16 * ti <= warp_last) {
                // S = Q K^T: c[u][nb] holds positions 16 (ti + u) + 8 nb .. + 7
                float c[TPR][2][4] = {};
                const int jk = 8 * (mi >> 1) + r8;  // this lane's ldmatrix row: position in the tile
    #pragma unroll
                for (int u = 0; u < TPR; u++) {
                    if (u >= nt) break;
    #pragma unroll
                    for (int ks = 0; ks < KS; ks++) {
                        const uint32_t ch = uint32_t(2 * (ks & 3) + (mi & 1));
                        uint32_t b[4];
                        ldsm4(saddr(&tile[st[u]][0][ks >> 2][jk][(ch ^ uint32_t(jk & 7)) * 16]), b);
                        mma16816(c[u][0], qa[ks], b[0], b[1]);
                        mma16816(c[u][1], qa[ks], b[2], b[3]);
                    }
                }
                float sc[4 * TPR];
    #pragma unroll
                for (int u = 0; u < TPR; u++)
    #pragma unroll
                    for (int nb = 0; nb < 2; nb++)
    #pragma unroll
                        for (int e = 0; e < 2; e++) {
                            const int j = 16 * (ti + u) + 8 * nb + 2 * tq + e;
                            sc[4 * u + 2 * nb + e] = u < nt && j <= last ? c[u][nb][e] + c[u][nb][e + 2] : -INFINITY;
                        }
                float mt = sc[0];
    #pragma unroll
                for (int e = 1; e < 4 * TPR; e++) mt = fmaxf(mt, sc[e]);
                mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, 1));
                mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, 2));
                // (a row past its last position in this round keeps its state: m_new = m_run)
                const float m_cand = fmaxf(m_run, mt);
                const bool hold = __all_sync(0xffffffffu, m_cand - m_run <= HOLD_LOG2);
                const float m_new = hold ? m_run : m_cand;
                const float alpha = m_run == m_new ? 1.f : (m_run == -INFINITY ? 0.f : exp2f(m_run - m_new));
                float pr[4 * TPR], ps = 0.f;
    #pragma unroll
                for (int e = 0; e < 4 * TPR; e++) {
                    pr[e] = sc[e] == -INFINITY ? 0.f : exp2f(sc[e] - m_new);
                    ps += pr[e];
                }
                ps += __shfl_xor_sync(0xffffffffu, ps, 1);
                ps += __shfl_xor_sync(0xffffffffu, ps, 2);
                l_run = l_run * alpha + ps;
                m_run = m_new;
                uint4 pa[TPR];
    #pragma unroll
                for (int u = 0; u < TPR; u++) {
                    const float *q4 = pr + 4 * u;
                    const uint32_t h01 = pack_bf16(q4[0], q4[1]), h23 = pack_bf16(q4[2], q4[3]);
                    const __nv_bfloat162 b01 = *reinterpret_cast<const __nv_bfloat162 *>(&h01);
                    const __nv_bfloat162 b23 = *reinterpret_cast<const __nv_bfloat162 *>(&h23);
                    pa[u] = make_uint4(h01, pack_bf16(q4[0] - __low2float(b01), q4[1] - __high2float(b01)), h23,
                                       pack_bf16(q4[2] - __low2float(b23), q4[3] - __high2float(b23)));
                }
                // O += P V: 8 dims per product, two per ldmatrix
                // (V rows past the block's last position read a zero row instead: the
                // cache there may hold anything, and 0 * Inf is NaN)
                const int jv = 8 * (mi & 1) + r8;
    #pragma unroll
                for (int dd = 0; dd < HD / 16; dd++) {
                    const uint32_t ch = uint32_t(2 * (dd & 3) + (mi >> 1));
                    uint32_t b[TPR][4];
    #pragma unroll
                    for (int u = 0; u < TPR; u++) {
                        const bool vrow = u < nt && 16 * (ti + u) + jv <= block_last;
                        ldsm4t(vrow ? saddr(&tile[st[u < nt ? u : 0]][1][dd >> 2][jv][(ch ^ uint32_t(jv & 7)) * 16])
                                    : saddr(zrow),
                               b[u]);
                    }
    #pragma unroll
                    for (int v = 0; v < 2; v++) {
                        const int d = 2 * dd + v;
                        float acc[4] = {o[d][0] * alpha, o[d][1] * alpha, 0.f, 0.f};
    #pragma unroll
                        for (int u = 0; u < TPR; u++) mma16816(acc, pa[u], b[u][2 * v], b[u][2 * v + 1]);
                        o[d][0] = acc[0] + acc[2];
                        o[d][1] = acc[1] + acc[3];
                    }
                }
            }
            __syncwarp();
            if (lane == 0)
                for (int u = 0; u < nt; u++)
                    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(saddr(&empty[st[u]])) : "memory");
        }
    } else {
        for (int ti = 0; ti < ntiles; ti++) {
            const int st = ti % AT_STAGES, j0 = 16 * ti;
            if (!mbar_wait(&full[st], (ti / AT_STAGES) & 1, a.timeout_ns, a.status, errp)) break;
            if (j0 <= warp_last) {
                // S = Q K^T: c[nb] holds positions j0 + 8 nb .. + 7
                float c[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
                const int jk = 8 * (mi >> 1) + r8;  // this lane's ldmatrix row: position in the tile
    #pragma unroll
                for (int ks = 0; ks < KS; ks++) {
                    const uint32_t ch = uint32_t(2 * (ks & 3) + (mi & 1));
                    uint32_t b[4];
                    ldsm4(saddr(&tile[st][0][ks >> 2][jk][(ch ^ uint32_t(jk & 7)) * 16]), b);
                    mma16816(c[0], qa[ks], b[0], b[1]);
                    mma16816(c[1], qa[ks], b[2], b[3]);
                }
                float sc[4];
    #pragma unroll
                for (int nb = 0; nb < 2; nb++)
    #pragma unroll
                    for (int e = 0; e < 2; e++) {
                        const int j = j0 + 8 * nb + 2 * tq + e;
                        sc[2 * nb + e] = j <= last ? c[nb][e] + c[nb][e + 2] : -INFINITY;
                    }
                float mt = fmaxf(fmaxf(sc[0], sc[1]), fmaxf(sc[2], sc[3]));
                mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, 1));
                mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, 2));
                // (a row past its last position in this tile keeps its state: m_new = m_run)
                const float m_cand = fmaxf(m_run, mt);
                const bool hold = __all_sync(0xffffffffu, m_cand - m_run <= HOLD_LOG2);
                const float m_new = hold ? m_run : m_cand;
                const float alpha = m_run == m_new ? 1.f : (m_run == -INFINITY ? 0.f : exp2f(m_run - m_new));
                float pr[4], ps = 0.f;
    #pragma unroll
                for (int e = 0; e < 4; e++) {
                    pr[e] = sc[e] == -INFINITY ? 0.f : exp2f(sc[e] - m_new);
                    ps += pr[e];
                }
                ps += __shfl_xor_sync(0xffffffffu, ps, 1);
                ps += __shfl_xor_sync(0xffffffffu, ps, 2);
                l_run = l_run * alpha + ps;
                m_run = m_new;
                const uint32_t h01 = pack_bf16(pr[0], pr[1]), h23 = pack_bf16(pr[2], pr[3]);
                const __nv_bfloat162 b01 = *reinterpret_cast<const __nv_bfloat162 *>(&h01);
                const __nv_bfloat162 b23 = *reinterpret_cast<const __nv_bfloat162 *>(&h23);
                const uint4 pa = make_uint4(h01, pack_bf16(pr[0] - __low2float(b01), pr[1] - __high2float(b01)), h23,
                                            pack_bf16(pr[2] - __low2float(b23), pr[3] - __high2float(b23)));
                // O += P V: 8 dims per product, two per ldmatrix
                // (V rows past the block's last position read a zero row instead: the
                // cache there may hold anything, and 0 * Inf is NaN)
                const int jv = 8 * (mi & 1) + r8;
                const bool vrow = j0 + jv <= block_last;
    #pragma unroll
                for (int dd = 0; dd < HD / 16; dd++) {
                    const uint32_t ch = uint32_t(2 * (dd & 3) + (mi >> 1));
                    uint32_t b[4];
                    ldsm4t(vrow ? saddr(&tile[st][1][dd >> 2][jv][(ch ^ uint32_t(jv & 7)) * 16]) : saddr(zrow), b);
    #pragma unroll
                    for (int u = 0; u < 2; u++) {
                        const int d = 2 * dd + u;
                        float acc[4] = {o[d][0] * alpha, o[d][1] * alpha, 0.f, 0.f};
                        mma16816(acc, pa, b[2 * u], b[2 * u + 1]);
                        o[d][0] = acc[0] + acc[2];
                        o[d][1] = acc[1] + acc[3];
                    }
                }
            }
            __syncwarp();
            if (lane == 0) asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(saddr(&empty[st])) : "memory");
        }
    }
    if (*errp || !row_ok || t >= a.n) return;
    // lane (gq, tq) holds its row at dims 8 d + 2 tq, + 1
    const size_t at = size_t(t) * qd + size_t(g * G + hh) * HD;
    const float inv = 1.0f / l_run;
#pragma unroll
    for (int d = 0; d < HD / 8; d++) {
        put_terms(o[d][0] * inv, a.o_t.t, at + 8 * d + 2 * tq);
        put_terms(o[d][1] * inv, a.o_t.t, at + 8 * d + 2 * tq + 1);
    }
}

int launch_attention(const KParams &p, const PrefillBufs &b, int layer, int pos0, int n, const Terms &to,
                     cudaStream_t st) {
    PfAttnArgs a;
    a.kmap = b.m_k;
    a.vmap = b.m_v;
    a.qkv = b.qkv;
    a.row0 = layer * p.nkv * p.max_seq;
    a.pos0 = pos0;
    a.n = n;
    a.nq = p.nq;
    a.nkv = p.nkv;
    a.max_seq = p.max_seq;
    a.o_t = to;
    a.status = p.status;
    a.timeout_ns = p.timeout_ns;
    const int qpb = AT_NW * (p.nq / p.nkv <= 4 ? 2 : 1);
    const dim3 grid((n + qpb - 1) / qpb, p.nkv);
    const cudaError_t e = p.hd == 64 ? launch_pdl(k_pf_attn_tc<64>, grid, dim3((AT_NW + 1) * 32), 0, st, a)
                                     : launch_pdl(k_pf_attn_tc<128>, grid, dim3((AT_NW + 1) * 32), 0, st, a);
    return e == cudaSuccess ? LL_OK : LL_ERR_CUDA;
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

// C = A B^T with B the nb (1 to 3) matrices bm[] stacked by output column (at
// splits s1, s2: multiples of GN), or, for EPI_GATEUP, the gate and up matrices.
template <int EPI>
int gemm(const TensorMap *a, const TensorMap *bm, int nb, int s1, int s2, int M, int N, int K, float *c, int ldc,
         const Terms *act, const KParams &p, cudaStream_t st) {
    constexpr int NB = EPI == EPI_GATEUP ? 2 : 1;
    constexpr int SMEM = gstages(gterms(EPI) + NB) * int(GTILE) * (gterms(EPI) + NB) + 1024;
    static_assert(SMEM <= 232448, "stages fit in shared memory");
    GemmArgs g;
    for (int q = 0; q < NTERMS; q++) {
        g.a[q] = a[q];
        g.act[q] = act ? act->t[q] : nullptr;
    }
    for (int j = 0; j < 3; j++) g.b[j] = bm[j < nb ? j : 0];
    g.bsplit1 = nb > 1 && EPI != EPI_GATEUP ? s1 : 1 << 30;
    g.bsplit2 = nb > 2 && EPI != EPI_GATEUP ? s2 : 1 << 30;
    g.M = M;
    g.N = N;
    g.K = K;
    g.c = c;
    g.ldc = ldc;
    g.status = p.status;
    g.timeout_ns = p.timeout_ns;
    static bool attr = false;
    if (!attr) {
        if (cudaFuncSetAttribute(k_gemm<EPI>, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM) != cudaSuccess)
            return LL_ERR_CUDA;
        attr = true;
    }
    // persistent: at most one block per SM, each walking its share of the tiles
    const int ntiles = ((N + GN - 1) / GN) * ((M + GM - 1) / GM);
    return launch_pdl(k_gemm<EPI>, dim3(std::min(ntiles, p.nsm)), dim3(GTHREADS), size_t(SMEM), st, g) == cudaSuccess
               ? LL_OK
               : LL_ERR_CUDA;
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
                 sz_o = r256(na * qd * 2), sz_a = r256(na * I * 2), sz_hr = r256(H * 4),
                 sz_l = r256(size_t(p.V) * 4);
    const size_t total = sz_x + NTERMS * sz_h + sz_qkv + NTERMS * sz_o + NTERMS * sz_a + sz_hr + sz_l;
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
    for (int q = 0; q < NTERMS; q++) b.a[q] = reinterpret_cast<uint16_t *>(take(sz_a));
    b.hrow = reinterpret_cast<float *>(take(sz_hr));
    b.logits = reinterpret_cast<float *>(take(sz_l));
    b.n_alloc = int(na);
    bool ok = true;
    for (int q = 0; q < NTERMS && ok; q++)
        ok = encode_operand(b.h[q], int64_t(na), p.H, b.m_h[q]) && encode_operand(b.o[q], int64_t(na), int(qd), b.m_o[q]) &&
             encode_operand(b.a[q], int64_t(na), p.I, b.m_a[q]);
    {  // the caches, [L * n_kv * max_seq][hd], in tiles of 16 rows x 64 columns
        EncodeTiled enc = encoder();
        const int64_t rows = int64_t(p.L) * p.nkv * p.max_seq;
        const cuuint64_t dims[2] = {cuuint64_t(p.hd), cuuint64_t(rows)};
        const cuuint64_t strides[1] = {cuuint64_t(p.hd) * 2};
        const cuuint32_t box[2] = {64, 16}, estr[2] = {1, 1};
        for (int i = 0; i < 2 && ok; i++) {
            CUtensorMap m;
            ok = enc && rows < (int64_t(1) << 31) &&
                 enc(&m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, i ? p.v_cache : p.k_cache, dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
            if (ok) std::memcpy(i ? &b.m_v : &b.m_k, &m, sizeof m);
        }
    }
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
    const int norm_threads = std::min(1024, (H / 8 + 31) / 32 * 32);  // a thread per 8 elements of a row
    k_pf_embed<<<n, 256, 0, st>>>(p.embed, tokens_dev, n, H, p.V, b.x, p.status);
    int rc = cudaGetLastError() == cudaSuccess ? LL_OK : LL_ERR_CUDA;
    for (int l = 0; l < p.L && rc == LL_OK; l++) {
        const LayerW &w = host_layers[l];
        const TensorMap *m = &b.m_w[size_t(l) * 7];
        const size_t lb = size_t(l) * per_layer;
        const int ld = qd + 2 * kd;
        auto ok = [](cudaError_t e) { return e == cudaSuccess ? LL_OK : LL_ERR_CUDA; };
        // every launch of the layer's chain lets the next one start early (see pdl_wait)
        rc = ok(launch_pdl(k_pf_norm_split, dim3(n), dim3(norm_threads), 0, st, (const float *)b.x,
                           (const uint16_t *)w.attn_norm, H, p.eps, th));
        if (rc == LL_OK && qd % GN == 0 && kd % GN == 0) {  // q, k and v in one GEMM over the stacked rows
            rc = gemm<EPI_STORE>(b.m_h, m, 3, qd, qd + kd, n, ld, H, b.qkv, ld, nullptr, p, st);
        } else if (rc == LL_OK) {
            rc = gemm<EPI_STORE>(b.m_h, m, 1, 0, 0, n, qd, H, b.qkv, ld, nullptr, p, st);
            if (rc == LL_OK) rc = gemm<EPI_STORE>(b.m_h, m + 1, 1, 0, 0, n, kd, H, b.qkv + qd, ld, nullptr, p, st);
            if (rc == LL_OK) rc = gemm<EPI_STORE>(b.m_h, m + 2, 1, 0, 0, n, kd, H, b.qkv + qd + kd, ld, nullptr, p, st);
        }
        if (rc == LL_OK)
            rc = ok(launch_pdl(k_pf_rope_kv, dim3(n), dim3(256), 0, st, b.qkv, (const float2 *)p.rope_cs, pos0, p.nq,
                               p.nkv, p.hd, p.k_cache, p.v_cache, lb, p.max_seq));
        if (rc == LL_OK) rc = launch_attention(p, b, l, pos0, n, to, st);
        if (rc == LL_OK) rc = gemm<EPI_ADD>(b.m_o, m + 3, 1, 0, 0, n, H, qd, b.x, H, nullptr, p, st);
        if (rc == LL_OK)
            rc = ok(launch_pdl(k_pf_norm_split, dim3(n), dim3(norm_threads), 0, st, (const float *)b.x,
                               (const uint16_t *)w.mlp_norm, H, p.eps, th));
        // gate and up in one GEMM (two accumulators), silu(gate) * up as terms
        if (rc == LL_OK) rc = gemm<EPI_GATEUP>(b.m_h, m + 4, 2, 0, 0, n, I, H, nullptr, I, &ta, p, st);
        if (rc == LL_OK) rc = gemm<EPI_ADD>(b.m_a, m + 6, 1, 0, 0, n, H, I, b.x, H, nullptr, p, st);
    }
    if (rc != LL_OK) return rc;
    if (cudaGetLastError() != cudaSuccess) return LL_ERR_CUDA;
    return launch_chain_head(p, b.x + size_t(n - 1) * H, b.hrow, logits ? logits : b.logits, next_dev, stream_);
}

}  // namespace ll
