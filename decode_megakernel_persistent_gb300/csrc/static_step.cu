// static_step.cu -- ll_decode_step_static: one decode step that allocates no
// device memory, for callers that cannot call cudaMalloc.
//
// It runs the one-kernel-per-operation path (chain.cu) with every scratch
// buffer carved out of one file-scope __device__ array of LL_STATIC_SCRATCH_BYTES
// bytes, whose address is looked up once per device. The RoPE row of the step's
// position is computed on the host in double precision, as ll_init computes its
// table, and copied into that array. Nothing here calls cudaMalloc, cudaFree or
// any allocating routine; the only per-call host state is on the stack.
//
// Every call on a device shares the one array, so calls whose GPU work overlaps
// (on different streams, or from different threads) race on it.
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdint>
#include <cstdio>
#include <mutex>

#include "ll_internal.h"

namespace {

constexpr size_t SCRATCH_BYTES = LL_STATIC_SCRATCH_BYTES;
constexpr int MAX_DEVICES = 64;

static __device__ __align__(256) uint8_t g_scratch[SCRATCH_BYTES];

struct DeviceSetup {
    bool done = false;
    uint8_t *scratch = nullptr;  // device address of g_scratch on this device
    int nsm = 0;
};

std::mutex g_setup_mu;
DeviceSetup g_setup[MAX_DEVICES];

int report(char *err, size_t err_len, int code, const char *fmt, ...) {
    if (err && err_len) {
        va_list ap;
        va_start(ap, fmt);
        std::vsnprintf(err, err_len, fmt, ap);
        va_end(ap);
    }
    return code;
}

bool aligned16(const void *p) { return p && (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

size_t round256(size_t n) { return (n + 255) / 256 * 256; }

// Once per device, with that device current: the address of g_scratch there,
// and the device's SM count (the launch grids of the per-operation kernels).
int setup_device(int dev, DeviceSetup &out, char *err, size_t err_len) {
    if (dev < 0 || dev >= MAX_DEVICES) return report(err, err_len, LL_ERR_DEVICE, "device ordinal %d out of range", dev);
    std::lock_guard<std::mutex> lock(g_setup_mu);
    DeviceSetup &d = g_setup[dev];
    if (!d.done) {
        int major = 0, minor = 0, nsm = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return report(err, err_len, LL_ERR_CUDA, "cannot query device %d", dev);
        if (major != 10 || minor != 3)
            return report(err, err_len, LL_ERR_DEVICE, "device is sm_%d%d, this library is built for sm_103a", major,
                          minor);
        void *ptr = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&ptr, g_scratch);
        if (e != cudaSuccess || !ptr)
            return report(err, err_len, LL_ERR_CUDA, "cudaGetSymbolAddress of the static scratch failed: %s",
                          cudaGetErrorString(e));
        d.scratch = static_cast<uint8_t *>(ptr);
        d.nsm = nsm;
        d.done = true;
    }
    out = d;
    return LL_OK;
}

}  // namespace

extern "C" int ll_decode_step_static(const ll_config *cfg, const ll_weights *w, uint16_t *k_cache,
                                     uint16_t *v_cache, int32_t token, int32_t pos, float *logits_dev,
                                     int32_t *next_token_host, void *stream, char *err, size_t err_len) {
    if (err && err_len) err[0] = '\0';
    if (!cfg || !w) return report(err, err_len, LL_ERR_ARG, "cfg or weights is NULL");
    const ll_config c = *cfg;
    // ---- shapes: the limits of ll_init, plus the layer count of the host-side table
    if (c.n_layers < 1 || c.hidden <= 0 || c.n_q_heads <= 0 || c.n_kv_heads <= 0 || c.inter <= 0 ||
        c.vocab <= 0 || c.max_seq <= 0)
        return report(err, err_len, LL_ERR_SHAPE, "every size must be positive");
    if (c.n_layers > LL_STATIC_MAX_LAYERS)
        return report(err, err_len, LL_ERR_SHAPE, "n_layers %d exceeds LL_STATIC_MAX_LAYERS (%d)", c.n_layers,
                      LL_STATIC_MAX_LAYERS);
    if (c.head_dim != 64 && c.head_dim != 128) return report(err, err_len, LL_ERR_SHAPE, "head_dim must be 64 or 128");
    if (c.n_q_heads % c.n_kv_heads != 0 || c.n_q_heads / c.n_kv_heads > ll::MAX_GQA ||
        (c.n_q_heads / c.n_kv_heads) * c.head_dim > 512)
        return report(err, err_len, LL_ERR_SHAPE,
                      "n_q_heads must be a multiple (at most 8x) of n_kv_heads, with group*head_dim <= 512");
    const int qd = c.n_q_heads * c.head_dim, kd = c.n_kv_heads * c.head_dim, half = c.head_dim / 2;
    ll::MvShape m{};
    if (qd > ll::XIN_FLOATS || !ll::mv_shape(c.hidden, m) || !ll::mv_shape(qd, m) || !ll::mv_shape(c.inter, m))
        return report(err, err_len, LL_ERR_SHAPE,
                      "hidden, n_q_heads*head_dim (<= 4096) and inter must be multiples of 256, at most 16384");
    if (!(c.rms_eps >= 0.f) || !(c.rope_theta > 0.f)) return report(err, err_len, LL_ERR_ARG, "rms_eps/rope_theta invalid");
    // ---- step arguments and pointers
    if (token < 0 || token >= c.vocab) return report(err, err_len, LL_ERR_ARG, "token %d out of range", token);
    if (pos < 0 || pos >= c.max_seq) return report(err, err_len, LL_ERR_ARG, "pos %d out of range", pos);
    if (!aligned16(k_cache) || !aligned16(v_cache))
        return report(err, err_len, LL_ERR_ARG, "KV caches must be 16-byte aligned");
    if (!aligned16(w->embed) || !aligned16(w->final_norm) || (!c.tied && !aligned16(w->lm_head)))
        return report(err, err_len, LL_ERR_ARG, "embed, final_norm and lm_head must be 16-byte aligned");
    if (logits_dev && !aligned16(logits_dev)) return report(err, err_len, LL_ERR_ARG, "logits_dev not 16-byte aligned");
    const uint16_t *const *lp[9] = {w->attn_norm, w->wq, w->wk, w->wv, w->wo, w->mlp_norm, w->wg, w->wu, w->wd};
    for (auto a : lp)
        if (!a) return report(err, err_len, LL_ERR_ARG, "a per-layer pointer array is NULL");
    ll::LayerW layers[LL_STATIC_MAX_LAYERS];
    for (int l = 0; l < c.n_layers; l++) {
        layers[l] = {w->attn_norm[l], w->wq[l], w->wk[l], w->wv[l], w->wo[l], w->mlp_norm[l], w->wg[l], w->wu[l], w->wd[l]};
        const uint16_t *all[9] = {layers[l].attn_norm, layers[l].wq, layers[l].wk, layers[l].wv, layers[l].wo,
                                  layers[l].mlp_norm, layers[l].wg, layers[l].wu, layers[l].wd};
        for (auto a : all)
            if (!aligned16(a)) return report(err, err_len, LL_ERR_ARG, "layer %d weight not 16-byte aligned", l);
    }
    // ---- the device's static scratch
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return report(err, err_len, LL_ERR_CUDA, "no CUDA device");
    DeviceSetup ds;
    int rc = setup_device(dev, ds, err, err_len);
    if (rc != LL_OK) return rc;
    // KV splits as the handle path picks them
    const int splits = ll::attn_splits(c.max_seq, c.n_kv_heads, ds.nsm);
    const size_t F = sizeof(float);
    const size_t sz[] = {
        round256(size_t(c.hidden) * F),                                           // x
        round256(size_t(c.hidden) * F),                                           // h
        round256(size_t(qd + 2 * kd) * F),                                        // qkv
        round256(size_t(c.n_q_heads) * splits * (c.head_dim + 2) * F),            // attention partials
        round256(size_t(qd) * F),                                                 // o
        round256(size_t(c.inter) * F),                                            // gate
        round256(size_t(c.inter) * F),                                            // up
        round256(size_t(c.inter) * F),                                            // act
        logits_dev ? size_t(0) : round256(size_t(c.vocab) * F),                   // logits
        round256(size_t(half) * sizeof(float2)),                                  // RoPE row of pos
        256,                                                                      // status, next token
    };
    size_t need = 0;
    for (size_t s : sz) need += s;
    if (need > SCRATCH_BYTES)
        return report(err, err_len, LL_ERR_SHAPE,
                      "this shape needs %zu bytes of scratch; the static array holds %zu (LL_STATIC_SCRATCH_BYTES)",
                      need, SCRATCH_BYTES);
    uint8_t *cur = ds.scratch;
    auto take = [&](size_t bytes) {
        uint8_t *p = cur;
        cur += bytes;
        return p;
    };
    ll::ChainBufs cb{};
    cb.host_layers = layers;
    cb.x = reinterpret_cast<float *>(take(sz[0]));
    cb.h = reinterpret_cast<float *>(take(sz[1]));
    cb.qkv = reinterpret_cast<float *>(take(sz[2]));
    cb.part = reinterpret_cast<float *>(take(sz[3]));
    cb.o = reinterpret_cast<float *>(take(sz[4]));
    cb.gate = reinterpret_cast<float *>(take(sz[5]));
    cb.up = reinterpret_cast<float *>(take(sz[6]));
    cb.act = reinterpret_cast<float *>(take(sz[7]));
    cb.logits = reinterpret_cast<float *>(take(sz[8]));
    cb.splits = splits;
    float2 *rope_row = reinterpret_cast<float2 *>(take(sz[9]));
    cb.rope_row = rope_row;  // the per-operation RoPE kernel reads this row as given
    int32_t *words = reinterpret_cast<int32_t *>(take(sz[10]));  // [0] status, [1] next token

    // RoPE (cos, sin) of position pos, in double as ll_init builds its table
    float2 rope[ll::MAX_HD / 2];
    for (int i = 0; i < half; i++) {
        const double inv = std::pow(static_cast<double>(c.rope_theta), -2.0 * i / c.head_dim);
        const double a = static_cast<double>(pos) * inv;
        rope[i] = make_float2(static_cast<float>(std::cos(a)), static_cast<float>(std::sin(a)));
    }

    ll::KParams p{};
    p.nsm = ds.nsm;
    p.embed = w->embed;
    p.lm_head = c.tied ? w->embed : w->lm_head;
    p.final_norm = w->final_norm;
    p.k_cache = k_cache;
    p.v_cache = v_cache;
    p.rope_cs = nullptr;  // no table here: cb.rope_row holds the one row the step needs
    p.L = c.n_layers;
    p.H = c.hidden;
    p.nq = c.n_q_heads;
    p.nkv = c.n_kv_heads;
    p.hd = c.head_dim;
    p.I = c.inter;
    p.V = c.vocab;
    p.max_seq = c.max_seq;
    p.eps = c.rms_eps;
    p.attn_splits = splits;
    p.status = words;
    p.token_out = words + 1;
    p.token = token;
    p.token_dev = nullptr;
    p.pos = pos;
    p.logits = logits_dev;
    p.next_token_dev = nullptr;

    cudaStream_t st = static_cast<cudaStream_t>(stream);
    // what must start at zero: the status word (the next token is always written)
    if (cudaMemsetAsync(words, 0, 2 * sizeof(int32_t), st) != cudaSuccess ||
        cudaMemcpyAsync(rope_row, rope, size_t(half) * sizeof(float2), cudaMemcpyHostToDevice, st) != cudaSuccess)
        return report(err, err_len, LL_ERR_CUDA, "scratch set-up failed: %s", cudaGetErrorString(cudaGetLastError()));
    rc = ll::launch_chain_step(p, cb, stream);
    if (rc != LL_OK) return report(err, err_len, rc, "launch failed: %s", cudaGetErrorString(cudaGetLastError()));
    int32_t out[2] = {0, -1};
    if (cudaMemcpyAsync(out, words, sizeof(out), cudaMemcpyDeviceToHost, st) != cudaSuccess ||
        cudaStreamSynchronize(st) != cudaSuccess)
        return report(err, err_len, LL_ERR_CUDA, "step failed: %s", cudaGetErrorString(cudaGetLastError()));
    if (out[0] != LL_OK) return report(err, err_len, out[0], "the device reported status %d", out[0]);
    if (next_token_host) *next_token_host = out[1];
    return LL_OK;
}
