// api.cpp -- the C ABI of libll.so (declared in include/ll.h): argument and
// shape checks, library memory, the RoPE table, schedule upload, launches and
// status handling.
#include <cuda.h>  // CUtensorMap and its enums (the encoder itself is fetched from the driver)
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <string>
#include <vector>

#include "ll_internal.h"

using ll::Instr;
using ll::KParams;

struct ll_handle {
    ll_config cfg{};
    int device = 0;
    int nsm = 0;
    int splits = 1;
    int smem_bytes = 0;
    cudaStream_t stream = nullptr;
    uint8_t *dmem = nullptr;
    size_t dmem_bytes = 0;
    KParams kp{};
    ll::ChainBufs cb{};
    std::vector<ll::LayerW> host_layers;
    ll::PrefillBufs pf;          // prefill buffers, allocated by the first ll_prefill (grown by a longer one)
    std::vector<std::vector<Instr>> lists;
    Instr *d_instrs = nullptr;
    int max_instr = 0;
    uint32_t epoch = 0;
    int nb = 1;                 // sequences decoded together (batched handles)
    bool batch_api = false;     // made by ll_init_batch: only ll_decode_steps_batch steps it
    bool bcc = false;           // a batch of two on CUDA-core pages (mv_shape_bc geometry)
    int32_t *pinned = nullptr;  // [0, nb) next tokens, [nb] status
    uint8_t *tagged = nullptr;  // the megakernel's tagged activation words (cleared on reset)
    size_t tagged_bytes = 0;
    std::string err;
};

namespace {

thread_local std::string g_init_error;

int fail(ll_handle *h, int code, const std::string &msg) {
    if (h) h->err = msg;
    return code;
}

bool aligned16(const void *p) { return p && (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

size_t round_up(size_t n, size_t a) { return (n + a - 1) / a * a; }

int upload_schedule(ll_handle *h) {
    std::vector<Instr> flat(size_t(h->nsm) * h->max_instr);
    std::vector<int32_t> counts(h->nsm);
    for (int sm = 0; sm < h->nsm; sm++) {
        counts[sm] = static_cast<int32_t>(h->lists[sm].size());
        std::copy(h->lists[sm].begin(), h->lists[sm].end(), flat.begin() + size_t(sm) * h->max_instr);
    }
    if (cudaMemcpy(h->d_instrs, flat.data(), flat.size() * sizeof(Instr), cudaMemcpyHostToDevice) != cudaSuccess ||
        cudaMemcpy(const_cast<int32_t *>(h->kp.n_instr), counts.data(), counts.size() * sizeof(int32_t),
                   cudaMemcpyHostToDevice) != cudaSuccess)
        return fail(h, LL_ERR_CUDA, "schedule upload failed");
    return LL_OK;
}

// The KV tensor maps of the per-warp attention variant (ll::TM_*): each cache as
// a 2-D bf16 tensor of head_dim columns and L * n_kv * max_seq rows, boxes of 64
// columns (128 bytes, the widest the 128-byte swizzle takes) by a page of rows or
// by one 16-row tile. False if the driver has no encoder or the rows do not fit
// the 32-bit signed coordinates of a copy.
bool encode_kv_maps(const ll_config &c, uint16_t *k_cache, uint16_t *v_cache, ll::TensorMap (&out)[ll::TM_COUNT]) {
    using EncodeTiled = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                     const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                     CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
    static_assert(sizeof(CUtensorMap) == sizeof(ll::TensorMap), "tensor map size");
    void *fn = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess || !fn) {
        cudaGetLastError();
        return false;
    }
    const auto encode = reinterpret_cast<EncodeTiled>(fn);
    const uint64_t rows = uint64_t(c.n_layers) * uint64_t(c.n_kv_heads) * uint64_t(c.max_seq);
    if (rows + ll::PAGE_BYTES >= (1ull << 31)) return false;
    const cuuint64_t dims[2] = {cuuint64_t(c.head_dim), cuuint64_t(rows)};
    const cuuint64_t strides[1] = {cuuint64_t(c.head_dim) * 2};
    const cuuint32_t page_rows = ll::PAGE_BYTES / (4 * c.head_dim), estr[2] = {1, 1};
    for (int i = 0; i < ll::TM_COUNT; i++) {
        const bool tile = i == ll::TM_K_TILE || i == ll::TM_V_TILE;
        const cuuint32_t box[2] = {64, tile ? cuuint32_t(ll::ATT_TILE) : page_rows};
        CUtensorMap m;
        if (encode(&m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, i < ll::TM_V_PAGE ? k_cache : v_cache, dims, strides, box,
                   estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return false;
        std::memcpy(&out[i], &m, sizeof m);
    }
    return true;
}

// The weight tensor maps of tensor-core pages (ll::wmap_index): each matrix as a
// 3-D bf16 tensor (64 columns, rows, K / 64 column blocks) with boxes of
// (64, nr, K / 64) for nr = 1..TC_ROWS, in the 128-byte swizzle, so that one copy
// brings nr whole rows in the layout the tensor-core page reads. Maps of
// matrices whose width has no tensor-core geometry stay zero. False if the
// driver has no encoder or refuses a map.
bool encode_weight_maps(const ll_config &c, const std::vector<ll::LayerW> &layers, const uint16_t *lm_head,
                        const ll::MvShape &mh, const ll::MvShape &mq, const ll::MvShape &mi,
                        std::vector<ll::TensorMap> &out) {
    using EncodeTiled = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                     const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                     CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
    void *fn = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess || !fn) {
        cudaGetLastError();
        return false;
    }
    const auto encode = reinterpret_cast<EncodeTiled>(fn);
    out.assign(size_t(c.n_layers + 1) * ll::TC_MATS_PER_LAYER * ll::TC_ROWS, ll::TensorMap{});
    // boxes of one column chunk (kc columns) of nr rows
    auto one = [&](const uint16_t *w, int64_t rows, int K, int kc, int l, int m) -> bool {
        const cuuint64_t dims[3] = {64, cuuint64_t(rows), cuuint64_t(K / 64)};
        const cuuint64_t strides[2] = {cuuint64_t(K) * 2, 128};  // bytes: next row, next 64-column block
        const cuuint32_t estr[3] = {1, 1, 1};
        for (int nr = 1; nr <= ll::TC_ROWS; nr++) {
            const cuuint32_t box[3] = {64, cuuint32_t(nr), cuuint32_t(kc / 64)};
            CUtensorMap map;
            if (encode(&map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<uint16_t *>(w), dims, strides, box, estr,
                       CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                       CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
                return false;
            std::memcpy(&out[ll::wmap_index(l, m, nr)], &map, sizeof map);
        }
        return true;
    };
    const int H = c.hidden, qd = c.n_q_heads * c.head_dim, kd = c.n_kv_heads * c.head_dim;
    for (int l = 0; l < c.n_layers; l++) {
        const ll::LayerW &L = layers[l];
        if (mh.tc && !(one(L.wq, qd, H, mh.kc, l, 0) && one(L.wk, kd, H, mh.kc, l, 1) && one(L.wv, kd, H, mh.kc, l, 2) &&
                       one(L.wg, c.inter, H, mh.kc, l, 4) && one(L.wu, c.inter, H, mh.kc, l, 5)))
            return false;
        if (mq.tc && !one(L.wo, H, qd, mq.kc, l, 3)) return false;
        if (mi.tc && !one(L.wd, H, c.inter, mi.kc, l, 6)) return false;
    }
    if (mh.tc && !one(lm_head, c.vocab, H, mh.kc, c.n_layers, 0)) return false;
    return true;
}

int attn_splits(const ll_config &c, int nsm, int nb = 1) { return ll::attn_splits(c.max_seq, c.n_kv_heads, nsm, nb); }

void build_lists_for(const ll_config &c, int nsm, int splits, std::vector<std::vector<Instr>> &lists, int nb = 1,
                     int lm_rows = 1 << 30) {
    ll::build_schedule(c.n_layers, c.hidden, c.n_q_heads * c.head_dim, c.n_kv_heads * c.head_dim, c.inter,
                       c.vocab, c.n_kv_heads, nsm, splits, lists, nb, lm_rows);
}

// The tensor-core kernel holds at most BACC_FLOATS (row, sequence) results per
// instruction, so it takes an SM's vocabulary rows in pieces of this many rows.
// The CUDA-core kernel keeps the (row, k-slice) partial sums of an instruction,
// at most KPART_FLOATS of them, so its LM-head pieces are cut to fit as well
// (whole pages of the hidden-width geometry).
int lm_rows_cuda(const ll::MvShape &mh, int nb = 1) {
    const int rows = ll::KPART_FLOATS / std::max(1, mh.ws * nb);
    return std::max(mh.rpp, rows / std::max(1, mh.rpp) * mh.rpp);
}

int lm_rows_of(const ll_handle *h) {
    return h->kp.mv_h.tc ? std::max(ll::TC_ROWS, ll::BACC_FLOATS / h->nb / ll::TC_ROWS * ll::TC_ROWS)
                         : lm_rows_cuda(h->kp.mv_h, h->nb);
}

void build_lists(ll_handle *h) { build_lists_for(h->cfg, h->nsm, h->splits, h->lists, h->nb, lm_rows_of(h)); }

// Clear counters, tagged activation words and the status word after a failed
// step so the next starts clean (the step count restarts, so no stale tag may
// survive).
int reset_device_state(ll_handle *h) {
    const size_t nctr = size_t(ll::CtrLayout::count(h->cfg.n_layers, h->cfg.n_kv_heads)) * ll::CTR_STRIDE;
    if (cudaMemsetAsync(h->kp.ctr, 0, nctr * sizeof(uint32_t), h->stream) != cudaSuccess ||
        cudaMemsetAsync(h->tagged, 0, h->tagged_bytes, h->stream) != cudaSuccess ||
        cudaMemsetAsync(h->kp.status, 0, sizeof(int32_t), h->stream) != cudaSuccess ||
        cudaStreamSynchronize(h->stream) != cudaSuccess)
        return LL_ERR_CUDA;
    h->epoch = 0;
    return LL_OK;
}

// One launch of n_steps steps. pos_b: each sequence's first position (batched
// handles), else pos for the one sequence.
int enqueue(ll_handle *h, int32_t token, const int32_t *token_dev, int32_t pos, float *logits,
            int32_t *next_token_dev, int32_t n_steps = 1, int32_t *tokens_dev = nullptr,
            const int32_t *pos_b = nullptr) {
    if (!pos_b && h->batch_api) return fail(h, LL_ERR_ARG, "a batched handle steps through ll_decode_steps_batch");
    for (int b = 0; pos_b && b < h->nb; b++)
        if (pos_b[b] < 0 || n_steps < 1 || int64_t(pos_b[b]) + n_steps > h->cfg.max_seq)
            return fail(h, LL_ERR_ARG, "sequence " + std::to_string(b) + ": steps " + std::to_string(pos_b[b]) + ".." +
                                           std::to_string(int64_t(pos_b[b]) + n_steps - 1) + " outside [0, max_seq)");
    if (pos_b) pos = pos_b[0];
    if (pos < 0 || pos >= h->cfg.max_seq)
        return fail(h, LL_ERR_ARG, "pos " + std::to_string(pos) + " outside [0, max_seq)");
    if (n_steps < 1 || int64_t(pos) + n_steps > h->cfg.max_seq)
        return fail(h, LL_ERR_ARG, "steps " + std::to_string(pos) + ".." + std::to_string(int64_t(pos) + n_steps - 1) +
                                       " outside [0, max_seq)");
    if (logits && !aligned16(logits)) return fail(h, LL_ERR_ARG, "logits buffer not 16-byte aligned");
    KParams p = h->kp;
    p.token = token;
    p.token_dev = token_dev;
    p.pos = pos;
    p.logits = logits;
    p.next_token_dev = next_token_dev;
    p.n_steps = n_steps;
    p.tokens_dev = tokens_dev;
    for (int b = 0; b < h->nb; b++) p.pos_b[b] = pos_b ? pos_b[b] : pos;
    p.epoch = h->epoch + 1;
    h->epoch += static_cast<uint32_t>(n_steps);
    int rc;
    if (h->cfg.backend == LL_BACKEND_CHAIN) {
        // one launch sequence per step: step i reads step i - 1's token from tokens_dev
        rc = LL_OK;
        for (int32_t i = 0; i < n_steps && rc == LL_OK; i++) {
            KParams q = p;
            q.n_steps = 1;
            q.tokens_dev = nullptr;
            q.pos = pos + i;
            q.epoch = p.epoch + static_cast<uint32_t>(i);
            if (tokens_dev) {
                q.token_dev = i == 0 ? token_dev : tokens_dev + (i - 1);
                q.next_token_dev = tokens_dev + i;
            }
            if (logits) q.logits = logits + size_t(i) * size_t(h->cfg.vocab);
            rc = ll::launch_chain_step(q, h->cb, h->stream);
        }
    } else {
        rc = ll::launch_megakernel(p, h->stream, h->smem_bytes);
    }
    if (rc != LL_OK) {
        cudaError_t e = cudaGetLastError();
        return fail(h, rc, std::string("kernel launch failed: ") + cudaGetErrorString(e));
    }
    return LL_OK;
}

const char *status_text(int s) {
    switch (s) {
        case LL_ERR_ARG: return "a token out of range";
        case LL_ERR_DEP_TIMEOUT: return "a device-side wait ran past its time limit";
        case LL_ERR_NUMERIC: return "the logits held no orderable value (all NaN): no greedy token";
        default: return "device error";
    }
}

}  // namespace

namespace ll {
int attn_splits(int max_seq, int n_kv_heads, int nsm, int nb) {
    int per = ATTN_SPLIT_POS;
    if (const char *e = std::getenv("LL_ATTN_SPLIT_POS")) per = std::max(1, std::atoi(e));
    const int want = (max_seq + per - 1) / per;
    return std::max(1, std::min(want, nsm / (n_kv_heads * nb)));
}
}  // namespace ll

namespace {

// ll_init (nb = 1, one cache pair) and ll_init_batch (nb sequences, batch_api):
// one handle, one library allocation, the schedule for nb sequences.
int init_handle(const ll_config *cfg, const ll_weights *w, uint16_t *const *k_caches, uint16_t *const *v_caches,
                int nb, bool batch_api, void *stream, ll_handle **out) {
    g_init_error.clear();
    auto bad = [&](int code, const std::string &msg) {
        g_init_error = msg;
        return code;
    };
    if (!out) return bad(LL_ERR_ARG, "out is NULL");
    *out = nullptr;
    if (!cfg || !w) return bad(LL_ERR_ARG, "cfg or weights is NULL");
    const ll_config c = *cfg;
    // ---- shape checks
    if (c.n_layers < 1 || c.hidden <= 0 || c.n_q_heads <= 0 || c.n_kv_heads <= 0 || c.inter <= 0 ||
        c.vocab <= 0 || c.max_seq <= 0)
        return bad(LL_ERR_SHAPE, "every size must be positive");
    if (c.head_dim != 64 && c.head_dim != 128) return bad(LL_ERR_SHAPE, "head_dim must be 64 or 128");
    if (c.n_q_heads % c.n_kv_heads != 0 || c.n_q_heads / c.n_kv_heads > ll::MAX_GQA)
        return bad(LL_ERR_SHAPE, "n_q_heads must be a multiple (at most 8x) of n_kv_heads");
    if ((c.n_q_heads / std::max(1, c.n_kv_heads)) * c.head_dim > 512)
        return bad(LL_ERR_SHAPE, "(n_q_heads / n_kv_heads) * head_dim must be at most 512");
    if (int64_t(c.n_q_heads) * c.head_dim > ll::XIN_FLOATS)
        return bad(LL_ERR_SHAPE, "n_q_heads*head_dim must be at most 4096");
    if (c.backend != LL_BACKEND_MEGAKERNEL && c.backend != LL_BACKEND_CHAIN)
        return bad(LL_ERR_ARG, "unknown backend");
    if (!(c.rms_eps >= 0.f) || !(c.rope_theta > 0.f)) return bad(LL_ERR_ARG, "rms_eps/rope_theta invalid");
    ll::MvShape mh{}, mq{}, mi{};
    // Input floats a lane may hold per team copy of a matvec input (tuning knob
    // LL_MV_LANE_FLOATS, 16 or 32). 32 allows more teams, so more pages in
    // progress at once: measured 1B 673 -> 656 us, 3B 1715 -> 1630 us, 8B 3270 ->
    // 3225 us, 1B at 32k 891 -> 872 us (same box, back to back).
    int lane_floats = 32;
    if (const char *e = std::getenv("LL_MV_LANE_FLOATS")) lane_floats = std::atoi(e) == 16 ? 16 : 32;
    if (!ll::mv_shape(c.hidden, mh, lane_floats) || !ll::mv_shape(c.n_q_heads * c.head_dim, mq, lane_floats) ||
        !ll::mv_shape(c.inter, mi, lane_floats))
        return bad(LL_ERR_SHAPE, "hidden, n_q_heads*head_dim and inter must be multiples of 256, at most 16384");
    // ---- pointer checks
    if (nb < 1 || nb > ll::MAX_B || (nb & (nb - 1)) != 0)
        return bad(LL_ERR_ARG, "the batch must be 1, 2, 4 or 8 sequences");
    if (!k_caches || !v_caches) return bad(LL_ERR_ARG, "KV cache arrays are NULL");
    for (int b = 0; b < nb; b++)
        if (!aligned16(k_caches[b]) || !aligned16(v_caches[b])) return bad(LL_ERR_ARG, "KV caches must be 16-byte aligned");
    uint16_t *const k_cache = k_caches[0], *const v_cache = v_caches[0];
    if (batch_api && c.backend != LL_BACKEND_MEGAKERNEL) return bad(LL_ERR_ARG, "batched decode runs on the megakernel backend");
    if (!aligned16(w->embed) || !aligned16(w->final_norm)) return bad(LL_ERR_ARG, "embed/final_norm not 16-byte aligned");
    if (!c.tied && !aligned16(w->lm_head)) return bad(LL_ERR_ARG, "lm_head not 16-byte aligned");
    const uint16_t *const *lp[9] = {w->attn_norm, w->wq, w->wk, w->wv, w->wo, w->mlp_norm, w->wg, w->wu, w->wd};
    for (auto a : lp)
        if (!a) return bad(LL_ERR_ARG, "a per-layer pointer array is NULL");
    std::vector<ll::LayerW> layers(c.n_layers);
    for (int l = 0; l < c.n_layers; l++) {
        ll::LayerW &L = layers[l];
        L = {w->attn_norm[l], w->wq[l], w->wk[l], w->wv[l], w->wo[l], w->mlp_norm[l], w->wg[l], w->wu[l], w->wd[l]};
        const uint16_t *all[9] = {L.attn_norm, L.wq, L.wk, L.wv, L.wo, L.mlp_norm, L.wg, L.wu, L.wd};
        for (auto a : all)
            if (!aligned16(a)) return bad(LL_ERR_ARG, "layer " + std::to_string(l) + " weight not 16-byte aligned");
    }
    // ---- device checks
    int dev = 0;
    cudaDeviceProp prop{};
    if (cudaGetDevice(&dev) != cudaSuccess || cudaGetDeviceProperties(&prop, dev) != cudaSuccess)
        return bad(LL_ERR_CUDA, "no CUDA device");
    if (prop.major != 10 || prop.minor != 3)
        return bad(LL_ERR_DEVICE, "device is sm_" + std::to_string(prop.major) + std::to_string(prop.minor) +
                                      ", this library is built for sm_103a");
    if (!prop.cooperativeLaunch) return bad(LL_ERR_DEVICE, "device lacks cooperative launch");

    ll_handle *h = new ll_handle();
    h->cfg = c;
    h->device = dev;
    h->nsm = prop.multiProcessorCount;
    h->stream = static_cast<cudaStream_t>(stream);
    h->nb = nb;
    h->batch_api = batch_api;
    h->splits = attn_splits(c, h->nsm, nb);
    h->smem_bytes = ll::megakernel_smem_bytes();
    h->host_layers = layers;
    const int qd = c.n_q_heads * c.head_dim, kd = c.n_kv_heads * c.head_dim;
    auto per_sm = [&](int64_t rows) { return (rows + h->nsm - 1) / h->nsm; };
    const int64_t qkv_rows = int64_t(c.n_q_heads + 2 * c.n_kv_heads) * c.head_dim;
    if (per_sm(qkv_rows) > ll::ACC_FLOATS || 2 * per_sm(c.inter) > ll::ACC_FLOATS ||
        per_sm(c.hidden) > ll::XOWN_MAX || per_sm(c.vocab) > ll::ACC_FLOATS ||
        per_sm(qkv_rows) * mh.ws > ll::KPART_FLOATS || 2 * per_sm(c.inter) * mh.ws > ll::KPART_FLOATS ||
        per_sm(c.hidden) * std::max(mq.ws, mi.ws) > ll::KPART_FLOATS) {
        delete h;
        return bad(LL_ERR_SHAPE, "a projection has more rows per SM than the kernel holds");
    }
    int rc = ll::megakernel_prepare(h->smem_bytes);
    if (rc != LL_OK) {
        delete h;
        return bad(rc, "cannot keep one megakernel block resident per SM");
    }
    // The tensor-core kernel (tensor-core pages for every width) for batched
    // handles, and for single-sequence handles when LL_MV_TC = 1 (tuning knob; at
    // batch 1 the CUDA-core pages measured faster, 1B at ctx 1024: 641 against
    // 865-950 us per token). It needs every width a multiple of 1024 and the
    // weight tensor maps; a single-sequence handle without them keeps the
    // CUDA-core kernel.
    std::vector<ll::TensorMap> wmaps;
    // A batch of two whose widths have two-sequence CUDA-core geometry runs on
    // CUDA-core pages (each page read once for both sequences); LL_BATCH_CC=0
    // keeps it on tensor-core pages.
    if (batch_api && nb == 2 && c.backend == LL_BACKEND_MEGAKERNEL) {
        ll::MvShape bh{}, bq{}, bi{};
        bool cc = ll::mv_shape_bc(c.hidden, bh) && ll::mv_shape_bc(qd, bq) && ll::mv_shape_bc(c.inter, bi) &&
                  per_sm(qkv_rows) * bh.ws * nb <= ll::KPART_FLOATS &&
                  2 * per_sm(c.inter) * bh.ws * nb <= ll::KPART_FLOATS &&
                  per_sm(c.hidden) * std::max(bq.ws, bi.ws) * nb <= ll::KPART_FLOATS &&
                  per_sm(c.hidden) <= ll::XOWN_MAX;
        if (const char *e = std::getenv("LL_BATCH_CC")) cc = cc && std::atoi(e) != 0;
        if (cc) {
            mh = bh;
            mq = bq;
            mi = bi;
            h->bcc = true;
        }
    }
    if (!h->bcc) {
        bool want_tc = batch_api;
        if (const char *e = std::getenv("LL_MV_TC")) want_tc = want_tc || std::atoi(e) != 0;
        ll::MvShape th{}, tq{}, ti{};
        const bool tc_all = ll::mv_shape_tc(c.hidden, th) && ll::mv_shape_tc(qd, tq) && ll::mv_shape_tc(c.inter, ti) &&
                            c.backend == LL_BACKEND_MEGAKERNEL;
        const bool fits = per_sm(qkv_rows) * nb <= ll::BACC_FLOATS && 2 * per_sm(c.inter) * nb <= ll::BACC_FLOATS &&
                          per_sm(c.hidden) * nb <= ll::BACC_FLOATS;
        if (want_tc && tc_all && fits && encode_weight_maps(c, layers, c.tied ? w->embed : w->lm_head, th, tq, ti, wmaps)) {
            mh = th;
            mq = tq;
            mi = ti;
        } else {
            wmaps.clear();
            if (batch_api) {
                delete h;
                return bad(LL_ERR_SHAPE, tc_all && fits ? "weight tensor maps could not be encoded"
                                                       : "batched decode needs hidden, n_q_heads*head_dim and inter "
                                                         "multiples of 1024 and rows per SM x batch within the "
                                                         "kernel's accumulator");
            }
        }
    }
    h->kp.mv_h = mh;
    h->kp.mv_q = mq;
    h->kp.mv_i = mi;
    build_lists(h);
    for (auto &l : h->lists) h->max_instr = std::max<int>(h->max_instr, static_cast<int>(l.size()));
    std::vector<ll::PDesc> pdesc;
    std::vector<int32_t> pdesc_off;
    ll::build_pdesc(h->lists, layers, c.tied ? w->embed : w->lm_head, c.hidden, qd, kd, c.inter, mh, mq, mi, pdesc,
                    pdesc_off);

    // ---- library memory: one allocation carved into 256-byte aligned pieces
    const size_t nctr = size_t(ll::CtrLayout::count(c.n_layers, c.n_kv_heads)) * ll::CTR_STRIDE;
    struct Piece { void **dst; size_t bytes; };
    Instr *d_instrs = nullptr;
    int32_t *d_n_instr = nullptr;
    ll::LayerW *d_layers = nullptr;
    ll::PDesc *d_pdesc = nullptr;
    ll::TensorMap *d_wmaps = nullptr;
    ll::TensorMap *d_kvmaps = nullptr;
    int32_t *d_pdesc_off = nullptr;
    float2 *d_rope = nullptr;
    float *x = nullptr, *qkv = nullptr, *part = nullptr, *o = nullptr, *act = nullptr;
    float *hbuf = nullptr, *gate = nullptr, *up = nullptr, *logits = nullptr;
    unsigned long long *keys = nullptr;
    uint32_t *ctr = nullptr;
    int32_t *status = nullptr, *tok = nullptr;
    long long *dbg = nullptr;
    uint64_t *t_qkv = nullptr, *t_part = nullptr, *t_o = nullptr, *t_xmid = nullptr, *t_act = nullptr,
             *t_xout = nullptr, *t_token = nullptr;
    const size_t part_floats = size_t(c.n_q_heads) * h->splits * (c.head_dim + 4);
    const size_t B = size_t(nb);
    Piece pieces[] = {
        {reinterpret_cast<void **>(&d_instrs), size_t(h->nsm) * h->max_instr * sizeof(Instr)},
        {reinterpret_cast<void **>(&d_n_instr), size_t(h->nsm) * sizeof(int32_t)},
        {reinterpret_cast<void **>(&d_layers), size_t(c.n_layers) * sizeof(ll::LayerW)},
        {reinterpret_cast<void **>(&d_pdesc), pdesc.size() * sizeof(ll::PDesc)},
        {reinterpret_cast<void **>(&d_wmaps), wmaps.size() * sizeof(ll::TensorMap)},
        {reinterpret_cast<void **>(&d_kvmaps), size_t(nb) * ll::TM_COUNT * sizeof(ll::TensorMap)},
        {reinterpret_cast<void **>(&d_pdesc_off), pdesc_off.size() * sizeof(int32_t)},
        {reinterpret_cast<void **>(&d_rope), size_t(c.max_seq) * (c.head_dim / 2) * sizeof(float2)},
        {reinterpret_cast<void **>(&x), size_t(c.hidden) * 4},
        {reinterpret_cast<void **>(&qkv), size_t(qd + 2 * kd) * 4},
        {reinterpret_cast<void **>(&part), part_floats * 4},
        {reinterpret_cast<void **>(&o), size_t(qd) * 4},
        {reinterpret_cast<void **>(&act), size_t(c.inter) * 4},
        {reinterpret_cast<void **>(&hbuf), size_t(c.hidden) * 4},
        {reinterpret_cast<void **>(&gate), size_t(c.inter) * 4},
        {reinterpret_cast<void **>(&up), size_t(c.inter) * 4},
        {reinterpret_cast<void **>(&logits), size_t(c.vocab) * 4},
        {reinterpret_cast<void **>(&keys), size_t(h->nsm) * 8 * B},
        {reinterpret_cast<void **>(&ctr), nctr * 4},
        // the next tokens and the status word side by side: one copy reads them all
        {reinterpret_cast<void **>(&tok), (B + 1) * 4},
        {reinterpret_cast<void **>(&dbg), 64},
        // the megakernel's tagged activations (one contiguous run, cleared together)
        {reinterpret_cast<void **>(&t_qkv), size_t(qd + 2 * kd) * 8 * B},
        {reinterpret_cast<void **>(&t_part), part_floats * 8 * B},
        {reinterpret_cast<void **>(&t_o), size_t(qd) * 8 * B},
        {reinterpret_cast<void **>(&t_xmid), size_t(c.hidden) * 8 * B},
        {reinterpret_cast<void **>(&t_act), size_t(c.inter) * 8 * B},
        {reinterpret_cast<void **>(&t_xout), size_t(c.hidden) * 8 * B},
        {reinterpret_cast<void **>(&t_token), 8 * B},
    };
    size_t total = 0;
    for (auto &pc : pieces) total += round_up(pc.bytes, 256);
    if (cudaMalloc(&h->dmem, total) != cudaSuccess) {
        cudaGetLastError();
        delete h;
        return bad(LL_ERR_OOM, "cudaMalloc of " + std::to_string(total) + " bytes failed");
    }
    h->dmem_bytes = total;
    size_t off = 0;
    for (auto &pc : pieces) {
        *pc.dst = h->dmem + off;
        off += round_up(pc.bytes, 256);
    }
    if (cudaMallocHost(&h->pinned, (B + 1) * sizeof(int32_t)) != cudaSuccess) {
        cudaFree(h->dmem);
        delete h;
        return bad(LL_ERR_OOM, "pinned host buffer allocation failed");
    }

    // RoPE table: angle pos * theta^(-2i/hd) taken in double, stored as float (cos, sin).
    const int half = c.head_dim / 2;
    std::vector<float2> rope(size_t(c.max_seq) * half);
    for (int i = 0; i < half; i++) {
        const double inv = std::pow(static_cast<double>(c.rope_theta), -2.0 * i / c.head_dim);
        for (int pos = 0; pos < c.max_seq; pos++) {
            const double a = pos * inv;
            rope[size_t(pos) * half + i] = make_float2(static_cast<float>(std::cos(a)), static_cast<float>(std::sin(a)));
        }
    }

    KParams &p = h->kp;
    p.instrs = d_instrs;
    p.n_instr = d_n_instr;
    p.pdesc = d_pdesc;
    p.pdesc_off = d_pdesc_off;
    p.max_instr = h->max_instr;
    p.nsm = h->nsm;
    p.layers = d_layers;
    p.embed = w->embed;
    p.lm_head = c.tied ? w->embed : w->lm_head;
    p.final_norm = w->final_norm;
    p.k_cache = k_cache;
    p.v_cache = v_cache;
    p.rope_cs = d_rope;
    p.L = c.n_layers;
    p.H = c.hidden;
    p.nq = c.n_q_heads;
    p.nkv = c.n_kv_heads;
    p.hd = c.head_dim;
    p.I = c.inter;
    p.V = c.vocab;
    p.max_seq = c.max_seq;
    p.eps = c.rms_eps;
    p.attn_splits = h->splits;
    {
        // kernel variant: per-warp (flash) softmax on tensor cores when the longest
        // attention item at max_seq spans at least 4 pages. Its merge of the warps
        // costs ~1.5 us per item, so on items of one or two pages the block-wide
        // pass is faster (measured: 1B at 1k context, 1-page items: 656 against
        // 683 us; 3B at 2k, 2-page items: 1631 against 1652 us; 8B at 8k, 7-page
        // items: 3224 against 3433 us; 1B at 32k, 14-page items: 869 against
        // 1148 us). Tuning knob LL_ATTN_FLASH = 0 / 1 overrides.
        const int per_split = (c.max_seq + h->splits - 1) / h->splits;
        const int pp = ll::PAGE_BYTES / (4 * c.head_dim);
        p.attn_flash = (per_split + pp - 1) / pp >= 4 ? 1 : 0;
        if (const char *e = std::getenv("LL_ATTN_FLASH")) p.attn_flash = std::atoi(e) ? 1 : 0;
        // its KV pages come through TMA tensor maps (each sequence's, for the
        // tensor-core kernel, in library memory); without them, the block variant
        if (!encode_kv_maps(c, k_cache, v_cache, p.kv_maps)) p.attn_flash = 0;
        std::vector<ll::TensorMap> kvm(size_t(nb) * ll::TM_COUNT);
        for (int b = 0; b < nb && p.attn_flash; b++) {
            ll::TensorMap one[ll::TM_COUNT];
            if (!encode_kv_maps(c, k_caches[b], v_caches[b], one)) p.attn_flash = 0;
            for (int i = 0; i < ll::TM_COUNT; i++) kvm[size_t(b) * ll::TM_COUNT + i] = one[i];
        }
        if (p.attn_flash &&
            cudaMemcpy(d_kvmaps, kvm.data(), kvm.size() * sizeof(ll::TensorMap), cudaMemcpyHostToDevice) != cudaSuccess) {
            ll_free(h);
            return bad(LL_ERR_CUDA, "KV tensor map upload failed");
        }
        p.kvmaps_b = d_kvmaps;
    }
    p.mv_h = mh;
    p.mv_q = mq;
    p.mv_i = mi;
    p.wmaps = wmaps.empty() ? nullptr : d_wmaps;
    p.nb = nb;
    for (int b = 0; b < ll::MAX_B; b++) {
        p.kc_b[b] = b < nb ? k_caches[b] : nullptr;
        p.vc_b[b] = b < nb ? v_caches[b] : nullptr;
        p.pos_b[b] = 0;
    }
    p.t_qkv = t_qkv;
    p.t_part = t_part;
    p.t_o = t_o;
    p.t_xmid = t_xmid;
    p.t_act = t_act;
    p.t_xout = t_xout;
    h->tagged = reinterpret_cast<uint8_t *>(t_qkv);
    p.t_token = t_token;
    h->tagged_bytes = static_cast<size_t>(reinterpret_cast<uint8_t *>(t_token) + round_up(8 * B, 256) -
                                          reinterpret_cast<uint8_t *>(t_qkv));
    p.lm_keys = keys;
    p.ctr = ctr;
    status = tok + nb;
    p.status = status;
    p.token_out = tok;
#ifdef LL_DEBUG_CHECKS
    p.dbg = dbg;
#endif
    p.timeout_ns = 1000000000ull;
    // tuning knobs (environment, read once here): L2 prefetch distance in pages and
    // the evict-first hint on weight pages
    p.l2_prefetch = 0;  // prefetching into L2 measured no gain, and a slowdown when issued in bursts
    p.evict_first = 1;
    if (const char *e = std::getenv("LL_L2_PREFETCH_PAGES")) p.l2_prefetch = static_cast<uint32_t>(std::atoi(e));
    if (const char *e = std::getenv("LL_EVICT_FIRST")) p.evict_first = static_cast<uint32_t>(std::atoi(e));
    p.max_inflight = ll::NPAGES;
    if (const char *e = std::getenv("LL_MAX_INFLIGHT")) p.max_inflight = static_cast<uint32_t>(std::atoi(e));
    p.producer_sleep_ns = 64;
    if (const char *e = std::getenv("LL_PRODUCER_SLEEP_NS")) p.producer_sleep_ns = static_cast<uint32_t>(std::atoi(e));
    // the kernel instantiation with only this model's matrix-vector geometries,
    // where one covers all three input widths (LL_GEO=0 forces the general one)
    {
        auto is = [](const ll::MvShape &m, int v, int r) { return !m.tc && m.vpl == v && m.rw == r; };
        auto fam = [&](const ll::MvShape &m, int geo) {
            return geo == ll::GEO_2048 ? (is(m, 2, 8) || is(m, 4, 2)) : (is(m, 4, 4) || is(m, 4, 1));
        };
        p.geo = ll::GEO_ALL;
        for (int geo : {ll::GEO_2048, ll::GEO_4096})
            if (fam(p.mv_h, geo) && fam(p.mv_q, geo) && fam(p.mv_i, geo)) p.geo = geo;
        if (const char *e = std::getenv("LL_GEO"))
            if (std::atoi(e) == 0) p.geo = ll::GEO_ALL;
        if (h->bcc) p.geo = ll::GEO_BCC;
    }
    p.consumer_sleep_ns = 0;
    if (const char *e = std::getenv("LL_CONSUMER_SLEEP_NS")) p.consumer_sleep_ns = static_cast<uint32_t>(std::atoi(e));
    h->d_instrs = d_instrs;

    ll::ChainBufs &cb = h->cb;
    cb.host_layers = h->host_layers.data();
    cb.x = x;
    cb.h = hbuf;
    cb.qkv = qkv;
    cb.part = part;
    cb.o = o;
    cb.gate = gate;
    cb.up = up;
    cb.act = act;
    cb.logits = logits;
    cb.splits = h->splits;
    cb.rope_row = nullptr;

    bool ok = cudaMemcpy(d_layers, layers.data(), layers.size() * sizeof(ll::LayerW), cudaMemcpyHostToDevice) ==
                  cudaSuccess &&
              cudaMemcpy(d_pdesc, pdesc.data(), pdesc.size() * sizeof(ll::PDesc), cudaMemcpyHostToDevice) ==
                  cudaSuccess &&
              (wmaps.empty() || cudaMemcpy(d_wmaps, wmaps.data(), wmaps.size() * sizeof(ll::TensorMap),
                                           cudaMemcpyHostToDevice) == cudaSuccess) &&
              cudaMemcpy(d_pdesc_off, pdesc_off.data(), pdesc_off.size() * sizeof(int32_t), cudaMemcpyHostToDevice) ==
                  cudaSuccess &&
              cudaMemcpy(d_rope, rope.data(), rope.size() * sizeof(float2), cudaMemcpyHostToDevice) == cudaSuccess &&
              cudaMemset(ctr, 0, nctr * 4) == cudaSuccess && cudaMemset(tok, 0, (B + 1) * 4) == cudaSuccess &&
              cudaMemset(dbg, 0, 64) == cudaSuccess &&
              cudaMemset(h->tagged, 0, h->tagged_bytes) == cudaSuccess;
    if (!ok || upload_schedule(h) != LL_OK) {
        ll_free(h);
        return bad(LL_ERR_CUDA, "initial upload failed");
    }
    *out = h;
    return LL_OK;
}

}  // namespace

extern "C" {

const char *ll_init_error(void) { return g_init_error.c_str(); }

int ll_init(const ll_config *cfg, const ll_weights *w, uint16_t *k_cache, uint16_t *v_cache, void *stream,
            ll_handle **out) {
    return init_handle(cfg, w, &k_cache, &v_cache, 1, false, stream, out);
}

int ll_init_batch(const ll_config *cfg, const ll_weights *w, uint16_t *const *k_caches, uint16_t *const *v_caches,
                  int32_t n_seq, void *stream, ll_handle **out) {
    return init_handle(cfg, w, k_caches, v_caches, n_seq, true, stream, out);
}

#ifdef LL_DEBUG_CHECKS
static void report_debug(ll_handle *h) {
    long long rec[8] = {0};
    if (h->kp.dbg && cudaMemcpy(rec, h->kp.dbg, sizeof rec, cudaMemcpyDeviceToHost) == cudaSuccess && rec[0])
        std::fprintf(stderr, "LL_DEBUG_CHECKS: code %lld sm %lld thread %lld index %lld limit %lld\n", rec[1], rec[2],
                     rec[3], rec[4], rec[5]);
}
#else
static void report_debug(ll_handle *) {}
#endif

int ll_decode_step(ll_handle *h, int32_t token, int32_t pos, float *logits_dev, int32_t *next_token_host) {
    if (!h) return LL_ERR_ARG;
    if (token < 0 || token >= h->cfg.vocab) return fail(h, LL_ERR_ARG, "token " + std::to_string(token) + " outside [0, vocab)");
    int rc = enqueue(h, token, nullptr, pos, logits_dev, nullptr);
    if (rc != LL_OK) return rc;
    if (cudaMemcpyAsync(h->pinned, h->kp.token_out, 8, cudaMemcpyDeviceToHost, h->stream) != cudaSuccess ||
        cudaStreamSynchronize(h->stream) != cudaSuccess) {
        cudaError_t e = cudaGetLastError();
        return fail(h, LL_ERR_CUDA, std::string("step failed: ") + cudaGetErrorString(e));
    }
    report_debug(h);
    const int32_t st = h->pinned[1];
    if (st != 0) {
        reset_device_state(h);
        return fail(h, st, status_text(st));
    }
    if (next_token_host) *next_token_host = h->pinned[0];
    return LL_OK;
}

int ll_decode_steps(ll_handle *h, const int32_t *token_dev, int32_t pos, int32_t n_steps, float *logits_dev,
                    int32_t *tokens_dev) {
    if (!h) return LL_ERR_ARG;
    if (!token_dev || !tokens_dev) return fail(h, LL_ERR_ARG, "token_dev or tokens_dev is NULL");
    return enqueue(h, 0, token_dev, pos, logits_dev, nullptr, n_steps, tokens_dev);
}

int ll_prefill(ll_handle *h, const int32_t *tokens_dev, int32_t n, int32_t pos0, float *logits_dev,
               int32_t *next_token_dev) {
    if (!h) return LL_ERR_ARG;
    if (h->batch_api) return fail(h, LL_ERR_ARG, "prefill takes a single-sequence handle");
    if (!tokens_dev || !next_token_dev) return fail(h, LL_ERR_ARG, "tokens_dev or next_token_dev is NULL");
    if (n < 1 || pos0 < 0 || int64_t(pos0) + n > h->cfg.max_seq)
        return fail(h, LL_ERR_ARG, "positions " + std::to_string(pos0) + ".." + std::to_string(int64_t(pos0) + n - 1) +
                                       " outside [0, max_seq)");
    if (logits_dev && !aligned16(logits_dev)) return fail(h, LL_ERR_ARG, "logits buffer not 16-byte aligned");
    if (h->cfg.hidden % 64 || (h->cfg.n_q_heads * h->cfg.head_dim) % 64 || h->cfg.inter % 64)
        return fail(h, LL_ERR_SHAPE, "prefill needs hidden, n_q_heads*head_dim and inter multiples of 64");
    if (!ll::prefill_prepare(h->kp, h->host_layers.data(), n, h->pf))
        return fail(h, LL_ERR_OOM, "prefill buffers for " + std::to_string(n) + " positions could not be made");
    const int rc = ll::launch_prefill(h->kp, h->host_layers.data(), h->pf, tokens_dev, n, pos0, logits_dev,
                                      next_token_dev, h->stream);
    if (rc != LL_OK) {
        cudaError_t e = cudaGetLastError();
        return fail(h, rc, std::string("prefill launch failed: ") + cudaGetErrorString(e));
    }
    return LL_OK;
}

int ll_decode_steps_batch(ll_handle *h, const int32_t *tokens_in_dev, const int32_t *pos_host, int32_t n_steps,
                          float *logits_dev, int32_t *tokens_dev) {
    if (!h) return LL_ERR_ARG;
    if (!h->batch_api) return fail(h, LL_ERR_ARG, "not a batched handle (ll_init_batch makes one)");
    if (!tokens_in_dev || !pos_host || !tokens_dev) return fail(h, LL_ERR_ARG, "tokens_in_dev, pos or tokens_dev is NULL");
    return enqueue(h, 0, tokens_in_dev, 0, logits_dev, nullptr, n_steps, tokens_dev, pos_host);
}

int ll_decode_step_async(ll_handle *h, const int32_t *token_dev, int32_t pos, float *logits_dev,
                         int32_t *next_token_dev) {
    if (!h) return LL_ERR_ARG;
    if (!token_dev) return fail(h, LL_ERR_ARG, "token_dev is NULL");
    return enqueue(h, 0, token_dev, pos, logits_dev, next_token_dev);
}

int ll_synchronize(ll_handle *h) {
    if (!h) return LL_ERR_ARG;
    if (cudaMemcpyAsync(h->pinned + 1, h->kp.status, 4, cudaMemcpyDeviceToHost, h->stream) != cudaSuccess ||
        cudaStreamSynchronize(h->stream) != cudaSuccess) {
        cudaError_t e = cudaGetLastError();
        return fail(h, LL_ERR_CUDA, std::string("synchronize failed: ") + cudaGetErrorString(e));
    }
    report_debug(h);
    const int32_t st = h->pinned[1];
    if (st != 0) {
        reset_device_state(h);
        return fail(h, st, status_text(st));
    }
    return LL_OK;
}

int ll_set_trace(ll_handle *h, uint64_t *trace_dev, size_t bytes) {
    if (!h) return LL_ERR_ARG;
    if (!trace_dev) {
        h->kp.trace = nullptr;
        h->kp.ptrace = nullptr;
        return LL_OK;
    }
    const size_t instr_words = size_t(h->nsm) * h->max_instr * ll::TRACE_WORDS;
    const size_t page_words = size_t(h->nsm) * ll::PTRACE_PAGES * 3;
    const size_t need = (instr_words + page_words) * sizeof(uint64_t);
    if (bytes < need || !aligned16(trace_dev))
        return fail(h, LL_ERR_ARG, "trace buffer needs " + std::to_string(need) + " bytes, 16-byte aligned");
    h->kp.trace = reinterpret_cast<unsigned long long *>(trace_dev);
    h->kp.ptrace = h->kp.trace + instr_words;
    return LL_OK;
}

int ll_set_timeout_ns(ll_handle *h, uint64_t ns) {
    if (!h || ns == 0) return LL_ERR_ARG;
    h->kp.timeout_ns = ns;
    return LL_OK;
}

int ll_query(const ll_handle *h, int what, int64_t *value) {
    if (!h || !value) return LL_ERR_ARG;
    switch (what) {
        case LL_Q_NUM_SMS: *value = h->nsm; break;
        case LL_Q_ATTN_SPLITS: *value = h->splits; break;
        case LL_Q_PAGE_BYTES: *value = ll::PAGE_BYTES; break;
        case LL_Q_NUM_PAGES: *value = ll::NPAGES; break;
        case LL_Q_SCRATCH_BYTES: *value = static_cast<int64_t>(h->dmem_bytes); break;
        case LL_Q_MAX_INSTRS: *value = h->max_instr; break;
        case LL_Q_LAUNCHES_PER_STEP:
            *value = h->cfg.backend == LL_BACKEND_CHAIN ? 1 + 13 * int64_t(h->cfg.n_layers) + 3 : 1;
            break;
        case LL_Q_SMEM_BYTES: *value = h->smem_bytes; break;
        case LL_Q_MV_TC: *value = (h->kp.mv_h.tc ? 1 : 0) | (h->kp.mv_q.tc ? 2 : 0) | (h->kp.mv_i.tc ? 4 : 0); break;
        case LL_Q_BATCH: *value = h->nb; break;
        case LL_Q_BATCH_CC: *value = h->bcc ? 1 : 0; break;
        case LL_Q_TRACE_BYTES:
            *value = (int64_t(h->nsm) * h->max_instr * ll::TRACE_WORDS + int64_t(h->nsm) * ll::PTRACE_PAGES * 3) *
                     int64_t(sizeof(uint64_t));
            break;
        default: return LL_ERR_ARG;
    }
    return LL_OK;
}

int ll_debug_inject(ll_handle *h, int kind, int layer, int op) {
    if (!h) return LL_ERR_ARG;
    if (cudaStreamSynchronize(h->stream) != cudaSuccess) return fail(h, LL_ERR_CUDA, "synchronize failed");
    build_lists(h);
    if (kind == LL_FAULT_DROP_SIGNAL) {
        if (layer < 0 || layer >= h->cfg.n_layers || op < ll::OP_QKV || op > ll::OP_DOWN)
            return fail(h, LL_ERR_ARG, "fault target out of range");
        for (auto &list : h->lists)
            for (auto &in : list)
                if (in.layer == layer && in.op == op) in.sig_ctr = -1;
    } else if (kind != LL_FAULT_NONE) {
        return fail(h, LL_ERR_ARG, "unknown fault kind");
    }
    return upload_schedule(h);
}

}  // extern "C"

namespace {
// Per-SM instruction lists as [nsm][max_instr][7] int32 records (op, layer, r0,
// r1, wait_ctr, wait_count, sig_ctr; op -1 past a list's end).
int dump_lists(const std::vector<std::vector<Instr>> &lists, int32_t *out, size_t out_len, int32_t *max_instr) {
    size_t mx = 0;
    for (auto &l : lists) mx = std::max(mx, l.size());
    if (max_instr) *max_instr = static_cast<int32_t>(mx);
    if (!out) return LL_OK;
    const size_t nsm = lists.size();
    if (out_len < nsm * mx * 7) return LL_ERR_ARG;
    for (size_t sm = 0; sm < nsm; sm++) {
        for (size_t i = 0; i < mx; i++) {
            int32_t *o = out + (sm * mx + i) * 7;
            if (i < lists[sm].size()) {
                const Instr &in = lists[sm][i];
                o[0] = in.op; o[1] = in.layer; o[2] = in.r0; o[3] = in.r1;
                o[4] = in.wait_ctr; o[5] = static_cast<int32_t>(in.wait_count); o[6] = in.sig_ctr;
            } else {
                o[0] = -1; o[1] = o[2] = o[3] = o[5] = 0; o[4] = o[6] = -1;
            }
        }
    }
    return LL_OK;
}
}  // namespace

extern "C" {

int ll_plan(const ll_config *cfg, int32_t nsm, int32_t *out, size_t out_len, int32_t *max_instr) {
    if (!cfg || nsm <= 0 || cfg->n_layers < 1 || cfg->n_kv_heads <= 0 || cfg->n_q_heads % cfg->n_kv_heads != 0)
        return LL_ERR_ARG;
    std::vector<std::vector<Instr>> lists;
    ll::MvShape mh{};
    if (!ll::mv_shape(cfg->hidden, mh, 32)) return LL_ERR_SHAPE;
    build_lists_for(*cfg, nsm, attn_splits(*cfg, nsm), lists, 1, lm_rows_cuda(mh));
    return dump_lists(lists, out, out_len, max_instr);
}

int ll_handle_plan(const ll_handle *h, int32_t *out, size_t out_len, int32_t *max_instr) {
    if (!h) return LL_ERR_ARG;
    return dump_lists(h->lists, out, out_len, max_instr);
}

const char *ll_last_error(const ll_handle *h) { return h ? h->err.c_str() : "null handle"; }

void ll_free(ll_handle *h) {
    if (!h) return;
    cudaStreamSynchronize(h->stream);
    if (h->dmem) cudaFree(h->dmem);
    if (h->pinned) cudaFreeHost(h->pinned);
    ll::prefill_release(h->pf);
    delete h;
}

}  // extern "C"
