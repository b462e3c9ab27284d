// schedule.cpp -- host-side builder of the per-SM instruction lists.
//
// The page "Hazy Research Llama-3.2-1B Megakernel" (paragraphs on the
// instruction interpreter and the counter system) has the host lay out, before
// the kernel runs, an ordered instruction list for every SM together with the
// dependencies between instructions, and reuses that plan for every token.
// Here every matrix-vector product is cut into one contiguous row range per SM,
// attention into (KV head, KV split) items, and every instruction names the one
// counter it waits on and the one it bumps.
#include <algorithm>
#include <cstdint>
#include <vector>

#include "ll_internal.h"

namespace ll {

namespace {

// Rows [R*i/n, R*(i+1)/n): contiguous, sizes differ by at most one.
inline void split_rows(int64_t R, int n, int i, int32_t &r0, int32_t &r1) {
    r0 = static_cast<int32_t>(R * i / n);
    r1 = static_cast<int32_t>(R * (i + 1) / n);
}

Instr make(Op op, int layer, int32_t r0, int32_t r1, int wait_ctr, uint32_t wait_count, int sig_ctr) {
    Instr in{};
    in.op = op;
    in.layer = static_cast<uint16_t>(layer);
    in.r0 = r0;
    in.r1 = r1;
    in.wait_ctr = wait_ctr;
    in.wait_count = wait_count;
    in.sig_ctr = sig_ctr;
    return in;
}

}  // namespace

// Fills `lists[sm]` for every SM. Within one SM the list is ordered by layer and
// by the order of the page's instruction list, so every wait refers to work that
// some SM schedules earlier; with all blocks resident at once this cannot deadlock.
void build_schedule(int L, int H, int qd, int kd, int I, int V, int nkv, int nsm, int splits,
                    std::vector<std::vector<Instr>> &lists, int nb, int lm_rows) {
    lists.assign(nsm, {});
    const uint32_t all = static_cast<uint32_t>(nsm);
    for (int l = 0; l < L; l++) {
        for (int sm = 0; sm < nsm; sm++) {
            int32_t r0, r1;
            split_rows(qd + 2 * kd, nsm, sm, r0, r1);
            lists[sm].push_back(make(OP_QKV, l, r0, r1, l ? CtrLayout::down(l - 1) : -1, l ? all : 0,
                                     CtrLayout::qkv(l)));
            if (sm < nb * nkv * splits) {
                const int item = sm % (nkv * splits);
                Instr a = make(OP_ATTN, l, item / splits, item % splits, CtrLayout::qkv(l), all, CtrLayout::attn(l));
                a.sub = static_cast<uint8_t>(sm / (nkv * splits));
                lists[sm].push_back(a);
            }
            split_rows(H, nsm, sm, r0, r1);
            lists[sm].push_back(make(OP_OPROJ, l, r0, r1, CtrLayout::attn(l),
                                     static_cast<uint32_t>(nb * nkv * splits), CtrLayout::oproj(l)));
            split_rows(I, nsm, sm, r0, r1);
            lists[sm].push_back(make(OP_GATEUP, l, r0, r1, CtrLayout::oproj(l), all, CtrLayout::gateup(l)));
            split_rows(H, nsm, sm, r0, r1);
            lists[sm].push_back(make(OP_DOWN, l, r0, r1, CtrLayout::gateup(l), all, CtrLayout::down(l)));
        }
    }
    for (int sm = 0; sm < nsm; sm++) {
        int32_t r0, r1;
        split_rows(V, nsm, sm, r0, r1);
        // (an SM with no vocabulary rows still gets one, empty, instruction)
        for (int32_t a = r0;;) {
            const int32_t e = std::min<int64_t>(r1, int64_t(a) + lm_rows);
            Instr in = make(OP_LMHEAD, 0, a, e, CtrLayout::down(L - 1), all, -1);
            in.sub = e >= r1 ? 1 : 0;
            lists[sm].push_back(in);
            if (e >= r1) break;
            a = e;
        }
    }
}

// Input-vector geometry for width K (see MvShape). Teams: as many as keep each
// lane's share of the input at or under 32 floats (a team holds a full copy of
// the input). Within a team: among the splits of a row into k-slices of
// 256*vpl elements (vpl <= 4), the one that keeps the most warps busy, then the
// most rows per page (rows per warp a power of two, at most 8). Returns false
// if K admits none.
// (vpl, rw) pairs the megakernel is compiled for.
static bool mv_combo_ok(int vpl, int rw) {
    static const int ok[][2] = {{1, 8}, {2, 8}, {3, 1}, {3, 2}, {3, 4}, {4, 1}, {4, 2}, {4, 4}};
    for (auto &c : ok)
        if (c[0] == vpl && c[1] == rw) return true;
    return false;
}

bool mv_shape_tc(int K, MvShape &m) {
    if (K <= 0 || K % 1024 != 0 || K > 16384) return false;
    const int kc = K % 2048 == 0 ? 2048 : 1024;
    m = MvShape{K, NCW, 0, TC_ROWS, 1, TC_ROWS, 1, 1, kc, K / kc, {}, {}, {}, {}};
    return true;
}

static bool mv_shape_with(int K, MvShape &m, int lane_floats, int max_vpl, bool (*combo_ok)(int, int));

bool mv_shape(int K, MvShape &m, int lane_floats) { return mv_shape_with(K, m, lane_floats, MAX_VPL, mv_combo_ok); }

// (vpl, rw) pairs the two-sequence CUDA-core kernel is compiled for.
static bool bc_combo_ok(int vpl, int rw) { return vpl == 2 && (rw == 8 || rw == 2); }

bool mv_shape_bc(int K, MvShape &m) { return mv_shape_with(K, m, 16, 2, bc_combo_ok); }

static bool mv_shape_with(int K, MvShape &m, int lane_floats, int max_vpl, bool (*combo_ok)(int, int)) {
    if (K <= 0 || K % 256 != 0 || K > 16384) return false;
    const int rows_fit = PAGE_BYTES / (2 * K);
    if (rows_fit < 1) return false;
    int teams = 1;
    while (teams < 4 && K * teams * 2 <= lane_floats * 32 * NCW) teams *= 2;
    const int W = NCW / teams;
    int best_active = 0, best_rpp = 0;
    for (int vpl = 1; vpl <= max_vpl; vpl++) {
        if (K % (256 * vpl) != 0) continue;
        const int ws = K / (256 * vpl);
        if (ws > W) continue;
        const int rg = std::min(W / ws, rows_fit);
        if (rg < 1) continue;
        int rw = 1;
        while (rw * 2 * rg <= rows_fit && rw * 2 <= 8) rw *= 2;
        const int rpp = rg * rw;
        if (rpp > MAX_RPP || rpp * ws > MAX_PART || !combo_ok(vpl, rw)) continue;
        const int active = ws * rg;
        if (active > best_active || (active == best_active && rpp > best_rpp)) {
            best_active = active;
            best_rpp = rpp;
            m = MvShape{K, ws, vpl, rpp, rg, rw, teams, 0, K, 1, {}, {}, {}, {}};
        }
    }
    if (best_active == 0) return false;
    // warp roles: warps [team * W, team * W + W) form a team; within it warp wt
    // takes k-slice wt % ws of row group wt / ws, and the ws * rg working warps
    // release a page with NCW arrivals in all (warp 0 of the team takes the rest)
    const int active = m.ws * m.rg;
    for (int w = 0; w < NCW; w++) {
        const int wt = w % W;
        m.w_team[w] = static_cast<uint8_t>(w / W);
        m.w_sw[w] = static_cast<uint8_t>(wt % m.ws);
        m.w_rgi[w] = static_cast<uint8_t>(wt / m.ws);
        m.w_arrive[w] = static_cast<uint8_t>(wt >= active ? 0 : wt == 0 ? NCW - (active - 1) * (NCW / active)
                                                                        : NCW / active);
    }
    return true;
}

// The producer lists: for every SM, the pages its consumers will take, in the
// order they take them (the same segment and row-page walk as the consumers).
void build_pdesc(const std::vector<std::vector<Instr>> &lists, const std::vector<LayerW> &layers,
                 const uint16_t *lm_head, int H, int qd, int kd, int I, const MvShape &mh, const MvShape &mq,
                 const MvShape &mi, std::vector<PDesc> &out, std::vector<int32_t> &off) {
    out.clear();
    off.assign(lists.size() + 1, 0);
    // pages of a segment: rows [row0, row0 + nrows) of matrix w; tensor-core
    // pages name the matrix's tensor map (layer l, matrix m) and column chunk
    // instead of an address, chunk after chunk (the consumers build the input's
    // fragments once per chunk)
    auto pages = [&](const uint16_t *w, int row0, int nrows, const MvShape &mv, int instr, int l, int m) {
        for (int c = 0; c < (mv.tc ? mv.nch : 1); c++) {
            for (int pr = 0; pr < nrows; pr += mv.rpp) {
                const int nr = std::min(mv.rpp, nrows - pr);
                PDesc d{};
                if (mv.tc) {
                    d.src = (static_cast<unsigned long long>(wmap_index(l, m, nr)) << 40) |
                            (static_cast<unsigned long long>(c * (mv.kc / 64)) << 32) | uint32_t(row0 + pr);
                    d.kind = PD_TMA_W;
                    d.bytes = uint32_t(nr) * uint32_t(mv.kc) * 2u;
                } else {
                    d.src = reinterpret_cast<unsigned long long>(w + size_t(row0 + pr) * mv.K);
                    d.kind = PD_WEIGHTS;
                    d.bytes = uint32_t(nr) * uint32_t(mv.K) * 2u;
                }
                d.instr = static_cast<uint16_t>(instr);
                out.push_back(d);
            }
        }
    };
    for (size_t sm = 0; sm < lists.size(); sm++) {
        off[sm] = static_cast<int32_t>(out.size());
        for (size_t i = 0; i < lists[sm].size(); i++) {
            const Instr &in = lists[sm][i];
            const int r0 = in.r0, r1 = in.r1;
            if (in.op == OP_ATTN) {
                PDesc d{};
                d.src = (static_cast<unsigned long long>(in.sub) << 48) | (static_cast<unsigned long long>(in.layer) << 32) |
                        (static_cast<unsigned long long>(r0) << 16) | static_cast<unsigned long long>(r1);
                d.instr = static_cast<uint16_t>(i);
                d.kind = PD_ATTN;
                out.push_back(d);
                continue;
            }
            if (r0 >= r1) continue;
            const LayerW *lw = in.op == OP_LMHEAD ? nullptr : &layers[in.layer];
            switch (in.op) {
                case OP_QKV: {
                    const int b[4] = {0, qd, qd + kd, qd + 2 * kd};
                    const uint16_t *m[3] = {lw->wq, lw->wk, lw->wv};
                    for (int k = 0; k < 3; k++) {
                        const int a = std::max(r0, b[k]), e = std::min(r1, b[k + 1]);
                        if (a < e) pages(m[k], a - b[k], e - a, mh, int(i), in.layer, k);
                    }
                    break;
                }
                case OP_OPROJ: pages(lw->wo, r0, r1 - r0, mq, int(i), in.layer, 3); break;
                case OP_GATEUP:
                    pages(lw->wg, r0, r1 - r0, mh, int(i), in.layer, 4);
                    pages(lw->wu, r0, r1 - r0, mh, int(i), in.layer, 5);
                    break;
                case OP_DOWN: pages(lw->wd, r0, r1 - r0, mi, int(i), in.layer, 6); break;
                default: pages(lm_head, r0, r1 - r0, mh, int(i), int(layers.size()), 0); break;
            }
        }
    }
    off[lists.size()] = static_cast<int32_t>(out.size());
    (void)H;
    (void)I;
}

}  // namespace ll
