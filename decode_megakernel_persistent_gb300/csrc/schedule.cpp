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
                    std::vector<std::vector<Instr>> &lists) {
    lists.assign(nsm, {});
    const uint32_t all = static_cast<uint32_t>(nsm);
    for (int l = 0; l < L; l++) {
        for (int sm = 0; sm < nsm; sm++) {
            int32_t r0, r1;
            split_rows(qd + 2 * kd, nsm, sm, r0, r1);
            lists[sm].push_back(make(OP_QKV, l, r0, r1, l ? CtrLayout::down(l - 1) : -1, l ? all : 0,
                                     CtrLayout::qkv(l)));
            if (sm < nkv * splits)
                lists[sm].push_back(make(OP_ATTN, l, sm / splits, sm % splits, CtrLayout::qkv(l), all,
                                         CtrLayout::attn(l)));
            split_rows(H, nsm, sm, r0, r1);
            lists[sm].push_back(make(OP_OPROJ, l, r0, r1, CtrLayout::attn(l), static_cast<uint32_t>(nkv * splits),
                                     CtrLayout::oproj(l)));
            split_rows(I, nsm, sm, r0, r1);
            lists[sm].push_back(make(OP_GATEUP, l, r0, r1, CtrLayout::oproj(l), all, CtrLayout::gateup(l)));
            split_rows(H, nsm, sm, r0, r1);
            lists[sm].push_back(make(OP_DOWN, l, r0, r1, CtrLayout::gateup(l), all, CtrLayout::down(l)));
        }
    }
    for (int sm = 0; sm < nsm; sm++) {
        int32_t r0, r1;
        split_rows(V, nsm, sm, r0, r1);
        lists[sm].push_back(make(OP_LMHEAD, 0, r0, r1, CtrLayout::down(L - 1), all, -1));
    }
}

// Input-vector geometry for width K (see MvShape): among the splits of a row
// into k-slices of 256*vpl elements (vpl <= 8), pick the one that keeps the most
// consumer warps busy, rows per warp a power of two and vpl * rw <= 8 (register
// budget), then the smallest vpl. Returns false if K admits none.
bool mv_shape(int K, MvShape &m) {
    if (K <= 0 || K % 256 != 0 || K > 16384) return false;
    const int rows_fit = PAGE_BYTES / (2 * K);
    int best_active = 0;
    for (int vpl = 1; vpl <= MAX_VPL; vpl++) {
        if (K % (256 * vpl) != 0) continue;
        const int ws = K / (256 * vpl);
        if (ws > NCW) continue;
        int rg = std::min(NCW / ws, rows_fit);
        if (rg < 1) continue;
        int rw = 1;
        while (rw * 2 * rg <= rows_fit && rw * 2 <= 8 && vpl * rw * 2 <= 8) rw *= 2;
        const int rpp = rg * rw;
        if (rpp > MAX_RPP || rpp * ws > MAX_PART) continue;
        const int active = ws * rg;
        if (active > best_active) {
            best_active = active;
            m = MvShape{K, ws, vpl, rpp, rg, rw};
        }
    }
    return best_active > 0;
}

}  // namespace ll
