"""Per-instruction timing of one megakernel decode step.

The page "Hazy Research Llama-3.2-1B Megakernel" breaks one forward pass down
into time spent waiting on dependencies and loads, on RMSNorm and matvec, on
weight-load stalls, synchronisation and set-up. This module measures the same
kind of breakdown from the kernel's own %globaltimer stamps (ll_set_trace):

  python -m decode_megakernel_persistent_gb300.trace [--workload 1b]

For every instruction kind it reports, averaged over layers and SMs, the time
from the instruction's start to its dependency being met and its input vector
loaded ("wait"), from there to its last page consumed ("body"), and to its
completion signal ("tail"), plus the time at which the last SM finished each
instruction kind of each layer.
"""
from __future__ import annotations

import argparse
import json

import numpy as np

OPS = ("qkv", "attn", "oproj", "gateup", "down", "lmhead")


def summarize(trace: np.ndarray, plan: np.ndarray) -> dict:
    """trace [nsm, max_instr, 12] uint64 stamps, plan [nsm, max_instr, 7] from ll_plan."""
    tr = trace.astype(np.int64)
    valid = plan[:, :, 0] >= 0
    t0 = tr[:, :, 0][valid].min()
    tr = tr - t0
    out = {"step_us": float(tr[:, :, 3][valid].max()) / 1e3, "ops": {}, "layers": []}
    for k, name in enumerate(OPS):
        m = valid & (plan[:, :, 0] == k)
        if not m.any():
            continue
        b, r, pg, e, pf, pl, f1, cd, w8, w9, w10, w11 = (tr[:, :, i][m] for i in range(12))
        issued = trace[:, :, 4][m] > 0
        had = trace[:, :, 6][m] > 0
        rec = {"wait_us": float(np.mean(r - b)) / 1e3, "body_us": float(np.mean(pg - r)) / 1e3,
               "tail_us": float(np.mean(e - pg)) / 1e3, "n": int(m.sum())}
        if had.any():
            # ready -> first page in hand, first page -> compute done, compute done -> pages done
            rec["to_first_page_us"] = float(np.mean((f1 - r)[had])) / 1e3
            rec["compute_us"] = float(np.mean((cd - f1)[had])) / 1e3
            rec["after_compute_us"] = float(np.mean((pg - cd)[had])) / 1e3
        if name == "attn" and (trace[:, :, 10][m] > 0).any():
            # phase stamps of the block-softmax variant (the per-warp one leaves them 0)
            sub = trace[:, :, 10][m] > 0
            rec["scores_us"] = float(np.mean((w8 - f1)[sub])) / 1e3
            rec["softmax_us"] = float(np.mean((w9 - w8)[sub])) / 1e3
            rec["pv_us"] = float(np.mean((w10 - w9)[sub])) / 1e3
        if issued.any():
            # producer: first page issued relative to the consumer reaching the
            # instruction (negative = issued ahead), and last issue relative to its end
            rec["first_issue_vs_begin_us"] = float(np.mean((pf - b)[issued])) / 1e3
            rec["last_issue_vs_end_us"] = float(np.mean((pl - e)[issued])) / 1e3
        out["ops"][name] = rec
    L = int(plan[:, :, 1][valid & (plan[:, :, 0] < 5)].max()) + 1
    for l in range(L):
        row = {}
        for k, name in enumerate(OPS[:5]):
            m = valid & (plan[:, :, 0] == k) & (plan[:, :, 1] == l)
            if m.any():
                row[name] = round(float(tr[:, :, 3][m].max()) / 1e3, 2)
        out["layers"].append(row)
    m = valid & (plan[:, :, 0] == 5)
    out["lmhead_end_us"] = float(tr[:, :, 3][m].max()) / 1e3
    return out


def page_stats(ptrace: np.ndarray, npages: int) -> dict:
    """ptrace [nsm, PTRACE_PAGES, 3]: issue, consumer start, release; npages used per SM."""
    pt = ptrace[:, :npages].astype(np.int64)
    ok = (pt > 0).all(axis=2)
    lat = (pt[:, :, 1] - pt[:, :, 0])[ok]   # issue -> first consumer starts on it
    work = (pt[:, :, 2] - pt[:, :, 1])[ok]  # consumer start -> release
    gap = np.diff(pt[:, :, 0], axis=1)[ok[:, 1:] & ok[:, :-1]]  # between issues
    pct = lambda a: {q: round(float(np.percentile(a, q)) / 1e3, 3) for q in (10, 50, 90)}
    return {"issue_to_start_us": pct(lat), "start_to_release_us": pct(work), "issue_gap_us": pct(gap)}


def issue_idle(tr: np.ndarray, pt: np.ndarray, plan: np.ndarray, bin_us: float = 0.5, idle_pages: int = 5,
               page_bytes: int = 32768) -> dict:
    """When the GPU as a whole issues no page loads. For each layer 1..L-2: its span
    (from the end of the previous layer's down projection on the slowest SM to the
    end of its own), the time in bins of bin_us in which all SMs together issued at
    most idle_pages pages, and the issue rate in the other bins (pages counted as
    page_bytes); means over those layers."""
    valid = plan[:, :, 0] >= 0
    t0 = tr[:, :, 0][valid].min()
    iss = (pt[:, :, 0].astype(np.int64) - t0) / 1e3
    iss = iss[pt[:, :, 0] > 0]
    nl = int(plan[:, :, 1][valid & (plan[:, :, 0] < 5)].max()) + 1
    spans, idle, rate = [], [], []
    for l in range(1, nl - 1):
        prev = valid & (plan[:, :, 1] == l - 1) & (plan[:, :, 0] == 4)
        cur = valid & (plan[:, :, 1] == l) & (plan[:, :, 0] == 4)
        if not prev.any() or not cur.any():
            continue
        b = (tr[:, :, 3][prev].max() - t0) / 1e3
        e = (tr[:, :, 3][cur].max() - t0) / 1e3
        nb = int((e - b) / bin_us)
        if nb < 1:
            continue
        h, _ = np.histogram(iss, bins=b + bin_us * np.arange(nb + 1))
        busy = h > idle_pages
        spans.append(e - b)
        idle.append(float((~busy).sum()) * bin_us)
        if busy.any():
            rate.append(float(h[busy].sum()) * page_bytes / (float(busy.sum()) * bin_us * 1e-6) / 1e9)
    if not spans:
        return {}
    return {"layer_span_us": round(float(np.mean(spans)), 2), "idle_us": round(float(np.mean(idle)), 2),
            "busy_issue_gbs": round(float(np.mean(rate)), 0) if rate else 0.0, "bin_us": bin_us,
            "idle_pages": idle_pages}


def main():
    import torch

    from . import build, ll, synth
    ap = argparse.ArgumentParser()
    ap.add_argument("--workload", default="1b")
    ap.add_argument("--steps", type=int, default=3, help="traced steps (the last is reported)")
    ap.add_argument("--save", default=None, help="write the raw trace and plan to this .npz")
    ap.add_argument("--load", default=None, help="summarise a trace written by --save (no GPU needed)")
    ap.add_argument("--notrace", action="store_true",
                    help="run the same steps with tracing off (a target for external profilers)")
    ap.add_argument("--l2-resident", action="store_true",
                    help="a 2-layer hidden-1024 model whose weights (~90 MB) stay in L2")
    ap.add_argument("--batch", type=int, default=0,
                    help="trace a batched handle of this many sequences (ll_init_batch)")
    ap.add_argument("--prefill", type=int, default=0,
                    help="with --notrace: run ll_prefill of this many prompt tokens (twice) instead of decode "
                         "steps (a target for external profilers)")
    ap.add_argument("--backend", default="megakernel", choices=["megakernel", "chain"],
                    help="with --notrace: the backend whose steps run")
    args = ap.parse_args()
    if args.load:
        d = np.load(args.load)
        tr, pt, plan = d["trace"], d["ptrace"], d["plan"]
        res = summarize(tr, plan)
        res["pages"] = page_stats(pt, pt.shape[1])
        res["issue"] = issue_idle(tr, pt, plan)
        print(json.dumps(res, indent=1))
        return
    build.build()
    wl = synth.WORKLOADS[args.workload]
    shape, ctx = wl.shape, wl.context
    if args.l2_resident:
        shape = synth.ModelShape("l2-resident", 2, 1024, 16, 4, 64, 4096, 16384, True)
        ctx = 1024
    max_seq = ctx + args.steps + 1
    w = synth.make_weights(shape, seed=0, device="cuda")
    if args.batch:
        kv = [synth.make_kv(shape, max_seq, ctx, seed=2 + b, device="cuda") for b in range(args.batch)]
        dec = ll.BatchDecoder(shape, w, [x[0] for x in kv], [x[1] for x in kv], max_seq)
    else:
        if args.prefill:
            max_seq = max(max_seq, args.prefill + 1)
        k, v = synth.make_kv(shape, max_seq, ctx if not args.prefill else 0, seed=2, device="cuda")
        dec = ll.Decoder(shape, w, k, v, max_seq,
                         ll.LL_BACKEND_CHAIN if args.backend == "chain" else ll.LL_BACKEND_MEGAKERNEL)
    nbytes = dec.query(ll.LL_Q_TRACE_BYTES)
    buf = torch.zeros(nbytes // 8, dtype=torch.int64, device="cuda")
    if not args.notrace:
        ll.ll_set_trace(dec.handle, buf)
    logits = torch.empty(shape.vocab, dtype=torch.float32, device="cuda")
    tok = 1
    if args.prefill and args.notrace:
        prompt = torch.tensor(synth.make_tokens(shape.vocab, args.prefill, seed=1), dtype=torch.int32, device="cuda")
        nxt = torch.zeros(1, dtype=torch.int32, device="cuda")
        for _ in range(2):
            dec.prefill(prompt, 0, logits, nxt)
        dec.synchronize()
        print(json.dumps({"prefill": args.prefill, "workload": wl.name, "traced": False}))
        dec.close()
        return
    for i in range(args.steps):
        if args.batch:  # every sequence one step, one launch per step
            toks = torch.ones((1, args.batch), dtype=torch.int32, device="cuda")
            dec.steps_batch(toks[0], [ctx + i] * args.batch, 1, None, toks)
            dec.synchronize()
        else:
            tok = dec.step(tok, ctx + i, logits)
    if args.notrace:
        torch.cuda.synchronize()
        print(json.dumps({"steps": args.steps, "workload": wl.name, "traced": False}))
        dec.close()
        return
    nsm = dec.query(ll.LL_Q_NUM_SMS)
    plan = ll.ll_handle_plan(dec.handle)
    flat = buf.cpu().numpy()
    n_instr_words = nsm * plan.shape[1] * 12
    tr = flat[:n_instr_words].reshape(nsm, plan.shape[1], 12)
    res = summarize(tr, plan)
    pt = flat[n_instr_words:].reshape(nsm, -1, 3)
    used = int(min(pt.shape[1], np.max(np.sum(pt[:, :, 0] > 0, axis=1))))
    res["pages"] = page_stats(pt, used)
    res["issue"] = issue_idle(tr, pt[:, :used], plan)
    if args.save:
        np.savez_compressed(args.save, trace=tr, ptrace=pt[:, :used], plan=plan)
    print(json.dumps(res, indent=1))
    dec.close()


if __name__ == "__main__":
    main()
