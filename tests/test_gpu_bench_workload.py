"""Parity on the workload bench.py times, as bench.py runs it: the Llama-3.2-1B
shape, a 1024-token random prompt through ll_prefill (tcgen05 GEMMs), then
greedy steps in one ll_decode_steps launch; and the same prompt prefilled one
position at a time by chained single-step launches (the chain-backend and
fallback way), whose per-position logits are checked too.

The oracle does not prefill 1024 positions in reasonable time, so:
  * it recomputes the first 32 prompt positions on its own from an empty cache,
    and each K/V entry the kernel wrote there must match its own;
  * it recomputes 4 random later positions p (and the last one) from the
    kernel's bf16 cache snapshot of positions 0..p-1: its K/V at p, and for the
    last position the logits, against the kernel's;
  * then, on the kernel's full 1024-position snapshot, every step of a 32-step
    greedy launch: logits element by element, and the token under the top-2
    margin rule (the oracle is fed the tokens the kernel chose, so both walk the
    same sequence).
"""
import numpy as np
import pytest

from decode_megakernel_persistent_gb300 import synth
from helpers import Pair, check_token, compare_logits, widen_bits, TOL_L2, TOL_MAX

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from decode_megakernel_persistent_gb300 import build
    build.build()


def _kv_entry_close(gpu_bits, orc_bits, what):
    """One position's K or V entries [L][n_kv][hd] on both sides, each layer
    against the logits' bar (as the other parity tests hold them)."""
    a = widen_bits(gpu_bits).astype(np.float64)
    b = widen_bits(orc_bits).astype(np.float64)
    for l in range(a.shape[0]):
        scale = max(float(np.max(np.abs(b[l]))), 1e-30)
        rel = float(np.linalg.norm(a[l] - b[l]) / max(np.linalg.norm(b[l]), 1e-30))
        assert np.max(np.abs(a[l] - b[l])) <= TOL_MAX * scale and rel <= TOL_L2, f"{what} layer {l}: rel {rel:.3e}"


@pytest.mark.parametrize("how", ["ll_prefill", "single-step launches"])
def test_prefilled_1b_ctx1024_then_greedy_launch(how):
    wl = synth.WORKLOADS["1b"]
    shape, ctx = wl.shape, wl.context
    n_dec = 32
    max_seq = ctx + n_dec + 1
    pr = Pair(shape, max_seq)
    rng = np.random.default_rng(4)
    probe = sorted(int(p) for p in rng.choice(np.arange(64, ctx - 1), size=4, replace=False)) + [ctx - 1]
    prompt = synth.make_tokens(shape.vocab, ctx, seed=1)
    prompt_dev = torch.tensor(prompt, dtype=torch.int32, device="cuda")
    logits = torch.empty((ctx, shape.vocab), dtype=torch.float32, device="cuda")
    nxt = torch.zeros(ctx, dtype=torch.int32, device="cuda")
    if how == "ll_prefill":  # as bench.py runs it: the prompt in one call
        pr.dec.prefill(prompt_dev, 0, logits[ctx - 1], nxt[ctx - 1:ctx])
        have = {ctx - 1}  # positions whose logits the call gives
    else:
        for pos in range(ctx):
            pr.dec.step_async(prompt_dev[pos:pos + 1], pos, logits[pos], nxt[pos:pos + 1])
        have = set(range(ctx))
    pr.dec.synchronize()
    k_snap, v_snap = synth.to_host_bits(pr.k), synth.to_host_bits(pr.v)

    # (1) the first 32 positions recomputed by the oracle from an empty cache
    for pos in range(32):
        ref, _ = pr.orc.decode_step(prompt[pos], pos)
        if pos in have:
            compare_logits(logits[pos].cpu().numpy(), ref, f"prompt pos {pos}")
        _kv_entry_close(k_snap[:, :, pos], pr.orc.k_cache[:, :, pos], f"K pos {pos}")
        _kv_entry_close(v_snap[:, :, pos], pr.orc.v_cache[:, :, pos], f"V pos {pos}")

    # (2) 4 random later positions and the last one, from the kernel's snapshot
    # of what precedes them
    for pos in probe:
        pr.orc.k_cache[:, :, :pos] = k_snap[:, :, :pos]
        pr.orc.v_cache[:, :, :pos] = v_snap[:, :, :pos]
        ref, _ = pr.orc.decode_step(prompt[pos], pos)
        if pos in have:
            compare_logits(logits[pos].cpu().numpy(), ref, f"prompt pos {pos}")
            if pos == ctx - 1:
                check_token(int(nxt[ctx - 1].item()), ref, "prompt's last position")
        _kv_entry_close(k_snap[:, :, pos], pr.orc.k_cache[:, :, pos], f"K pos {pos}")
        _kv_entry_close(v_snap[:, :, pos], pr.orc.v_cache[:, :, pos], f"V pos {pos}")

    # (3) a 32-step greedy launch on the full snapshot, every step against the oracle
    pr.orc.k_cache[:, :, :ctx] = k_snap[:, :, :ctx]
    pr.orc.v_cache[:, :, :ctx] = v_snap[:, :, :ctx]
    dec_logits = torch.empty((n_dec, shape.vocab), dtype=torch.float32, device="cuda")
    toks = torch.zeros(n_dec, dtype=torch.int32, device="cuda")
    pr.dec.steps(nxt[ctx - 1:ctx], ctx, n_dec, dec_logits, toks)
    pr.dec.synchronize()
    got_t, got_l = toks.cpu().numpy(), dec_logits.cpu().numpy()
    tok = int(nxt[ctx - 1].item())
    for i in range(n_dec):
        ref, _ = pr.orc.decode_step(tok, ctx + i)
        compare_logits(got_l[i], ref, f"decode step {i}")
        check_token(int(got_t[i]), ref, f"decode step {i}")
        tok = int(got_t[i])
    pr.kv_close(slice(ctx, ctx + n_dec))
    pr.close()
