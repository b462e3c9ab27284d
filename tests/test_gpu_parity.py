"""Parity of the CUDA path (through the C ABI) with the CPU oracle, element by
element on every logit, plus the KV-cache entries each step writes.

Workloads: the tiny decoder run end to end (128-token prompt prefilled one
position at a time, then 16 greedy steps teacher-forced with the oracle's
token), and the full-size shapes at their own context lengths with the KV cache
filled from the seeded N(0,1) generator, both sides reading the same cache.
"""
import numpy as np
import pytest

from decode_megakernel_persistent_gb300 import ll, synth
from helpers import Pair, compare_logits, check_token

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu

BACKENDS = [pytest.param(ll.LL_BACKEND_MEGAKERNEL, id="megakernel"),
            pytest.param(ll.LL_BACKEND_CHAIN, id="chain")]


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from decode_megakernel_persistent_gb300 import build
    build.build()


@pytest.mark.parametrize("backend", BACKENDS)
@pytest.mark.parametrize("jitter", [0.0, 0.25], ids=["unit-gains", "random-gains"])
def test_tiny_prefill_and_greedy_decode(backend, jitter):
    wl = synth.WORKLOADS["tiny"]
    shape = wl.shape
    n_prompt, n_dec = wl.context, wl.decode_steps
    pr = Pair(shape, n_prompt + n_dec, backend, gain_jitter=jitter)
    prompt = synth.make_tokens(shape.vocab, n_prompt, seed=1)
    tok = prompt[0]
    worst = 0.0
    for pos in range(n_prompt + n_dec):
        nxt, ref_next, (md, rel) = pr.step(tok, pos)
        worst = max(worst, md)
        tok = prompt[pos + 1] if pos + 1 < n_prompt else ref_next
    pr.kv_close(slice(0, n_prompt + n_dec))
    pr.close()


@pytest.mark.parametrize("backend", BACKENDS)
def test_tiny_last_position_and_ragged_splits(backend):
    # pos = max_seq - 1 with a KV cache filled directly, at several lengths whose
    # split sizes are ragged (and at pos < number of splits, where splits are empty)
    shape = synth.TINY
    for max_seq in (1, 3, 77, 151, 300):
        pr = Pair(shape, max_seq, backend, kv_fill=max_seq - 1)
        pr.step(5, max_seq - 1, what=f"max_seq {max_seq}")
        pr.kv_close(slice(max_seq - 1, max_seq))
        pr.close()


# Head layouts beyond the Llama shapes: eight query heads per KV head, plain
# multi-head attention, and four 128-dim query heads per KV head.
GQA_SHAPES = [
    synth.ModelShape("gqa8-hd64", 2, 512, 8, 1, 64, 1024, 4096, True),
    synth.ModelShape("mha-hd64", 2, 512, 4, 4, 64, 1024, 4096, False),
    synth.ModelShape("gqa4-hd128", 2, 512, 8, 2, 128, 1536, 4096, True),
]


@pytest.mark.parametrize("shape", GQA_SHAPES, ids=lambda s: s.name)
@pytest.mark.parametrize("backend", BACKENDS)
def test_head_layouts(shape, backend):
    # positions on both sides of a 128-position split and of a page boundary
    max_seq = 300
    pr = Pair(shape, max_seq, backend, kv_fill=260, gain_jitter=0.25)
    tok = 11
    for pos in (260, 261):
        _, tok, _ = pr.step(tok, pos, what=f"{shape.name} pos {pos}")
    pr.kv_close(slice(260, 262))
    pr.close()


@pytest.mark.parametrize("shape", GQA_SHAPES + [synth.TINY], ids=lambda s: s.name)
def test_per_warp_softmax_variant(shape, monkeypatch):
    # the kernel variant that long attention items use (picked at init by the
    # longest item), forced here on short ones: several pages per item, the new
    # token folded in, and items with no cached positions (pos 0)
    monkeypatch.setenv("LL_ATTN_FLASH", "1")
    monkeypatch.setenv("LL_ATTN_SPLIT_POS", "256")
    max_seq = 400
    pr = Pair(shape, max_seq, ll.LL_BACKEND_MEGAKERNEL, kv_fill=390, gain_jitter=0.25)
    tok = 3
    for pos in (390, 391):
        _, tok, _ = pr.step(tok, pos, what=f"{shape.name} pos {pos}")
    pr.kv_close(slice(390, 392))
    pr.close()
    pr = Pair(shape, 8, ll.LL_BACKEND_MEGAKERNEL)
    pr.step(5, 0, what=f"{shape.name} pos 0")
    pr.close()


def _full_size(key, backend, steps=2):
    wl = synth.WORKLOADS[key]
    shape, ctx = wl.shape, wl.context
    pr = Pair(shape, ctx + steps, backend, kv_fill=ctx)
    toks = synth.make_tokens(shape.vocab, steps, seed=1)
    tok = toks[0]
    for i in range(steps):
        nxt, ref_next, _ = pr.step(tok, ctx + i, what=f"{key} pos {ctx + i}")
        tok = ref_next
    pr.kv_close(slice(ctx, ctx + steps))
    pr.close()


@pytest.mark.parametrize("backend", BACKENDS)
def test_llama1b_ctx1024(backend):
    _full_size("1b", backend)


def test_llama1b_ctx32768_megakernel():
    _full_size("1b-32k", ll.LL_BACKEND_MEGAKERNEL, steps=1)


def test_llama3b_ctx2048_megakernel():
    _full_size("3b", ll.LL_BACKEND_MEGAKERNEL, steps=1)


def test_llama8b_ctx8192_megakernel():
    _full_size("8b", ll.LL_BACKEND_MEGAKERNEL, steps=1)


def test_llama1b_from_empty_cache():
    # the first positions of a real prefill, KV written by the kernels themselves
    shape = synth.LLAMA_1B
    pr = Pair(shape, 8)
    toks = synth.make_tokens(shape.vocab, 4, seed=1)
    for pos, t in enumerate(toks):
        pr.step(t, pos)
    pr.kv_close(slice(0, 4))
    pr.close()


def test_async_chain_matches_sync_steps():
    # the launch configuration the benchmark times: tokens chained on the device
    shape = synth.LLAMA_1B
    ctx, n = 64, 6
    w = synth.make_weights(shape, seed=0, device="cuda")
    outs = []
    for mode in ("sync", "async"):
        k, v = synth.make_kv(shape, ctx + n, ctx, seed=2, device="cuda")
        dec = ll.Decoder(shape, w, k, v, ctx + n)
        logits = torch.empty(shape.vocab, dtype=torch.float32, device="cuda")
        toks = []
        if mode == "sync":
            t = 7
            for i in range(n):
                t = dec.step(t, ctx + i, logits)
                toks.append(t)
        else:
            tok = torch.tensor([7], dtype=torch.int32, device="cuda")
            for i in range(n):
                dec.step_async(tok, ctx + i, logits, tok)
                toks.append(None)
            dec.synchronize()
            toks[-1] = int(tok.item())
        outs.append((toks[-1], logits.cpu().numpy().copy(), synth.to_host_bits(k)))
        dec.close()
    assert outs[0][0] == outs[1][0]
    np.testing.assert_array_equal(outs[0][1], outs[1][1])
    np.testing.assert_array_equal(outs[0][2], outs[1][2])


def test_megakernel_is_deterministic_and_agrees_with_chain():
    shape = synth.TINY
    w = synth.make_weights(shape, seed=3, device="cuda", gain_jitter=0.1)
    res = []
    for backend in (ll.LL_BACKEND_MEGAKERNEL, ll.LL_BACKEND_MEGAKERNEL, ll.LL_BACKEND_CHAIN):
        k, v = synth.make_kv(shape, 40, 32, seed=2, device="cuda")
        dec = ll.Decoder(shape, w, k, v, 40, backend)
        logits = torch.empty(shape.vocab, dtype=torch.float32, device="cuda")
        for pos in range(32, 40):
            dec.step(11 + pos, pos, logits)
        res.append(logits.cpu().numpy().copy())
        dec.close()
    np.testing.assert_array_equal(res[0], res[1])
    compare_logits(res[0], res[2], "megakernel vs chain")


def test_resume_equals_uninterrupted():
    # 8 steps, free the handle, a new handle on the same caches continues: same as 16 in one go
    shape = synth.TINY
    w = synth.make_weights(shape, seed=4, device="cuda")
    toks = synth.make_tokens(shape.vocab, 16, seed=5)

    def run(split):
        k, v = synth.make_kv(shape, 16, 0, device="cuda")
        logits = torch.empty(shape.vocab, dtype=torch.float32, device="cuda")
        dec = ll.Decoder(shape, w, k, v, 16)
        for pos, t in enumerate(toks):
            if pos == split:
                dec.close()
                dec = ll.Decoder(shape, w, k, v, 16)
            dec.step(t, pos, logits)
        dec.close()
        return logits.cpu().numpy(), synth.to_host_bits(k)

    a, ka = run(8)
    b, kb = run(-1)
    np.testing.assert_array_equal(a, b)
    np.testing.assert_array_equal(ka, kb)
