"""Small-batch decode (ll_init_batch / ll_decode_steps_batch): n = 2, 4 and 8
sequences share every pass over the weights, each with its own KV cache,
position and greedy tokens. Each sequence is checked against its own CPU oracle
instance, element by element on every step's logits (the oracle is fed the
tokens the kernel chose for that sequence), with the KV entries the steps wrote.
"""
import numpy as np
import pytest

import oracle
from decode_megakernel_persistent_gb300 import ll, synth
from helpers import check_token, compare_logits, widen_bits, TOL_L2, TOL_MAX

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu

# a shape whose every width is a multiple of 1024 (the batched kernel's pages):
# hidden 1024 (one chunk), n_q*head_dim 1024, inter 3072 (three chunks), GQA 4:1
SMALL = synth.ModelShape("h1024", 2, 1024, 16, 4, 64, 3072, 4096, True)
# the same with inter 2048: every width has two-sequence CUDA-core geometry, so a
# batch of two runs on CUDA-core pages
SMALL_CC = synth.ModelShape("h1024i2048", 2, 1024, 16, 4, 64, 2048, 4096, True)


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from decode_megakernel_persistent_gb300 import build
    build.build()


def _i32(vals):
    return torch.tensor(vals, dtype=torch.int32, device="cuda")


def run_batch(shape, n, fills, n_steps, seed=0, jitter=0.0, tok0=None, expect_cc=None):
    """n sequences whose caches hold N(0,1) entries for their first fills[b]
    positions; one launch of n_steps steps from position fills[b]. Returns the
    oracles (fed the kernel's tokens), tokens [n_steps][n], logits [n_steps][n][V]."""
    max_seq = max(fills) + n_steps + 1
    w = synth.make_weights(shape, seed=seed, device="cuda", gain_jitter=jitter)
    wh = synth.weights_to_host_bits(w)
    ks, vs, orcs = [], [], []
    for b in range(n):
        k, v = synth.make_kv(shape, max_seq, fills[b], seed=10 + b, device="cuda")
        ks.append(k)
        vs.append(v)
        o = oracle.OracleModel(shape.as_dict(), wh, max_seq, prec=32)
        o.k_cache[...] = synth.to_host_bits(k)
        o.v_cache[...] = synth.to_host_bits(v)
        orcs.append(o)
    dec = ll.BatchDecoder(shape, w, ks, vs, max_seq)
    # tensor-core pages, or (two sequences whose widths allow it) CUDA-core pages
    assert dec.query(ll.LL_Q_BATCH) == n
    assert dec.query(ll.LL_Q_MV_TC) == 7 or (n == 2 and dec.query(ll.LL_Q_BATCH_CC) == 1)
    if expect_cc is not None:
        assert dec.query(ll.LL_Q_BATCH_CC) == int(expect_cc)
    first = tok0 if tok0 is not None else synth.make_tokens(shape.vocab, n, seed=3)
    logits = torch.full((n_steps, n, shape.vocab), float("nan"), dtype=torch.float32, device="cuda")
    toks = torch.zeros((n_steps, n), dtype=torch.int32, device="cuda")
    dec.steps_batch(_i32(first), list(fills), n_steps, logits, toks)
    dec.synchronize()
    out = (toks.cpu().numpy(), logits.cpu().numpy(), [synth.to_host_bits(k) for k in ks],
           [synth.to_host_bits(v) for v in vs])
    dec.close()
    return orcs, first, out


def check_against_oracles(orcs, first, out, fills, n_steps, what):
    toks, logits, kb, vb = out
    for b, o in enumerate(orcs):
        tok = int(first[b])
        for i in range(n_steps):
            ref, _ = o.decode_step(tok, fills[b] + i)
            compare_logits(logits[i, b], ref, f"{what} seq {b} step {i}")
            check_token(int(toks[i, b]), ref, f"{what} seq {b} step {i}")
            tok = int(toks[i, b])
        # the K/V entries the kernel wrote for this sequence, each layer at the logits' bar
        for g, ob, name in ((kb[b], o.k_cache, "K"), (vb[b], o.v_cache, "V")):
            sl = slice(fills[b], fills[b] + n_steps)
            a = widen_bits(g[:, :, sl]).astype(np.float64)
            r = widen_bits(ob[:, :, sl]).astype(np.float64)
            for l in range(a.shape[0]):
                rel = np.linalg.norm(a[l] - r[l]) / max(np.linalg.norm(r[l]), 1e-30)
                assert np.max(np.abs(a[l] - r[l])) <= TOL_MAX * np.max(np.abs(r[l])) and rel <= TOL_L2, \
                    f"{what} seq {b} {name} layer {l}: rel {rel:.3e}"


@pytest.mark.parametrize("n", [2, 4, 8])
def test_batch_small_model_every_step_matches_oracles(n):
    # different positions per sequence, on both sides of a 128-position split
    fills = [40 + 37 * b for b in range(n)]
    orcs, first, out = run_batch(SMALL, n, fills, 6, jitter=0.25)
    check_against_oracles(orcs, first, out, fills, 6, f"batch {n}")


@pytest.mark.parametrize("n", [2, 4])
def test_batch_per_warp_attention_variant(n, monkeypatch):
    # the per-warp (flash) attention on each sequence's own KV tensor maps
    monkeypatch.setenv("LL_ATTN_FLASH", "1")
    fills = [200 + 61 * b for b in range(n)]
    orcs, first, out = run_batch(SMALL, n, fills, 5)
    check_against_oracles(orcs, first, out, fills, 5, f"per-warp batch {n}")


def test_batch_from_empty_caches():
    # every sequence from position 0 (its cache written by the launch itself),
    # 20 greedy steps, every step against the oracles
    n, steps = 4, 20
    orcs, first, out = run_batch(SMALL, n, [0] * n, steps)
    check_against_oracles(orcs, first, out, [0] * n, steps, "from empty")


def test_batch_of_one_equals_single_sequence_tensor_core_handle(monkeypatch):
    monkeypatch.setenv("LL_MV_TC", "1")
    shape, ctx, steps = SMALL, 50, 5
    w = synth.make_weights(shape, seed=0, device="cuda")
    res = []
    for batched in (True, False):
        k, v = synth.make_kv(shape, ctx + steps, ctx, seed=2, device="cuda")
        logits = torch.empty((steps, shape.vocab), dtype=torch.float32, device="cuda")
        toks = torch.zeros(steps, dtype=torch.int32, device="cuda")
        if batched:
            dec = ll.BatchDecoder(shape, w, [k], [v], ctx + steps)
            dec.steps_batch(_i32([9]), [ctx], steps, logits, toks)
        else:
            dec = ll.Decoder(shape, w, k, v, ctx + steps)
            assert dec.query(ll.LL_Q_MV_TC) == 7
            dec.steps(_i32([9]), ctx, steps, logits, toks)
        dec.synchronize()
        res.append((logits.cpu().numpy(), toks.cpu().numpy(), k.clone(), v.clone()))
        dec.close()
    np.testing.assert_array_equal(res[0][0], res[1][0])
    np.testing.assert_array_equal(res[0][1], res[1][1])
    assert torch.equal(res[0][2], res[1][2]) and torch.equal(res[0][3], res[1][3])


@pytest.mark.parametrize("n", [2, 8])
def test_batch_llama1b_ctx1024(n):
    shape, ctx = synth.LLAMA_1B, 1024
    fills = [ctx - 8 * b for b in range(n)]
    orcs, first, out = run_batch(shape, n, fills, 2)
    check_against_oracles(orcs, first, out, fills, 2, f"1b batch {n}")


def test_batch_sequences_are_independent():
    # sequence 0's results do not depend on what the other sequences decode
    n, steps, fills = 4, 4, [60, 60, 60, 60]
    _, _, a = run_batch(SMALL, n, fills, steps, tok0=[5, 6, 7, 8])
    _, _, b = run_batch(SMALL, n, fills, steps, tok0=[5, 100, 200, 300])
    np.testing.assert_array_equal(a[0][:, 0], b[0][:, 0])
    np.testing.assert_array_equal(a[1][:, 0], b[1][:, 0])


@pytest.mark.parametrize("n", [2, 4])
@pytest.mark.parametrize("flash", ["0", "1"], ids=["block-softmax", "per-warp"])
def test_batch_128_dim_heads(n, flash, monkeypatch):
    # 128-dim heads (four query heads per KV head) in both attention variants:
    # two sequences on CUDA-core pages, four on tensor-core pages
    monkeypatch.setenv("LL_ATTN_FLASH", flash)
    shape = synth.ModelShape("h1024hd128", 2, 1024, 8, 2, 128, 2048, 4096, True)
    fills = [150 + 37 * b for b in range(n)]
    orcs, first, out = run_batch(shape, n, fills, 4, jitter=0.25, expect_cc=(n == 2))
    check_against_oracles(orcs, first, out, fills, 4, f"hd128 batch {n}")


def test_batch_argument_checks():
    shape = SMALL
    w = synth.make_weights(shape, seed=0, device="cuda")
    kv = [synth.make_kv(shape, 16, 0, device="cuda") for _ in range(3)]
    with pytest.raises(ll.LLError) as e:
        ll.BatchDecoder(shape, w, [x[0] for x in kv], [x[1] for x in kv], 16)
    assert e.value.code == ll.LL_ERR_ARG  # 3 sequences
    dec = ll.BatchDecoder(shape, w, [x[0] for x in kv[:2]], [x[1] for x in kv[:2]], 16)
    logits = torch.empty((2, 2, shape.vocab), dtype=torch.float32, device="cuda")
    toks = torch.zeros((2, 2), dtype=torch.int32, device="cuda")
    with pytest.raises(ll.LLError) as e:
        dec.steps_batch(_i32([1, 2]), [0, 15], 2, logits, toks)  # past max_seq
    assert e.value.code == ll.LL_ERR_ARG
    with pytest.raises(ll.LLError) as e:
        dec.step(1, 0)  # single-sequence calls are refused on a batched handle
    assert e.value.code == ll.LL_ERR_ARG
    with pytest.raises(ll.LLError) as e:
        dec.steps_batch(_i32([1, shape.vocab]), [0, 0], 2, logits, toks)
        dec.synchronize()
    assert e.value.code == ll.LL_ERR_ARG  # a token out of range, seen on the device
    dec.steps_batch(_i32([1, 2]), [0, 0], 2, logits, toks)  # works afterwards
    dec.synchronize()
    dec.close()
    tiny = synth.TINY  # widths not multiples of 1024
    wt = synth.make_weights(tiny, seed=0, device="cuda")
    kt = [synth.make_kv(tiny, 16, 0, device="cuda") for _ in range(2)]
    with pytest.raises(ll.LLError) as e:
        ll.BatchDecoder(tiny, wt, [x[0] for x in kt], [x[1] for x in kt], 16)
    assert e.value.code == ll.LL_ERR_SHAPE


def test_batch_of_two_on_cuda_core_pages_every_step():
    # each page read once for both sequences; the sequences at different positions
    fills = [70, 190]
    orcs, first, out = run_batch(SMALL_CC, 2, fills, 8, jitter=0.25, expect_cc=True)
    check_against_oracles(orcs, first, out, fills, 8, "cuda-core batch 2")


def test_batch_of_two_on_cuda_core_pages_from_empty_and_per_warp(monkeypatch):
    orcs, first, out = run_batch(SMALL_CC, 2, [0, 0], 12, expect_cc=True)
    check_against_oracles(orcs, first, out, [0, 0], 12, "cuda-core batch 2 from empty")
    monkeypatch.setenv("LL_ATTN_FLASH", "1")
    fills = [300, 213]
    orcs, first, out = run_batch(SMALL_CC, 2, fills, 4, expect_cc=True)
    check_against_oracles(orcs, first, out, fills, 4, "cuda-core batch 2, per-warp attention")


def test_batch_of_two_tensor_core_pages_on_request(monkeypatch):
    monkeypatch.setenv("LL_BATCH_CC", "0")
    fills = [70, 190]
    orcs, first, out = run_batch(SMALL_CC, 2, fills, 3, expect_cc=False)
    check_against_oracles(orcs, first, out, fills, 3, "tensor-core batch 2")


def test_batch_llama1b_two_sequences_on_cuda_core_pages():
    shape, ctx = synth.LLAMA_1B, 1024
    fills = [ctx, ctx - 300]
    orcs, first, out = run_batch(shape, 2, fills, 3, expect_cc=True)
    check_against_oracles(orcs, first, out, fills, 3, "1b cuda-core batch 2")


@pytest.mark.parametrize("cc", [True, False])
def test_batch_dropped_signal_times_out_and_recovers(cc, monkeypatch):
    # a gate/up instruction that stores its outputs with a tag no reader accepts:
    # the launch reports a dependency timeout, and after the fault is removed the
    # same steps run and match the oracles (CUDA-core and tensor-core pages)
    if not cc:
        monkeypatch.setenv("LL_BATCH_CC", "0")
    shape, n, fills, steps = SMALL_CC, 2, [30, 57], 3
    max_seq = max(fills) + steps + 1
    w = synth.make_weights(shape, seed=0, device="cuda")
    wh = synth.weights_to_host_bits(w)
    ks, vs, orcs = [], [], []
    for b in range(n):
        k, v = synth.make_kv(shape, max_seq, fills[b], seed=10 + b, device="cuda")
        ks.append(k)
        vs.append(v)
        o = oracle.OracleModel(shape.as_dict(), wh, max_seq, prec=32)
        o.k_cache[...] = synth.to_host_bits(k)
        o.v_cache[...] = synth.to_host_bits(v)
        orcs.append(o)
    dec = ll.BatchDecoder(shape, w, ks, vs, max_seq)
    assert dec.query(ll.LL_Q_BATCH_CC) == int(cc)
    first = synth.make_tokens(shape.vocab, n, seed=3)
    toks = torch.zeros((steps, n), dtype=torch.int32, device="cuda")
    ll.ll_set_timeout_ns(dec.handle, 20_000_000)  # 20 ms
    ll.ll_debug_inject(dec.handle, ll.LL_FAULT_DROP_SIGNAL, 1, ll.OP_GATEUP)
    dec.steps_batch(_i32(first), list(fills), 1, None, toks[:1])
    with pytest.raises(ll.LLError) as e:
        dec.synchronize()
    assert e.value.code == ll.LL_ERR_DEP_TIMEOUT
    ll.ll_debug_inject(dec.handle, ll.LL_FAULT_NONE)
    ll.ll_set_timeout_ns(dec.handle, 1_000_000_000)
    logits = torch.full((steps, n, shape.vocab), float("nan"), dtype=torch.float32, device="cuda")
    dec.steps_batch(_i32(first), list(fills), steps, logits, toks)
    dec.synchronize()
    out = (toks.cpu().numpy(), logits.cpu().numpy(), [synth.to_host_bits(k) for k in ks],
           [synth.to_host_bits(v) for v in vs])
    dec.close()
    check_against_oracles(orcs, first, out, fills, steps, f"after a dropped signal (cc={cc})")
