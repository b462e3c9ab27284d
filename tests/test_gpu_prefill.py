"""ll_prefill (a prompt's positions through the model at once, tcgen05 GEMMs)
against the CPU oracle run position by position: every K/V entry the prefill
writes, the last position's logits element by element and its greedy token,
then decode steps that continue from the prefilled cache. Also a prefill that
continues a cache already holding earlier positions, and ragged position counts
(not multiples of the GEMM's 128-row tiles)."""
import numpy as np
import pytest

from decode_megakernel_persistent_gb300 import ll, synth
from helpers import Pair, check_token, compare_logits

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from decode_megakernel_persistent_gb300 import build
    build.build()


def _prefill(pr, toks, pos0):
    t = torch.tensor(toks, dtype=torch.int32, device="cuda")
    logits = torch.empty(pr.shape.vocab, dtype=torch.float32, device="cuda")
    nxt = torch.zeros(1, dtype=torch.int32, device="cuda")
    pr.dec.prefill(t, pos0, logits, nxt)
    pr.dec.synchronize()
    return logits.cpu().numpy(), int(nxt.item())


def _oracle_run(pr, toks, pos0):
    ref = None
    for i, t in enumerate(toks):
        ref, _ = pr.orc.decode_step(t, pos0 + i)
    return ref


@pytest.mark.parametrize("n", [1, 100, 200])
def test_tiny_prefill_matches_oracle(n):
    shape = synth.TINY
    pr = Pair(shape, 256, gain_jitter=0.25)
    toks = synth.make_tokens(shape.vocab, n, seed=1)
    got, nxt = _prefill(pr, toks, 0)
    ref = _oracle_run(pr, toks, 0)
    compare_logits(got, ref, f"prefill of {n}: last logits")
    check_token(nxt, ref, f"prefill of {n}")
    pr.kv_close(slice(0, n))
    pr.close()


def test_prefill_continues_a_cache_then_decodes():
    # 60 positions by decode steps, 90 by one prefill from position 60, then 8
    # greedy decode steps on top, all against the oracle
    shape = synth.TINY
    pr = Pair(shape, 200)
    toks = synth.make_tokens(shape.vocab, 150, seed=5)
    for pos in range(60):
        pr.step(toks[pos], pos)
    got, nxt = _prefill(pr, toks[60:150], 60)
    ref = _oracle_run(pr, toks[60:150], 60)
    compare_logits(got, ref, "continued prefill: last logits")
    check_token(nxt, ref, "continued prefill")
    pr.kv_close(slice(60, 150))
    tok = int(np.argmax(ref))
    for pos in range(150, 158):
        _, tok, _ = pr.step(tok, pos)
    pr.close()


def test_llama1b_prefill_of_64_positions():
    shape = synth.LLAMA_1B
    pr = Pair(shape, 80)
    toks = synth.make_tokens(shape.vocab, 64, seed=1)
    got, nxt = _prefill(pr, toks, 0)
    ref = _oracle_run(pr, toks, 0)
    compare_logits(got, ref, "1B prefill: last logits")
    check_token(nxt, ref, "1B prefill")
    pr.kv_close(slice(0, 64))
    pr.close()


@pytest.mark.parametrize("shape", [
    # 128-dim heads, four query heads per KV head: two K/V tiles per softmax round
    synth.ModelShape("h1024hd128", 2, 1024, 8, 2, 128, 2048, 4096, True),
    # eight query heads per KV head: one query position per warp
    synth.ModelShape("h1024gqa8", 2, 1024, 16, 2, 64, 2048, 4096, True),
], ids=["hd128", "gqa8"])
def test_prefill_head_layouts(shape):
    # 141 positions: two 128-row GEMM tiles, the second ragged, and an odd number
    # of 16-position K/V tiles (the last two-tile round has one)
    pr = Pair(shape, 160, gain_jitter=0.25)
    toks = synth.make_tokens(shape.vocab, 141, seed=7)
    got, nxt = _prefill(pr, toks, 0)
    ref = _oracle_run(pr, toks, 0)
    compare_logits(got, ref, f"{shape.name} prefill: last logits")
    check_token(nxt, ref, f"{shape.name} prefill")
    pr.kv_close(slice(0, 141))
    pr.close()


def test_prefill_argument_checks():
    shape = synth.TINY
    w = synth.make_weights(shape, seed=0, device="cuda")
    k, v = synth.make_kv(shape, 16, 0, device="cuda")
    dec = ll.Decoder(shape, w, k, v, 16)
    t = torch.zeros(17, dtype=torch.int32, device="cuda")
    nxt = torch.zeros(1, dtype=torch.int32, device="cuda")
    with pytest.raises(ll.LLError) as e:
        dec.prefill(t, 0, None, nxt)  # 17 positions in a 16-position cache
    assert e.value.code == ll.LL_ERR_ARG
    bad = torch.tensor([1, shape.vocab, 2], dtype=torch.int32, device="cuda")
    dec.prefill(bad, 0, None, nxt)
    with pytest.raises(ll.LLError) as e:
        dec.synchronize()
    assert e.value.code == ll.LL_ERR_ARG  # the out-of-range token, seen on the device
    dec.prefill(t[:5], 0, None, nxt)  # works afterwards
    dec.synchronize()
    dec.close()
