"""The greedy token on exact ties: the smallest index among the equal largest
logits (the argmax step of the decode step), on every path that picks a token:
the megakernel's single and multi-step launches, the per-operation chain, the
prompt prefill, and batches on CUDA-core (2) and tensor-core (4) pages.

The model is made to tie: the final RMSNorm gain passes one hidden unit J only,
so logit i is the single product E[i, J] * h_J (the LM head is the tied
embedding E), the same for equal E[i, J] whatever the summation order. Rows UP
hold +1 at J and rows DOWN -1 (the other entries are ~N(0, 0.02)), so the
largest logit is shared by the UP rows when h_J > 0 and by the DOWN rows when
h_J < 0. The UP and DOWN rows straddle SM boundaries and share a page, so the
tie is decided within a warp, across warps and across SMs.
"""
import numpy as np
import pytest

import oracle
from decode_megakernel_persistent_gb300 import ll, synth

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu

# widths with both two-sequence CUDA-core and tensor-core batch geometry
SHAPE = synth.ModelShape("h1024i2048", 2, 1024, 16, 4, 64, 2048, 4096, True)
J = 77
UP = (1000, 1001, 3000)
DOWN = (1500, 3500)


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from decode_megakernel_persistent_gb300 import build
    build.build()


def tie_weights():
    w = synth.make_weights(SHAPE, seed=0, device="cuda")
    g = torch.zeros_like(w["final_norm"])
    g[J] = 1.0
    w["final_norm"] = g
    for r in UP:
        w["embed"][r, J] = 1.0
    for r in DOWN:
        w["embed"][r, J] = -1.0
    return w


def oracle_for(w, max_seq):
    return oracle.OracleModel(SHAPE.as_dict(), synth.weights_to_host_bits(w), max_seq, prec=32)


def expected(ref) -> int:
    """The lowest index among the oracle's largest logits, after checking that
    the largest value is the constructed tie."""
    ref = np.asarray(ref)
    winners = np.flatnonzero(ref == ref.max())
    assert tuple(winners) in (UP, DOWN), f"no constructed tie: {winners}"
    return int(winners[0])


def check_gpu_tie(logits, tok: int, want: int, what: str):
    lg = np.asarray(logits)
    rows = UP if want == UP[0] else DOWN
    assert np.all(lg[list(rows)] == lg[rows[0]]), f"{what}: tied rows differ on the GPU: {lg[list(rows)]}"
    assert tok == want, f"{what}: token {tok}, the lowest tied index is {want}"


@pytest.mark.parametrize("backend", [pytest.param(ll.LL_BACKEND_MEGAKERNEL, id="megakernel"),
                                     pytest.param(ll.LL_BACKEND_CHAIN, id="chain")])
def test_single_steps_take_lowest_tied_index(backend):
    max_seq = 16
    w = tie_weights()
    k, v = synth.make_kv(SHAPE, max_seq, 0, device="cuda")
    dec = ll.Decoder(SHAPE, w, k, v, max_seq, backend)
    orc = oracle_for(w, max_seq)
    logits = torch.empty(SHAPE.vocab, dtype=torch.float32, device="cuda")
    tok = 5
    for pos in range(8):
        nxt = dec.step(tok, pos, logits)
        ref, ref_next = orc.decode_step(tok, pos)
        want = expected(ref)
        assert ref_next == want
        check_gpu_tie(logits.cpu().numpy(), nxt, want, f"pos {pos}")
        tok = nxt
    dec.close()


def test_multi_step_launch_takes_lowest_tied_index():
    max_seq, n = 24, 12
    w = tie_weights()
    k, v = synth.make_kv(SHAPE, max_seq, 0, device="cuda")
    dec = ll.Decoder(SHAPE, w, k, v, max_seq)
    orc = oracle_for(w, max_seq)
    logits = torch.empty((n, SHAPE.vocab), dtype=torch.float32, device="cuda")
    toks = torch.zeros(n, dtype=torch.int32, device="cuda")
    dec.steps(torch.tensor([7], dtype=torch.int32, device="cuda"), 0, n, logits, toks)
    dec.synchronize()
    lg, tk = logits.cpu().numpy(), toks.cpu().numpy()
    tok = 7
    for i in range(n):
        ref, _ = orc.decode_step(tok, i)
        check_gpu_tie(lg[i], int(tk[i]), expected(ref), f"step {i}")
        tok = int(tk[i])
    dec.close()


def test_prefill_takes_lowest_tied_index():
    max_seq, n = 32, 9
    w = tie_weights()
    k, v = synth.make_kv(SHAPE, max_seq, 0, device="cuda")
    dec = ll.Decoder(SHAPE, w, k, v, max_seq)
    orc = oracle_for(w, max_seq)
    prompt = synth.make_tokens(SHAPE.vocab, n, seed=4)
    logits = torch.empty(SHAPE.vocab, dtype=torch.float32, device="cuda")
    tok = torch.zeros(1, dtype=torch.int32, device="cuda")
    dec.prefill(torch.tensor(prompt, dtype=torch.int32, device="cuda"), 0, logits, tok)
    dec.synchronize()
    for p, t in enumerate(prompt):
        ref, _ = orc.decode_step(t, p)
    check_gpu_tie(logits.cpu().numpy(), int(tok.item()), expected(ref), "prefill")
    dec.close()


@pytest.mark.parametrize("n", [2, 4])
def test_batch_takes_lowest_tied_index(n):
    max_seq, steps = 16, 6
    w = tie_weights()
    ks, vs = [], []
    for b in range(n):
        k, v = synth.make_kv(SHAPE, max_seq, 0, device="cuda")
        ks.append(k)
        vs.append(v)
    dec = ll.BatchDecoder(SHAPE, w, ks, vs, max_seq)
    assert dec.query(ll.LL_Q_BATCH_CC) == int(n == 2)
    first = [11 + 100 * b for b in range(n)]
    logits = torch.empty((steps, n, SHAPE.vocab), dtype=torch.float32, device="cuda")
    toks = torch.zeros((steps, n), dtype=torch.int32, device="cuda")
    dec.steps_batch(torch.tensor(first, dtype=torch.int32, device="cuda"), [0] * n, steps, logits, toks)
    dec.synchronize()
    lg, tk = logits.cpu().numpy(), toks.cpu().numpy()
    for b in range(n):
        orc = oracle_for(w, max_seq)
        tok = first[b]
        for i in range(steps):
            ref, _ = orc.decode_step(tok, i)
            check_gpu_tie(lg[i, b], int(tk[i, b]), expected(ref), f"batch {n} seq {b} step {i}")
            tok = int(tk[i, b])
    dec.close()
