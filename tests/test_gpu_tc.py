"""The tensor-core matrix-vector pages (LL_MV_TC=1) against the CPU oracle, and
against the CUDA-core pages of the same kernel design.

The tensor-core pages hold up to eight rows of one 2048- (or 1024-) column chunk
of a matrix, loaded by TMA in the 128-byte swizzle, and multiply them with
three bf16 terms of the input on mma.sync; the tensor-core kernel takes every
width on them, so it needs every width a multiple of 1024 (the 1B, 3B and 8B
shapes, the H=1024 test shape). The parity rule is the logits' rule.
"""
import numpy as np
import pytest

from decode_megakernel_persistent_gb300 import ll, synth
from helpers import Pair, compare_logits, check_token

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _tc(monkeypatch):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from decode_megakernel_persistent_gb300 import build
    build.build()
    monkeypatch.setenv("LL_MV_TC", "1")


def test_tensor_core_pages_are_active_for_1b():
    wl = synth.WORKLOADS["1b"]
    pr = Pair(wl.shape, 8)
    assert pr.dec.query(ll.LL_Q_MV_TC) == 7  # hidden, n_q*head_dim and inter widths
    pr.close()


def test_llama1b_ctx1024_tensor_core_pages():
    wl = synth.WORKLOADS["1b"]
    shape, ctx = wl.shape, wl.context
    pr = Pair(shape, ctx + 2, kv_fill=ctx)
    tok = 17
    for i in range(2):
        _, tok, _ = pr.step(tok, ctx + i, what=f"1b tc pos {ctx + i}")
    pr.kv_close(slice(ctx, ctx + 2))
    pr.close()


@pytest.mark.parametrize("flash", ["0", "1"], ids=["block-attention", "per-warp-attention"])
def test_h1024_prefill_and_decode_tensor_core_pages(flash, monkeypatch):
    # H = 1024: one 1024-column chunk, 16 warps of 64 columns each; inter 3072:
    # three chunks; pages of 8 rows with ragged last pages
    monkeypatch.setenv("LL_ATTN_FLASH", flash)
    shape = synth.ModelShape("h1024", 2, 1024, 16, 4, 64, 3072, 4096, True)
    pr = Pair(shape, 160, gain_jitter=0.25)
    assert pr.dec.query(ll.LL_Q_MV_TC) == 7
    toks = synth.make_tokens(shape.vocab, 150, seed=1)
    tok = toks[0]
    for pos in range(150):
        _, ref_next, _ = pr.step(tok, pos)
        tok = toks[pos + 1] if pos + 1 < 140 else ref_next
    pr.close()


def test_multi_step_launch_equals_chained_steps_tensor_core_pages():
    shape, ctx, n = synth.LLAMA_1B, 64, 6
    w = synth.make_weights(shape, seed=0, device="cuda")
    out = []
    for multi in (False, True):
        k, v = synth.make_kv(shape, ctx + n + 1, ctx, seed=2, device="cuda")
        dec = ll.Decoder(shape, w, k, v, ctx + n + 1)
        assert dec.query(ll.LL_Q_MV_TC) == 7
        logits = torch.empty((n, shape.vocab), dtype=torch.float32, device="cuda")
        toks = torch.zeros(n, dtype=torch.int32, device="cuda")
        tok = torch.tensor([5], dtype=torch.int32, device="cuda")
        if multi:
            dec.steps(tok, ctx, n, logits, toks)
        else:
            t = tok.clone()
            for i in range(n):
                dec.step_async(t, ctx + i, logits[i], toks[i:i + 1])
                t = toks[i:i + 1]
        dec.synchronize()
        out.append((logits.cpu().numpy(), toks.cpu().numpy(), k.clone(), v.clone()))
        dec.close()
    np.testing.assert_array_equal(out[0][0], out[1][0])
    np.testing.assert_array_equal(out[0][1], out[1][1])
    assert torch.equal(out[0][2], out[1][2]) and torch.equal(out[0][3], out[1][3])


def test_tensor_core_and_cuda_core_pages_agree(monkeypatch):
    wl = synth.WORKLOADS["1b"]
    shape, ctx = wl.shape, wl.context
    w = synth.make_weights(shape, seed=0, device="cuda")
    res = []
    for tc in ("1", "0"):
        monkeypatch.setenv("LL_MV_TC", tc)
        k, v = synth.make_kv(shape, ctx + 1, ctx, seed=2, device="cuda")
        dec = ll.Decoder(shape, w, k, v, ctx + 1)
        assert dec.query(ll.LL_Q_MV_TC) == (7 if tc == "1" else 0)
        logits = torch.empty(shape.vocab, dtype=torch.float32, device="cuda")
        nxt = dec.step(11, ctx, logits)
        res.append((nxt, logits.cpu().numpy()))
        dec.close()
    compare_logits(res[0][1], res[1][1], "tensor-core vs CUDA-core pages")
    check_token(res[0][0], res[1][1], "tensor-core vs CUDA-core pages")
