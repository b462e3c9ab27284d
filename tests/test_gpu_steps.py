"""Multi-step launches (ll_decode_steps): n greedy steps in one launch of the
persistent kernel, each fed the token the previous step chose.

They run the same kernels' arithmetic in the same order as n single-step
launches chained on the device, so tokens, logits and the KV entries they write
must be bit-identical to those; and every step's logits must match the CPU
oracle fed the same tokens, within the parity bar of the other tests.
"""
import os

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


def _i32(vals):
    return torch.tensor(vals, dtype=torch.int32, device="cuda")


def run(shape, w, ctx, n, mode, backend=ll.LL_BACKEND_MEGAKERNEL, tok0=7, split=None):
    """Decode n steps from position ctx on a seeded cache; returns tokens, logits [n][V], K, V."""
    k, v = synth.make_kv(shape, ctx + n, ctx, seed=2, device="cuda")
    dec = ll.Decoder(shape, w, k, v, ctx + n, backend)
    logits = torch.full((n, shape.vocab), float("nan"), dtype=torch.float32, device="cuda")
    toks = torch.zeros(n, dtype=torch.int32, device="cuda")
    first = _i32([tok0])
    if mode == "launch":
        cuts = [0, n] if split is None else [0, split, n]
        for a, b in zip(cuts[:-1], cuts[1:]):
            src = first if a == 0 else toks[a - 1:a]
            dec.steps(src, ctx + a, b - a, logits[a:b], toks[a:b])
    else:  # chained single-step launches
        for i in range(n):
            src = first if i == 0 else toks[i - 1:i]
            dec.step_async(src, ctx + i, logits[i], toks[i:i + 1])
    dec.synchronize()
    out = (toks.cpu().numpy(), logits.cpu().numpy(), synth.to_host_bits(k), synth.to_host_bits(v))
    dec.close()
    return out


def assert_same(a, b):
    np.testing.assert_array_equal(a[0], b[0])
    np.testing.assert_array_equal(a[1], b[1])
    np.testing.assert_array_equal(a[2], b[2])
    np.testing.assert_array_equal(a[3], b[3])


@pytest.mark.parametrize("shape,ctx,n", [(synth.TINY, 32, 16), (synth.LLAMA_1B, 64, 6)], ids=["tiny", "1b"])
def test_one_launch_equals_chained_steps(shape, ctx, n):
    w = synth.make_weights(shape, seed=0, device="cuda")
    a = run(shape, w, ctx, n, "launch")
    b = run(shape, w, ctx, n, "chained")
    assert np.all(np.isfinite(a[1]))
    assert_same(a, b)


@pytest.mark.parametrize("shape,ctx,n", [(synth.LLAMA_3B, 300, 3), (synth.LLAMA_8B, 5000, 3)], ids=["3b", "8b"])
def test_one_launch_equals_chained_steps_128_dim_heads(shape, ctx, n):
    # 128-dim heads: the 3B shape (block attention) and the untied 8B shape, whose
    # attention items at this context span several pages (per-warp variant)
    w = synth.make_weights(shape, seed=0, device="cuda")
    a = run(shape, w, ctx, n, "launch")
    b = run(shape, w, ctx, n, "chained")
    assert np.all(np.isfinite(a[1]))
    assert_same(a, b)
    del w
    torch.cuda.empty_cache()


def test_one_launch_equals_chained_steps_per_warp_attention():
    # the per-warp (tensor-core) attention variant, whose K/V pages come through
    # tensor maps: 1B shape at a context where each attention item spans pages
    shape = synth.LLAMA_1B
    w = synth.make_weights(shape, seed=0, device="cuda")
    old = os.environ.get("LL_ATTN_FLASH")
    os.environ["LL_ATTN_FLASH"] = "1"
    try:
        a = run(shape, w, 700, 4, "launch")
        b = run(shape, w, 700, 4, "chained")
    finally:
        if old is None:
            del os.environ["LL_ATTN_FLASH"]
        else:
            os.environ["LL_ATTN_FLASH"] = old
    assert_same(a, b)


def test_two_launches_equal_one():
    shape = synth.TINY
    w = synth.make_weights(shape, seed=6, device="cuda", gain_jitter=0.1)
    assert_same(run(shape, w, 20, 16, "launch", split=9), run(shape, w, 20, 16, "launch"))


def test_chain_backend_steps():
    shape = synth.TINY
    w = synth.make_weights(shape, seed=0, device="cuda")
    a = run(shape, w, 32, 8, "launch", backend=ll.LL_BACKEND_CHAIN)
    b = run(shape, w, 32, 8, "chained", backend=ll.LL_BACKEND_CHAIN)
    assert_same(a, b)
    m = run(shape, w, 32, 8, "launch")
    for i in range(8):
        compare_logits(m[1][i], a[1][i], f"step {i}: megakernel vs chain")


def test_every_step_matches_oracle():
    # the oracle is fed the tokens the GPU chose, so both walk the same sequence;
    # each GPU token must be the oracle's argmax unless its top-2 margin is tiny
    shape = synth.TINY
    ctx, n = 48, 12
    pr = Pair(shape, ctx + n, kv_fill=ctx)
    logits = torch.empty((n, shape.vocab), dtype=torch.float32, device="cuda")
    toks = torch.zeros(n, dtype=torch.int32, device="cuda")
    pr.dec.steps(_i32([3]), ctx, n, logits, toks)
    pr.dec.synchronize()
    got_t, got_l = toks.cpu().numpy(), logits.cpu().numpy()
    tok = 3
    for i in range(n):
        ref, _ = pr.orc.decode_step(tok, ctx + i)
        compare_logits(got_l[i], ref, f"step {i}")
        check_token(int(got_t[i]), ref, f"step {i}")
        tok = int(got_t[i])
    pr.kv_close(slice(ctx, ctx + n))
    pr.close()


def test_timed_configuration_matches_oracle_1b():
    # the launch bench.py times, at its model and context: one ll_decode_steps
    # launch at the 1B shape from a 1024-entry cache, every step against the oracle
    shape = synth.LLAMA_1B
    ctx, n = 1024, 3
    pr = Pair(shape, ctx + n, kv_fill=ctx)
    logits = torch.empty((n, shape.vocab), dtype=torch.float32, device="cuda")
    toks = torch.zeros(n, dtype=torch.int32, device="cuda")
    pr.dec.steps(_i32([17]), ctx, n, logits, toks)
    pr.dec.synchronize()
    got_t, got_l = toks.cpu().numpy(), logits.cpu().numpy()
    tok = 17
    for i in range(n):
        ref, _ = pr.orc.decode_step(tok, ctx + i)
        compare_logits(got_l[i], ref, f"step {i}")
        check_token(int(got_t[i]), ref, f"step {i}")
        tok = int(got_t[i])
    pr.kv_close(slice(ctx, ctx + n))
    pr.close()


def test_steps_argument_checks():
    shape = synth.TINY
    w = synth.make_weights(shape, seed=0, device="cuda")
    k, v = synth.make_kv(shape, 16, 0, device="cuda")
    dec = ll.Decoder(shape, w, k, v, 16)
    toks = torch.zeros(16, dtype=torch.int32, device="cuda")
    for pos, n in ((10, 7), (0, 0), (-1, 2)):
        with pytest.raises(ll.LLError) as e:
            dec.steps(_i32([1]), pos, n, None, toks)
        assert e.value.code == ll.LL_ERR_ARG
    dec.steps(_i32([1]), 10, 6, None, toks)  # up to the last position
    dec.synchronize()
    dec.close()


def test_steps_errors_are_reported_and_cleared():
    # a dependency wait that runs out inside a multi-step launch (an instruction's
    # completion removed from the schedule), then a first token out of range: each
    # is reported by ll_synchronize, and the next launch decodes normally again
    shape = synth.TINY
    w = synth.make_weights(shape, seed=0, device="cuda")
    ctx, n = 16, 4
    k, v = synth.make_kv(shape, ctx + 3 * n, ctx, seed=2, device="cuda")
    dec = ll.Decoder(shape, w, k, v, ctx + 3 * n)
    toks = torch.zeros(n, dtype=torch.int32, device="cuda")
    ll.ll_set_timeout_ns(dec.handle, 20_000_000)  # 20 ms
    ll.ll_debug_inject(dec.handle, ll.LL_FAULT_DROP_SIGNAL, 1, ll.OP_DOWN)
    dec.steps(_i32([1]), ctx, n, None, toks)
    with pytest.raises(ll.LLError) as e:
        dec.synchronize()
    assert e.value.code == ll.LL_ERR_DEP_TIMEOUT
    ll.ll_debug_inject(dec.handle, ll.LL_FAULT_NONE)
    ll.ll_set_timeout_ns(dec.handle, 1_000_000_000)
    dec.steps(_i32([shape.vocab + 3]), ctx, n, None, toks)
    with pytest.raises(ll.LLError) as e:
        dec.synchronize()
    assert e.value.code == ll.LL_ERR_ARG
    logits = torch.empty((n, shape.vocab), dtype=torch.float32, device="cuda")
    dec.steps(_i32([1]), ctx, n, logits, toks)
    dec.synchronize()
    got = toks.cpu().numpy()
    dec.close()
    # the same steps on a fresh handle and cache
    ref = run(shape, w, ctx, n, "launch", tok0=1)
    np.testing.assert_array_equal(got, ref[0])
    np.testing.assert_array_equal(logits.cpu().numpy(), ref[1])
