"""ll_decode_step_static, the decode step that allocates no device memory, against
the handle-based entry point ll_decode_step on the same weights and the same
KV-cache contents, on two calls in a row (the second call's token is the first
call's greedy output, at the next position).

Collected last on purpose (file name): it must pass alone in a fresh process and
after every other test, when the library and its module are long loaded.
"""
import ctypes

import numpy as np
import pytest

from decode_megakernel_persistent_gb300 import ll, synth
from helpers import compare_logits, check_token

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from decode_megakernel_persistent_gb300 import build
    build.build()


def _two_steps_each_way(shape, ctx, backend, jitter=0.0):
    w = synth.make_weights(shape, seed=0, device="cuda", gain_jitter=jitter)
    max_seq = ctx + 2
    cfg = ll.make_config(shape, max_seq)
    k_ref, v_ref = synth.make_kv(shape, max_seq, ctx, seed=2, device="cuda")
    k_st, v_st = synth.make_kv(shape, max_seq, ctx, seed=2, device="cuda")
    dec = ll.Decoder(shape, w, k_ref, v_ref, max_seq, backend)
    ref_logits = torch.empty(shape.vocab, dtype=torch.float32, device="cuda")
    st_logits = torch.empty(shape.vocab, dtype=torch.float32, device="cuda")
    tok_ref = tok_st = 17
    out = []
    for pos in (ctx, ctx + 1):
        tok_ref = dec.step(tok_ref, pos, ref_logits)
        tok_st = ll.ll_decode_step_static(cfg, w, k_st, v_st, tok_st, pos, st_logits)
        out.append((tok_ref, ref_logits.cpu().numpy().copy(), tok_st, st_logits.cpu().numpy().copy()))
    dec.close()
    return out, (k_ref, v_ref, k_st, v_st)


@pytest.mark.parametrize("key", ["tiny", "1b"])
def test_static_step_matches_megakernel_two_calls(key):
    wl = synth.WORKLOADS[key]
    out, _ = _two_steps_each_way(wl.shape, wl.context, ll.LL_BACKEND_MEGAKERNEL, jitter=0.25)
    for i, (tr, lr, ts, ls) in enumerate(out):
        compare_logits(ls, lr, f"{key} call {i}")
        check_token(ts, lr, f"{key} call {i}")
        # the second call takes the first call's token: follow the handle's if they differ
        assert tr == ts or i == len(out) - 1


def test_static_step_equals_chain_backend_bit_for_bit():
    # the same per-operation kernels, launch shapes, KV splits and RoPE values
    wl = synth.WORKLOADS["1b"]
    out, (k_ref, v_ref, k_st, v_st) = _two_steps_each_way(wl.shape, wl.context, ll.LL_BACKEND_CHAIN)
    for tr, lr, ts, ls in out:
        assert tr == ts
        np.testing.assert_array_equal(ls, lr)
    assert torch.equal(k_ref, k_st) and torch.equal(v_ref, v_st)


def test_static_step_without_logits_buffer():
    shape = synth.TINY
    w = synth.make_weights(shape, seed=0, device="cuda")
    k, v = synth.make_kv(shape, 16, 8, seed=2, device="cuda")
    k2, v2 = k.clone(), v.clone()
    cfg = ll.make_config(shape, 16)
    logits = torch.empty(shape.vocab, dtype=torch.float32, device="cuda")
    a = ll.ll_decode_step_static(cfg, w, k, v, 3, 8, logits)
    b = ll.ll_decode_step_static(cfg, w, k2, v2, 3, 8, None)
    assert a == b == int(torch.argmax(logits).item())


def test_static_step_rejects_oversized_scratch_and_bad_args():
    shape = synth.TINY
    w = synth.make_weights(shape, seed=0, device="cuda")
    k, v = synth.make_kv(shape, 16, 0, seed=2, device="cuda")
    big = ll.make_config(shape, 16)
    big.vocab = ll.LL_STATIC_SCRATCH_BYTES // 4 + 1  # logits alone overflow the array
    # the binding refuses weights that do not fit the configuration ...
    with pytest.raises(ll.LLError) as e:
        ll.ll_decode_step_static(big, w, k, v, 1, 0, None)
    assert e.value.code == ll.LL_ERR_ARG
    # ... and the library itself refuses the scratch it cannot hold, before any
    # launch (the raw C call, past the binding's checks)
    ws, keep = ll._weights_struct(w)
    nxt = ctypes.c_int32(-1)
    err = ctypes.create_string_buffer(256)
    rc = ll.lib().ll_decode_step_static(ctypes.byref(big), ctypes.byref(ws), k.data_ptr(), v.data_ptr(), 1, 0, None,
                                        ctypes.byref(nxt), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream),
                                        err, len(err))
    del keep
    assert rc == ll.LL_ERR_SHAPE and b"LL_STATIC_SCRATCH_BYTES" in err.value
    cfg = ll.make_config(shape, 16)
    with pytest.raises(ll.LLError) as e:
        ll.ll_decode_step_static(cfg, w, k, v, shape.vocab, 0, None)
    assert e.value.code == ll.LL_ERR_ARG
    with pytest.raises(ll.LLError) as e:
        ll.ll_decode_step_static(cfg, w, k, v, 1, 16, None)
    assert e.value.code == ll.LL_ERR_ARG
    assert ll.ll_decode_step_static(cfg, w, k, v, 1, 0, None) >= 0  # still works afterwards
