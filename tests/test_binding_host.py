"""The Python binding's checks of the buffers a step writes or reads (no GPU):
the library takes raw device pointers and cannot see sizes, so a buffer that is
too small, of the wrong dtype or device, or strided must be refused before
anything is launched."""
import pytest
import torch

from decode_megakernel_persistent_gb300 import ll


class FakeCuda:
    """Stands in for a CUDA tensor (none exists on a CPU-only machine)."""

    def __init__(self, n, dtype=torch.float32, device="cuda:0", contiguous=True):
        self.is_cuda = True
        self.dtype = dtype
        self.device = torch.device(device)
        self._n = n
        self._c = contiguous

    def numel(self):
        return self._n

    def is_contiguous(self):
        return self._c


DEV = torch.device("cuda:0")


def refused(t, dtype=torch.float32, n=10, optional=True):
    with pytest.raises(ll.LLError) as e:
        ll._need(t, "buf", dtype, n, DEV, optional)
    assert e.value.code == ll.LL_ERR_ARG
    return str(e.value)


def test_accepts_a_fitting_buffer_and_optional_none():
    ll._need(FakeCuda(10), "buf", torch.float32, 10, DEV)
    ll._need(FakeCuda(11), "buf", torch.float32, 10, DEV)
    ll._need(None, "buf", torch.float32, 10, DEV)


def test_refuses_bad_buffers():
    assert "required" in refused(None, optional=False)
    assert "CUDA" in refused(torch.zeros(10))                       # host tensor
    assert "int32" in refused(FakeCuda(10), dtype=torch.int32)       # wrong dtype
    assert "cuda:1" in refused(FakeCuda(10, device="cuda:1"))        # other device
    assert "contiguous" in refused(FakeCuda(10, contiguous=False))
    assert "needs 10" in refused(FakeCuda(9))                        # one element short


def fake_model(shape, max_seq):
    H, V, I, L = shape.hidden, shape.vocab, shape.inter, shape.n_layers
    q, kv = shape.n_q_heads * shape.head_dim, shape.n_kv_heads * shape.head_dim
    bf = torch.bfloat16
    w = {"embed": FakeCuda(V * H, bf), "final_norm": FakeCuda(H, bf)}
    if not shape.tied:
        w["lm_head"] = FakeCuda(V * H, bf)
    per = {"attn_norm": H, "wq": q * H, "wk": kv * H, "wv": kv * H, "wo": H * q,
           "mlp_norm": H, "wg": I * H, "wu": I * H, "wd": H * I}
    for k, n in per.items():
        w[k] = [FakeCuda(n, bf) for _ in range(L)]
    cache = L * kv * max_seq
    return w, FakeCuda(cache, bf), FakeCuda(cache, bf)


@pytest.mark.parametrize("name", ["llama-3.2-1b", "llama-3.1-8b"])
def test_model_check_accepts_the_shapes(name):
    from decode_megakernel_persistent_gb300 import synth
    shape = {s.name: s for s in (synth.LLAMA_1B, synth.LLAMA_8B)}[name]
    w, k, v = fake_model(shape, 1100)
    ll.check_model(shape, w, k, v, 1100)


def test_model_check_refuses_misfits():
    from decode_megakernel_persistent_gb300 import synth
    shape = synth.LLAMA_8B  # untied: the LM head is checked too

    def refused(mutate, max_seq=64):
        w, k, v = fake_model(shape, 64)
        mutate(w, k, v)
        with pytest.raises(ll.LLError) as e:
            ll.check_model(shape, w, k, v, max_seq)
        assert e.value.code == ll.LL_ERR_ARG
        return str(e.value)

    bf = torch.bfloat16
    assert "wd[3]" in refused(lambda w, k, v: w["wd"].__setitem__(3, FakeCuda(shape.hidden * shape.inter - 1, bf)))
    assert "wo[0]" in refused(lambda w, k, v: w["wo"].__setitem__(0, FakeCuda(shape.hidden * 4096, torch.float16)))
    assert "lm_head" in refused(lambda w, k, v: w.pop("lm_head"))
    assert "one tensor per layer" in refused(lambda w, k, v: w["wq"].pop())
    assert "k_cache" in refused(lambda w, k, v: None, max_seq=65)  # caches sized for 64 positions


def _static_refused(mutate):
    from decode_megakernel_persistent_gb300 import synth
    shape = synth.TINY
    w, k, v = fake_model(shape, 16)
    logits = FakeCuda(shape.vocab)
    cfg = ll.make_config(shape, 16)
    w, k, v, logits = mutate(w, k, v, logits)
    with pytest.raises(ll.LLError) as e:
        ll.check_static_args(cfg, w, k, v, logits)
    assert e.value.code == ll.LL_ERR_ARG
    return str(e.value)


def test_static_step_args_refuse_misfits():
    # a short per-layer list would make the C side read past its host array
    assert "one tensor per layer" in _static_refused(lambda w, k, v, lg: (dict(w, wg=w["wg"][:1]), k, v, lg))
    # an undersized logits buffer or cache would take out-of-bounds device writes
    assert "logits" in _static_refused(lambda w, k, v, lg: (w, k, v, FakeCuda(4095)))
    assert "k_cache" in _static_refused(lambda w, k, v, lg: (w, FakeCuda(k.numel() - 1, torch.bfloat16), v, lg))
    assert "v_cache" in _static_refused(lambda w, k, v, lg: (w, k, FakeCuda(v.numel(), torch.float16), lg))
    assert "wq[1]" in _static_refused(
        lambda w, k, v, lg: (dict(w, wq=[w["wq"][0], FakeCuda(10, torch.bfloat16)]), k, v, lg))
    assert "cuda:1" in _static_refused(lambda w, k, v, lg: (w, k, v, FakeCuda(4096, device="cuda:1")))
