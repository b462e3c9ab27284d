"""The seeded synthetic inputs (no GPU) follow their stated recipe: bf16
matrices of 0.02 * N(0, 1), unit norm gains (or 1 + jitter * N(0, 1)), tokens
uniform in [0, vocab), K/V fills of N(0, 1) with zeros past the fill, the same
bits for the same seed and other bits for another."""
import numpy as np
import torch

from decode_megakernel_persistent_gb300 import synth

SH = synth.ModelShape("recipe", 2, 512, 8, 2, 64, 1536, 4096, False)


def f64(t):
    return t.float().double().numpy()


def test_weight_shapes_dtypes_and_statistics():
    w = synth.make_weights(SH, seed=0)
    H, V, I = SH.hidden, SH.vocab, SH.inter
    q, kv = SH.n_q_heads * SH.head_dim, SH.n_kv_heads * SH.head_dim
    want = {"wq": (q, H), "wk": (kv, H), "wv": (kv, H), "wo": (H, q), "wg": (I, H), "wu": (I, H), "wd": (H, I)}
    assert tuple(w["embed"].shape) == (V, H) and tuple(w["lm_head"].shape) == (V, H)
    mats = [w["embed"], w["lm_head"]]
    for k, s in want.items():
        assert len(w[k]) == SH.n_layers
        for t in w[k]:
            assert t.dtype == torch.bfloat16 and tuple(t.shape) == s
            mats.append(t)
    allv = np.concatenate([f64(t).ravel() for t in mats])
    assert abs(allv.std() / 0.02 - 1) < 0.01 and abs(allv.mean()) < 1e-4
    for k in ("attn_norm", "mlp_norm"):
        for t in w[k]:
            assert np.all(f64(t) == 1.0)
    assert np.all(f64(w["final_norm"]) == 1.0)


def test_gain_jitter_and_tied_head():
    w = synth.make_weights(SH, seed=0, gain_jitter=0.25)
    g = np.concatenate([f64(t) for t in w["attn_norm"] + w["mlp_norm"]] + [f64(w["final_norm"])])
    assert abs(g.mean() - 1) < 0.03 and abs(g.std() / 0.25 - 1) < 0.1
    tied = synth.make_weights(synth.TINY, seed=0)
    assert tied["lm_head"] is None


def test_same_seed_same_bits_other_seed_other_bits():
    a = synth.weights_to_host_bits(synth.make_weights(synth.TINY, seed=0))
    b = synth.weights_to_host_bits(synth.make_weights(synth.TINY, seed=0))
    c = synth.weights_to_host_bits(synth.make_weights(synth.TINY, seed=1))
    for k in a:
        if a[k] is None:
            continue
        if isinstance(a[k], list):
            for x, y, z in zip(a[k], b[k], c[k]):
                np.testing.assert_array_equal(x, y)
                if k not in ("attn_norm", "mlp_norm"):
                    assert np.any(x != z)
        else:
            np.testing.assert_array_equal(a[k], b[k])
    assert synth.make_tokens(4096, 64, seed=1) == synth.make_tokens(4096, 64, seed=1)
    assert synth.make_tokens(4096, 64, seed=1) != synth.make_tokens(4096, 64, seed=2)


def test_tokens_and_kv_fill():
    toks = np.array(synth.make_tokens(SH.vocab, 20000, seed=1))
    assert toks.min() >= 0 and toks.max() < SH.vocab
    assert abs(toks.mean() / ((SH.vocab - 1) / 2) - 1) < 0.02
    k, v = synth.make_kv(SH, 96, 64, seed=2)
    assert tuple(k.shape) == (SH.n_layers, SH.n_kv_heads, 96, SH.head_dim) and k.dtype == torch.bfloat16
    for t in (k, v):
        fill = f64(t[:, :, :64])
        assert abs(fill.std() - 1) < 0.02 and abs(fill.mean()) < 0.02
        assert np.all(f64(t[:, :, 64:]) == 0)
    assert np.any(f64(k[:, :, :64]) != f64(v[:, :, :64]))
