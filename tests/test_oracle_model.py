"""Pins of the oracle's whole decode step (no GPU).

Each test picks weights for which the decode step reduces to a closed form
(a layer that is the identity, attention over one entry, a diagonal MLP, a
rotation) and checks the oracle's logits and KV-cache writes against it. The
special cases are chosen so that swapped gate/up roles, a transposed
projection, a wrong GQA head mapping, a gain taken from the wrong norm, a
missing residual add or RoPE left off q or k each fail one of them.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from decode_megakernel_persistent_gb300 import synth


def bits(x) -> np.ndarray:
    t = torch.as_tensor(np.asarray(x, dtype=np.float64)).to(torch.float32).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def widen(b) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def small_model(L=1, H=32, nq=4, nkv=2, hd=8, I=48, V=61, tied=True, std=0.2, seed=0,
                theta=10000.0, eps=1e-5):
    rng = np.random.default_rng(seed)
    cfg = dict(n_layers=L, hidden=H, n_q_heads=nq, n_kv_heads=nkv, head_dim=hd, inter=I,
               vocab=V, tied=tied, rms_eps=eps, rope_theta=theta)
    w = {"embed": bits(rng.standard_normal((V, H)) * std),
         "final_norm": bits(1 + 0.3 * rng.standard_normal(H))}
    if not tied:
        w["lm_head"] = bits(rng.standard_normal((V, H)) * std)
    shapes = {"attn_norm": (H,), "wq": (nq * hd, H), "wk": (nkv * hd, H), "wv": (nkv * hd, H),
              "wo": (H, nq * hd), "mlp_norm": (H,), "wg": (I, H), "wu": (I, H), "wd": (H, I)}
    for k, s in shapes.items():
        if k.endswith("norm"):
            w[k] = [bits(1 + 0.3 * rng.standard_normal(s)) for _ in range(L)]
        else:
            w[k] = [bits(rng.standard_normal(s) * std) for _ in range(L)]
    return cfg, w


def rms(x, g, eps):
    return x / math.sqrt(np.mean(x * x) + eps) * widen(g)


def head_logits(cfg, w, x):
    lm = w["embed"] if cfg["tied"] else w["lm_head"]
    return widen(lm) @ rms(x, w["final_norm"], cfg["rms_eps"])


def rope_np(x, pos, theta):
    hd = x.size
    z = (x[: hd // 2] + 1j * x[hd // 2:]) * np.exp(1j * pos * theta ** (-2.0 * np.arange(hd // 2) / hd))
    return np.concatenate([z.real, z.imag])


def run(cfg, w, token, pos, prec=64, max_seq=32, kv=None):
    m = oracle.OracleModel(cfg, w, max_seq=max_seq, prec=prec)
    if kv is not None:
        m.k_cache[...] = kv[0]
        m.v_cache[...] = kv[1]
    logits, nxt = m.decode_step(token, pos)
    return m, logits.astype(np.float64), nxt


def tol(prec):
    return dict(rtol=1e-4, atol=1e-4) if prec == 32 else dict(rtol=1e-10, atol=1e-10)


@pytest.mark.parametrize("prec", (32, 64))
@pytest.mark.parametrize("tied", (True, False))
def test_zero_layers_is_norm_then_head(prec, tied):
    cfg, w = small_model(L=0, tied=tied)
    t = 17
    _, logits, nxt = run(cfg, w, t, 0, prec)
    want = head_logits(cfg, w, widen(w["embed"][t]))
    np.testing.assert_allclose(logits, want, **tol(prec))
    assert nxt == int(np.argmax(want))


@pytest.mark.parametrize("prec", (32, 64))
def test_tied_head_argmax_is_input_token(prec):
    # tied head, unit gains: logit_i = r * <e_i, e_t>, largest at i = t when rows are
    # much longer than their mutual overlaps
    cfg, w = small_model(L=0, V=50, H=256)
    w["final_norm"] = bits(np.ones(256))
    e = widen(w["embed"])
    t = 31
    _, logits, nxt = run(cfg, w, t, 0, prec)
    r = 1.0 / math.sqrt(np.mean(e[t] ** 2) + cfg["rms_eps"])
    assert abs(logits[t] - r * np.dot(e[t], e[t])) < 1e-3 * abs(logits[t])
    assert nxt == t


@pytest.mark.parametrize("prec", (32, 64))
def test_zero_output_projections_make_layers_identity(prec):
    cfg, w = small_model(L=3)
    for l in range(3):
        w["wo"][l] = bits(np.zeros_like(widen(w["wo"][l])))
        w["wd"][l] = bits(np.zeros_like(widen(w["wd"][l])))
    t, pos = 5, 4
    m, logits, _ = run(cfg, w, t, pos, prec)
    np.testing.assert_allclose(logits, head_logits(cfg, w, widen(w["embed"][t])), **tol(prec))
    # every layer still wrote its k, v at pos and nowhere else
    for l in range(3):
        assert np.any(m.k_cache[l, :, pos] != 0) and np.any(m.v_cache[l, :, pos] != 0)
    assert not np.any(m.k_cache[:, :, :pos]) and not np.any(m.k_cache[:, :, pos + 1:])


@pytest.mark.parametrize("prec", (32, 64))
def test_position_zero_attention_block(prec):
    # At pos 0 each query head attends to one entry, so attention returns the new v of
    # its KV head: x1 = e + Wo * expand(bf16(Wv * rmsnorm(e, attn_norm))). The MLP is
    # switched off with Wd = 0. Heads 0,1 read KV head 0 and heads 2,3 read KV head 1.
    cfg, w = small_model(L=1)
    w["wd"][0] = bits(np.zeros_like(widen(w["wd"][0])))
    t = 9
    e = widen(w["embed"][t])
    h = rms(e, w["attn_norm"][0], cfg["rms_eps"])
    v = widen(bits(widen(w["wv"][0]) @ h))
    G, hd = cfg["n_q_heads"] // cfg["n_kv_heads"], cfg["head_dim"]
    o = np.concatenate([v[(qh // G) * hd:(qh // G + 1) * hd] for qh in range(cfg["n_q_heads"])])
    x1 = e + widen(w["wo"][0]) @ o
    _, logits, _ = run(cfg, w, t, 0, prec)
    np.testing.assert_allclose(logits, head_logits(cfg, w, x1), rtol=2e-3, atol=2e-3)


@pytest.mark.parametrize("prec", (32, 64))
def test_mlp_with_permuted_diagonal_weights(prec):
    # Attention off (Wo = 0); gate, up and down are permuted diagonals, so
    # x1[pd[c]] = e[pd[c]] + d_c * silu(a_c h[pg[c]]) * b_c h[pu[c]], h = rmsnorm(e, mlp_norm).
    H = I = 32
    cfg, w = small_model(L=1, H=H, I=I)
    rng = np.random.default_rng(11)
    pg, pu, pd = rng.permutation(I), rng.permutation(I), rng.permutation(H)
    a = widen(bits(rng.uniform(0.5, 3.0, I)))
    b = widen(bits(rng.uniform(-2.0, 2.0, I)))
    d = widen(bits(rng.uniform(-1.0, 1.0, H)))
    wg, wu, wd = np.zeros((I, H)), np.zeros((I, H)), np.zeros((H, I))
    wg[np.arange(I), pg] = a
    wu[np.arange(I), pu] = b
    wd[pd, np.arange(I)] = d
    w["wg"][0], w["wu"][0], w["wd"][0] = bits(wg), bits(wu), bits(wd)
    w["wo"][0] = bits(np.zeros((H, cfg["n_q_heads"] * cfg["head_dim"])))
    t = 23
    e = widen(w["embed"][t])
    hm = rms(e, w["mlp_norm"][0], cfg["rms_eps"])
    z = a * hm[pg]
    act = z / (1 + np.exp(-z)) * (b * hm[pu])
    x1 = e.copy()
    x1[pd] += d * act
    _, logits, _ = run(cfg, w, t, 3, prec)
    np.testing.assert_allclose(logits, head_logits(cfg, w, x1), **tol(prec))


@pytest.mark.parametrize("prec", (32, 64))
def test_kv_cache_write_is_rotated_k_and_plain_v(prec):
    cfg, w = small_model(L=2)
    t, pos = 14, 6
    m, _, _ = run(cfg, w, t, pos, prec)
    e = widen(w["embed"][t])
    h = rms(e, w["attn_norm"][0], cfg["rms_eps"])
    k = widen(w["wk"][0]) @ h
    v = widen(w["wv"][0]) @ h
    hd = cfg["head_dim"]
    for g in range(cfg["n_kv_heads"]):
        kr = rope_np(k[g * hd:(g + 1) * hd], pos, cfg["rope_theta"])
        np.testing.assert_allclose(widen(m.k_cache[0, g, pos]), kr, rtol=1e-2, atol=1e-2)
        np.testing.assert_allclose(widen(m.v_cache[0, g, pos]), v[g * hd:(g + 1) * hd], rtol=1e-2, atol=1e-2)


@pytest.mark.parametrize("prec", (32, 64))
@pytest.mark.parametrize("pos", (1, 5, 17))
def test_self_score_does_not_depend_on_position(prec, pos):
    # Cache entries 0..pos-1 are zero, so each query head puts weight
    # exp(s) / (exp(s) + pos) on its new v, where s = <R_pos q, R_pos k> / sqrt(hd)
    # = <q, k> / sqrt(hd) whatever pos is. RoPE left off q or off k breaks that.
    cfg, w = small_model(L=1, std=0.3)
    w["wd"][0] = bits(np.zeros_like(widen(w["wd"][0])))
    t = 2
    e = widen(w["embed"][t])
    h = rms(e, w["attn_norm"][0], cfg["rms_eps"])
    q, k = widen(w["wq"][0]) @ h, widen(w["wk"][0]) @ h
    v = widen(bits(widen(w["wv"][0]) @ h))
    G, hd = cfg["n_q_heads"] // cfg["n_kv_heads"], cfg["head_dim"]
    o = []
    for qh in range(cfg["n_q_heads"]):
        g = qh // G
        s = np.dot(q[qh * hd:(qh + 1) * hd], k[g * hd:(g + 1) * hd]) / math.sqrt(hd)
        o.append(v[g * hd:(g + 1) * hd] * (math.exp(s) / (math.exp(s) + pos)))
    x1 = e + widen(w["wo"][0]) @ np.concatenate(o)
    _, logits, _ = run(cfg, w, t, pos, prec)
    np.testing.assert_allclose(logits, head_logits(cfg, w, x1), rtol=1e-2, atol=1e-2)


@pytest.mark.parametrize("prec", (32, 64))
def test_entries_after_pos_are_not_read(prec):
    cfg, w = small_model(L=2)
    rng = np.random.default_rng(12)
    shape = (2, cfg["n_kv_heads"], 32, cfg["head_dim"])
    k = bits(rng.standard_normal(shape))
    v = bits(rng.standard_normal(shape))
    pos = 10
    _, l1, _ = run(cfg, w, 3, pos, prec, kv=(k, v))
    k2, v2 = k.copy(), v.copy()
    k2[:, :, pos + 1:] = bits(rng.standard_normal(k2[:, :, pos + 1:].shape) * 9)
    v2[:, :, pos + 1:] = bits(rng.standard_normal(v2[:, :, pos + 1:].shape) * 9)
    _, l2, _ = run(cfg, w, 3, pos, prec, kv=(k2, v2))
    np.testing.assert_array_equal(l1, l2)
    # entries before pos are read
    k3 = k.copy()
    k3[:, :, 4] = bits(rng.standard_normal(k3[:, :, 4].shape) * 9)
    _, l3, _ = run(cfg, w, 3, pos, prec, kv=(k3, v))
    assert np.max(np.abs(l3 - l1)) > 1e-4


def test_float_and_double_agree_on_tiny_workload():
    shape = synth.TINY
    w = synth.weights_to_host_bits(synth.make_weights(shape, seed=0, device="cpu"))
    cfg = shape.as_dict()
    toks = synth.make_tokens(shape.vocab, 12, seed=1)
    m32 = oracle.OracleModel(cfg, w, max_seq=16, prec=32)
    m64 = oracle.OracleModel(cfg, w, max_seq=16, prec=64)
    for pos, t in enumerate(toks):
        l32, n32 = m32.decode_step(t, pos)
        l64, n64 = m64.decode_step(t, pos)
        scale = np.max(np.abs(l64))
        assert np.max(np.abs(l32 - l64)) <= 1e-4 * scale
        top2 = np.sort(l64)[-2:]
        if top2[1] - top2[0] > 1e-3:
            assert n32 == n64


def test_bad_arguments_rejected():
    cfg, w = small_model(L=1)
    m = oracle.OracleModel(cfg, w, max_seq=8, prec=32)
    with pytest.raises(ValueError):
        m.decode_step(cfg["vocab"], 0)
    with pytest.raises(ValueError):
        m.decode_step(0, 8)


def test_results_do_not_depend_on_thread_count():
    # each output row is summed by one thread, left to right, so the oracle's
    # logits and cache are bit-identical on one thread and on several
    shape = synth.TINY
    w = synth.weights_to_host_bits(synth.make_weights(shape, seed=2, device="cpu"))
    cfg = shape.as_dict()
    toks = synth.make_tokens(shape.vocab, 6, seed=3)
    before = oracle.num_threads()
    out = []
    try:
        for n in (1, max(2, before)):
            oracle.set_threads(n)
            assert oracle.num_threads() == n
            m = oracle.OracleModel(cfg, w, max_seq=8, prec=32)
            logs = [m.decode_step(t, pos)[0].copy() for pos, t in enumerate(toks)]
            out.append((np.stack(logs), m.k_cache.copy(), m.v_cache.copy()))
    finally:
        oracle.set_threads(before)
    for a, b in zip(out[0], out[1]):
        np.testing.assert_array_equal(a, b)
