"""The oracle's double build against a second, independently written float64
forward pass in numpy (no GPU).

The numpy forward below is written from the decode step's instruction list on
the page "Hazy Research Llama-3.2-1B Megakernel" (RMSNorm + QKV + RoPE,
attention over the cache, O projection + residual, RMSNorm + SiLU-gated MLP +
down projection + residual, final RMSNorm + LM head), in matrix form: BLAS
matrix products instead of the oracle's left-to-right loops, RoPE as a complex
multiplication instead of the rotate-half formulas, softmax over whole score
vectors per head group. It shares nothing with oracle.c but the bf16 bit
patterns of the weights, so a structural slip in the oracle that its float and
double builds would share (a dropped term, a wrong head mapping, a transposed
operand) shows up here as a difference far above float64 rounding.
"""
import numpy as np
import pytest
import torch

import oracle


def bits(x) -> np.ndarray:
    t = torch.as_tensor(np.asarray(x, dtype=np.float64)).to(torch.float32).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def widen(b) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def bf16_rne(x: np.ndarray) -> np.ndarray:
    """float64 -> bf16 bits, rounding the double straight to 8 significant bits,
    ties to even (normal range; the models here stay far from subnormals)."""
    m, e = np.frexp(np.asarray(x, dtype=np.float64))
    r = np.ldexp(np.rint(np.ldexp(m, 8)), e - 8)
    return (r.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)


def make_model(L, H, nq, nkv, hd, I, V, tied, seed):
    rng = np.random.default_rng(seed)
    cfg = dict(n_layers=L, hidden=H, n_q_heads=nq, n_kv_heads=nkv, head_dim=hd, inter=I, vocab=V,
               tied=tied, rms_eps=1e-5, rope_theta=10000.0)
    w = {"embed": bits(rng.standard_normal((V, H)) * 0.3),
         "final_norm": bits(1 + 0.3 * rng.standard_normal(H))}
    if not tied:
        w["lm_head"] = bits(rng.standard_normal((V, H)) * 0.3)
    shapes = {"attn_norm": (H,), "wq": (nq * hd, H), "wk": (nkv * hd, H), "wv": (nkv * hd, H),
              "wo": (H, nq * hd), "mlp_norm": (H,), "wg": (I, H), "wu": (I, H), "wd": (H, I)}
    for k, s in shapes.items():
        if k.endswith("norm"):
            w[k] = [bits(1 + 0.3 * rng.standard_normal(s)) for _ in range(L)]
        else:
            w[k] = [bits(rng.standard_normal(s) * 0.3) for _ in range(L)]
    return cfg, w


class NumpyForward:
    """float64 decode steps with a bf16 KV cache of its own."""

    def __init__(self, cfg, w, max_seq):
        self.c = cfg
        self.w = {k: ([widen(t) for t in v] if isinstance(v, list) else widen(v)) for k, v in w.items()}
        L, nkv, hd = cfg["n_layers"], cfg["n_kv_heads"], cfg["head_dim"]
        self.kc = np.zeros((L, nkv, max_seq, hd), dtype=np.uint16)
        self.vc = np.zeros_like(self.kc)

    def _norm(self, x, g):
        return x / np.sqrt(np.mean(x * x) + self.c["rms_eps"]) * g

    def _rope(self, heads, pos):
        # heads [n, hd]: dims (i, i + hd/2) as the complex number x_i + j x_{i+hd/2},
        # turned by pos * theta^(-2i/hd)
        hd = heads.shape[1]
        half = hd // 2
        ang = pos * self.c["rope_theta"] ** (-2.0 * np.arange(half) / hd)
        z = (heads[:, :half] + 1j * heads[:, half:]) * np.exp(1j * ang)
        return np.concatenate([z.real, z.imag], axis=1)

    def step(self, token, pos):
        c, w = self.c, self.w
        nq, nkv, hd = c["n_q_heads"], c["n_kv_heads"], c["head_dim"]
        grp = nq // nkv
        x = w["embed"][token].copy()
        for l in range(c["n_layers"]):
            h = self._norm(x, w["attn_norm"][l])
            q = self._rope((w["wq"][l] @ h).reshape(nq, hd), pos)
            k = self._rope((w["wk"][l] @ h).reshape(nkv, hd), pos)
            v = (w["wv"][l] @ h).reshape(nkv, hd)
            self.kc[l, :, pos] = bf16_rne(k)
            self.vc[l, :, pos] = bf16_rne(v)
            K = widen(self.kc[l, :, :pos + 1])  # [nkv, pos+1, hd]
            Vv = widen(self.vc[l, :, :pos + 1])
            o = np.empty((nq, hd))
            for g in range(nkv):
                qs = q[g * grp:(g + 1) * grp]                       # the group's query heads
                s = qs @ K[g].T / np.sqrt(hd)                       # [grp, pos+1]
                p = np.exp(s - s.max(axis=1, keepdims=True))
                o[g * grp:(g + 1) * grp] = (p / p.sum(axis=1, keepdims=True)) @ Vv[g]
            x = x + w["wo"][l] @ o.reshape(-1)
            h = self._norm(x, w["mlp_norm"][l])
            gate, up = w["wg"][l] @ h, w["wu"][l] @ h
            x = x + w["wd"][l] @ (gate / (1.0 + np.exp(-gate)) * up)
        head = w["embed"] if c["tied"] else w["lm_head"]
        return head @ self._norm(x, w["final_norm"])


@pytest.mark.parametrize("L,H,nq,nkv,hd,I,V,tied", [
    (2, 64, 4, 2, 16, 96, 101, True),    # GQA 2:1
    (2, 48, 6, 1, 8, 80, 67, False),     # all query heads on one KV head, untied head
    (1, 32, 2, 2, 16, 64, 53, True),     # plain multi-head
])
def test_oracle_fp64_matches_numpy_forward(L, H, nq, nkv, hd, I, V, tied):
    cfg, w = make_model(L, H, nq, nkv, hd, I, V, tied, seed=L * 100 + H)
    max_seq = 9
    orc = oracle.OracleModel(cfg, w, max_seq, prec=64)
    ref = NumpyForward(cfg, w, max_seq)
    rng = np.random.default_rng(5)
    tok = int(rng.integers(V))
    for pos in range(max_seq):
        got, nxt = orc.decode_step(tok, pos)
        want = ref.step(tok, pos)
        scale = np.max(np.abs(want))
        assert np.max(np.abs(got - want)) <= 1e-12 * scale, f"pos {pos}: {np.max(np.abs(got - want)) / scale:.3e}"
        assert nxt == int(np.argmax(want))
        np.testing.assert_array_equal(orc.k_cache[:, :, :pos + 1], ref.kc[:, :, :pos + 1])
        np.testing.assert_array_equal(orc.v_cache[:, :, :pos + 1], ref.vc[:, :, :pos + 1])
        tok = nxt if pos % 2 else int(rng.integers(V))  # greedy and fresh tokens alternate


def test_numpy_forward_catches_a_planted_head_mapping_slip():
    # the comparison has teeth: a forward whose query heads read the wrong KV
    # head (interleaved instead of contiguous groups) differs far above 1e-12
    cfg, w = make_model(1, 64, 4, 2, 16, 96, 101, True, seed=3)
    orc = oracle.OracleModel(cfg, w, 4, prec=64)
    ref = NumpyForward(cfg, w, 4)
    orig = ref.step

    def slipped(token, pos):
        c = ref.c
        saved = ref.w["wq"][0].copy()
        hd, nq = c["head_dim"], c["n_q_heads"]
        perm = np.concatenate([np.arange(h * hd, (h + 1) * hd) for h in (0, 2, 1, 3)])
        ref.w["wq"][0] = saved[perm]
        try:
            return orig(token, pos)
        finally:
            ref.w["wq"][0] = saved

    worst = 0.0
    for pos in range(4):
        got, _ = orc.decode_step(7 + pos, pos)
        want = slipped(7 + pos, pos)
        worst = max(worst, np.max(np.abs(got - want)) / np.max(np.abs(want)))
    assert worst > 1e-6
