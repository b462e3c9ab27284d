"""Shared helpers of the GPU tests: model set-up through the C ABI and the parity
rule against the CPU oracle.

Parity rule (fp32 logits of the CUDA path vs the float oracle on the same bf16
weights and the same KV cache): max |delta| <= 2e-2 * max |logit| and relative L2
error <= 1e-2; the greedy token must equal the oracle's unless the oracle's top-2
margin is below 1e-2.
"""
from __future__ import annotations

import numpy as np

import oracle
from decode_megakernel_persistent_gb300 import ll, synth

TOL_MAX = 2e-2
TOL_L2 = 1e-2
MARGIN = 1e-2


def compare_logits(gpu, ref, what: str = ""):
    g = np.asarray(gpu, dtype=np.float64)
    r = np.asarray(ref, dtype=np.float64)
    assert g.shape == r.shape
    assert np.all(np.isfinite(g)), f"{what}: non-finite GPU logits"
    scale = float(np.max(np.abs(r)))
    maxd = float(np.max(np.abs(g - r)))
    rel = float(np.linalg.norm(g - r) / np.linalg.norm(r))
    assert maxd <= TOL_MAX * scale and rel <= TOL_L2, (
        f"{what}: max|d|={maxd:.3e} (limit {TOL_MAX * scale:.3e}) relL2={rel:.3e} (limit {TOL_L2})")
    return maxd / scale, rel


def top2_margin(ref) -> float:
    r = np.sort(np.asarray(ref, dtype=np.float64))
    return float(r[-1] - r[-2])


def check_token(gpu_tok: int, ref, what: str = ""):
    want = int(np.argmax(ref))  # numpy returns the lowest index among equal maxima
    if gpu_tok != want:
        assert top2_margin(ref) < MARGIN, f"{what}: token {gpu_tok} != oracle {want}, margin {top2_margin(ref):.3e}"


def widen_bits(b) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


class Pair:
    """The same model on the GPU (through the C ABI) and in the CPU oracle."""

    def __init__(self, shape, max_seq: int, backend=ll.LL_BACKEND_MEGAKERNEL, gain_jitter=0.0,
                 kv_fill: int = 0, seed: int = 0, prec: int = 32):
        import torch
        self.torch = torch
        self.shape = shape
        self.max_seq = max_seq
        self.w = synth.make_weights(shape, seed=seed, device="cuda", gain_jitter=gain_jitter)
        self.k, self.v = synth.make_kv(shape, max_seq, kv_fill, seed=2, device="cuda")
        self.dec = ll.Decoder(shape, self.w, self.k, self.v, max_seq, backend)
        self.orc = oracle.OracleModel(shape.as_dict(), synth.weights_to_host_bits(self.w), max_seq, prec=prec)
        if kv_fill:
            self.orc.k_cache[...] = synth.to_host_bits(self.k)
            self.orc.v_cache[...] = synth.to_host_bits(self.v)
        self.logits = torch.empty(shape.vocab, dtype=torch.float32, device="cuda")

    def step(self, token: int, pos: int, what: str = ""):
        nxt = self.dec.step(token, pos, self.logits)
        got = self.logits.cpu().numpy()
        ref, ref_next = self.orc.decode_step(token, pos)
        stats = compare_logits(got, ref, what or f"pos {pos}")
        check_token(nxt, ref, what or f"pos {pos}")
        return nxt, ref_next, stats

    def kv_close(self, positions):
        """GPU and oracle K/V entries at `positions` agree.

        Layer 0 sees identical inputs on both sides, so its entries may differ
        only where fp32 summation order tips a bf16 rounding (well under 1%).
        Deeper layers inherit the fp32 rounding noise of the layers below, and
        the random-weight models amplify it with depth: on the 1B shape the
        float and double oracles themselves differ by more than two bf16 steps
        in some deep-layer entries. So each layer is held to the bar the logits
        are held to: max |delta| <= TOL_MAX * max |oracle| and relative L2 <= TOL_L2.
        """
        gk = synth.to_host_bits(self.k)[:, :, positions]
        gv = synth.to_host_bits(self.v)[:, :, positions]
        ok = self.orc.k_cache[:, :, positions]
        ov = self.orc.v_cache[:, :, positions]
        for g, o, name in ((gk, ok, "K"), (gv, ov, "V")):
            a, b = widen_bits(g).astype(np.float64), widen_bits(o).astype(np.float64)
            for l in range(a.shape[0]):
                d = np.abs(a[l] - b[l])
                scale = max(float(np.max(np.abs(b[l]))), 1e-30)
                rel = float(np.linalg.norm(a[l] - b[l]) / max(np.linalg.norm(b[l]), 1e-30))
                assert np.max(d) <= TOL_MAX * scale and rel <= TOL_L2, (
                    f"{name} layer {l}: max|d|={np.max(d):.3e} (limit {TOL_MAX * scale:.3e}) relL2={rel:.3e}")
            assert np.mean(g[0] != o[0]) < 0.01, f"{name}: {np.mean(g[0] != o[0]):.4f} of layer-0 entries differ"

    def close(self):
        self.dec.close()
