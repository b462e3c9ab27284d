"""Seeded synthetic inputs: model shapes, bf16 weights, token streams, KV fills.

This module holds no arithmetic of the decode step; it only draws random
numbers. Both the CUDA path and the CPU oracle take their inputs from here.

Recipe:
  * weights: every matrix is bf16(0.02 * N(0, 1)) drawn in float32 from one
    torch generator seeded with ``seed`` (default 0), tensor by tensor in a
    fixed order (embed, then per layer attn_norm, wq, wk, wv, wo, mlp_norm,
    wg, wu, wd, then final_norm, lm_head); norm gains are 1.0 unless
    ``gain_jitter`` > 0 draws them as bf16(1 + gain_jitter * N(0, 1));
  * prompt / input tokens: uniform in [0, vocab) from a CPU generator, seed 1;
  * direct KV fills: bf16(N(0, 1)), seed 2.
"""
from __future__ import annotations

import dataclasses

import torch

LAYER_KEYS = ("attn_norm", "wq", "wk", "wv", "wo", "mlp_norm", "wg", "wu", "wd")


@dataclasses.dataclass(frozen=True)
class ModelShape:
    name: str
    n_layers: int
    hidden: int
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    inter: int
    vocab: int
    tied: bool
    rms_eps: float = 1e-5
    rope_theta: float = 500000.0

    def as_dict(self) -> dict:
        return dataclasses.asdict(self)

    @property
    def q_dim(self) -> int:
        return self.n_q_heads * self.head_dim

    @property
    def kv_dim(self) -> int:
        return self.n_kv_heads * self.head_dim

    def layer_shapes(self) -> dict:
        H, q, kv, I = self.hidden, self.q_dim, self.kv_dim, self.inter
        return {"attn_norm": (H,), "wq": (q, H), "wk": (kv, H), "wv": (kv, H),
                "wo": (H, q), "mlp_norm": (H,), "wg": (I, H), "wu": (I, H), "wd": (H, I)}


@dataclasses.dataclass(frozen=True)
class Workload:
    """A decode run: prompt/KV context length, greedy steps, and how KV is filled."""
    name: str
    shape: ModelShape
    context: int
    decode_steps: int
    kv_fill: str  # "prefill": run the prompt through the model; "normal": bf16 N(0,1)


TINY = ModelShape("tiny", 2, 256, 4, 2, 64, 1024, 4096, True)
LLAMA_1B = ModelShape("llama-3.2-1b", 16, 2048, 32, 8, 64, 8192, 128256, True)
LLAMA_3B = ModelShape("llama-3.2-3b", 28, 3072, 24, 8, 128, 8192, 128256, True)
LLAMA_8B = ModelShape("llama-3.1-8b", 32, 4096, 32, 8, 128, 14336, 128256, False)

WORKLOADS = {
    "tiny": Workload("tiny-2L-h256-ctx128", TINY, 128, 16, "prefill"),
    "1b": Workload("llama-3.2-1b-ctx1024", LLAMA_1B, 1024, 128, "prefill"),
    "1b-32k": Workload("llama-3.2-1b-ctx32768", LLAMA_1B, 32768, 64, "normal"),
    "3b": Workload("llama-3.2-3b-ctx2048", LLAMA_3B, 2048, 128, "prefill"),
    "8b": Workload("llama-3.1-8b-ctx8192", LLAMA_8B, 8192, 64, "prefill"),
}


def _normal_bf16(shape, gen, device, scale=1.0, offset=0.0) -> torch.Tensor:
    """bf16(offset + scale * N(0,1)), drawn in float32 in row chunks to bound memory."""
    out = torch.empty(shape, dtype=torch.bfloat16, device=device)
    flat = out.view(-1)
    chunk = 1 << 26
    for s in range(0, flat.numel(), chunk):
        n = min(chunk, flat.numel() - s)
        t = torch.randn(n, generator=gen, device=device, dtype=torch.float32)
        if scale != 1.0:
            t.mul_(scale)
        if offset != 0.0:
            t.add_(offset)
        flat[s:s + n].copy_(t)
    return out


def make_weights(shape: ModelShape, seed: int = 0, device="cpu", gain_jitter: float = 0.0,
                 std: float = 0.02) -> dict:
    """All weights of ``shape`` as bf16 tensors on ``device`` (see module recipe)."""
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    H, V = shape.hidden, shape.vocab

    def gain(n):
        if gain_jitter > 0:
            return _normal_bf16((n,), gen, device, gain_jitter, 1.0)
        return torch.ones(n, dtype=torch.bfloat16, device=device)

    w = {"embed": _normal_bf16((V, H), gen, device, std)}
    for k in LAYER_KEYS:
        w[k] = []
    ls = shape.layer_shapes()
    for _ in range(shape.n_layers):
        for k in LAYER_KEYS:
            if k.endswith("norm"):
                w[k].append(gain(ls[k][0]))
            else:
                w[k].append(_normal_bf16(ls[k], gen, device, std))
    w["final_norm"] = gain(H)
    w["lm_head"] = None if shape.tied else _normal_bf16((V, H), gen, device, std)
    return w


def make_tokens(vocab: int, n: int, seed: int = 1) -> list:
    """n token ids uniform in [0, vocab)."""
    gen = torch.Generator(device="cpu")
    gen.manual_seed(seed)
    return torch.randint(0, vocab, (n,), generator=gen).tolist()


def make_kv(shape: ModelShape, max_seq: int, n_fill: int, seed: int = 2, device="cpu"):
    """K and V caches [L, n_kv, max_seq, hd] bf16 whose first n_fill positions are N(0,1)."""
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    dims = (shape.n_layers, shape.n_kv_heads, max_seq, shape.head_dim)
    k = torch.zeros(dims, dtype=torch.bfloat16, device=device)
    v = torch.zeros(dims, dtype=torch.bfloat16, device=device)
    if n_fill > 0:
        fill = (shape.n_layers, shape.n_kv_heads, n_fill, shape.head_dim)
        k[:, :, :n_fill].copy_(_normal_bf16(fill, gen, device))
        v[:, :, :n_fill].copy_(_normal_bf16(fill, gen, device))
    return k, v


def to_host_bits(t: torch.Tensor):
    """bf16 tensor -> contiguous uint16 numpy array of its bit patterns (host copy)."""
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view("uint16")


def weights_to_host_bits(w: dict) -> dict:
    out = {}
    for k, v in w.items():
        if v is None:
            continue
        out[k] = [to_host_bits(t) for t in v] if isinstance(v, list) else to_host_bits(v)
    return out
