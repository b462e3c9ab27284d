"""Algorithmic bytes and flops of one batch-1 decode step (for roofline figures).

A decode step must stream every weight byte once: the layer matrices and norm
gains, the final gain, the LM head (the embedding matrix when tied) and one
embedding row. On top of that it reads the cached K and V of positions
0..pos-1 and writes K and V at pos. Logits are 4 bytes per vocabulary entry
when they are written out.
"""
from __future__ import annotations

from .synth import ModelShape


def weight_bytes(shape: ModelShape) -> int:
    per_layer = sum(_numel(s) for s in shape.layer_shapes().values())
    total = shape.n_layers * per_layer + shape.hidden            # + final norm gain
    total += shape.vocab * shape.hidden                          # LM head
    total += shape.hidden                                        # one embedding row
    return 2 * total


def kv_bytes(shape: ModelShape, pos: int) -> int:
    """K/V bytes of a step at ``pos``: read entries 0..pos-1, write entry pos."""
    per_pos = 2 * shape.n_layers * shape.n_kv_heads * shape.head_dim * 2
    return per_pos * (pos + 1)


def step_bytes(shape: ModelShape, pos: int, logits: bool = True) -> int:
    return weight_bytes(shape) + kv_bytes(shape, pos) + (4 * shape.vocab if logits else 0)


def batch_step_bytes(shape: ModelShape, pos: int, n: int, logits: bool = False) -> int:
    """One step of n sequences at ``pos`` sharing a pass over the weights: the
    weights once, and per sequence its K/V, its embedding row and its logits."""
    per_seq = kv_bytes(shape, pos) + 2 * shape.hidden + (4 * shape.vocab if logits else 0)
    return weight_bytes(shape) - 2 * shape.hidden + n * per_seq


def step_flops(shape: ModelShape, pos: int) -> int:
    """2 flops per weight element of the matrices plus 4*hd per (query head, position)."""
    mats = shape.n_layers * sum(_numel(s) for k, s in shape.layer_shapes().items()
                                if not k.endswith("norm"))
    mats += shape.vocab * shape.hidden
    attn = 4 * shape.n_layers * shape.n_q_heads * shape.head_dim * (pos + 1)
    return 2 * mats + attn


def layer_weight_elements(shape: ModelShape) -> int:
    """Elements of the layer matrices (every projection a prefill GEMM runs): the
    algorithmic flops of a prefill of n positions are 2 * n * this (its attention
    and the last position's LM head aside)."""
    return shape.n_layers * sum(_numel(s) for k, s in shape.layer_shapes().items() if not k.endswith("norm"))


def _numel(s) -> int:
    n = 1
    for d in s:
        n *= int(d)
    return n
