"""The algorithmic bytes behind bench.py's roofline figures, pinned to closed
forms written out here from the model shapes (not from the byte model's own
helpers), and to the page's figure for the 1B model.

The page "Hazy Research Llama-3.2-1B Megakernel" (its results paragraph) puts a
Llama-3.2-1B forward pass at about 2.48 GB of weights streamed.
"""
import pytest

from decode_megakernel_persistent_gb300 import bytemodel, synth


def layer_elems(h, q, kv, inter):
    # attn_norm, wq, wk, wv, wo, mlp_norm, wg, wu, wd
    return h + q * h + kv * h + kv * h + h * q + h + inter * h + inter * h + h * inter


def test_llama1b_weight_bytes_closed_form():
    per_layer = layer_elems(2048, 2048, 512, 8192)
    assert per_layer == 60_821_504
    elems = 16 * per_layer + 2048 + 128256 * 2048 + 2048  # + final gain, tied LM head, one embedding row
    assert bytemodel.weight_bytes(synth.LLAMA_1B) == 2 * elems == 2_471_632_896
    assert abs(2 * elems / 1e9 - 2.48) / 2.48 < 0.01  # the page's figure


def test_llama8b_untied_weight_bytes_closed_form():
    per_layer = layer_elems(4096, 4096, 1024, 14336)
    elems = 32 * per_layer + 4096 + 128256 * 4096 + 4096  # untied: the LM head, plus one embedding row
    assert bytemodel.weight_bytes(synth.LLAMA_8B) == 2 * elems == 15_009_857_536


@pytest.mark.parametrize("shape,per_pos", [(synth.LLAMA_1B, 2 * 16 * 8 * 64 * 2),
                                           (synth.LLAMA_3B, 2 * 28 * 8 * 128 * 2),
                                           (synth.LLAMA_8B, 2 * 32 * 8 * 128 * 2)])
def test_kv_bytes_read_then_written(shape, per_pos):
    # positions 0..pos-1 read, position pos written: pos + 1 entries of K and V
    assert bytemodel.kv_bytes(shape, 0) == per_pos
    assert bytemodel.kv_bytes(shape, 1100) == per_pos * 1101


def test_step_bytes_at_the_1b_benchmark_positions():
    # weights + K/V at pos 1100 + fp32 logits
    want = 2_471_632_896 + 32_768 * 1101 + 4 * 128256
    assert bytemodel.step_bytes(synth.LLAMA_1B, 1100) == want == 2_508_223_488
    assert bytemodel.step_bytes(synth.LLAMA_1B, 1100, logits=False) == want - 4 * 128256


def test_step_flops_two_per_matrix_weight():
    h, q, kv, inter, L, V = 2048, 2048, 512, 8192, 16, 128256
    mats = L * (q * h + 2 * kv * h + h * q + 3 * inter * h) + V * h
    attn = 4 * L * 32 * 64 * (1100 + 1)
    assert bytemodel.step_flops(synth.LLAMA_1B, 1100) == 2 * mats + attn


def test_batch_step_bytes_weights_once_kv_per_sequence():
    # n sequences: the weights (less the one embedding row) once, then each
    # sequence's K/V at pos 1100 and its own embedding row
    weights_wo_row = 2_471_632_896 - 2 * 2048
    for n in (1, 2, 8):
        want = weights_wo_row + n * (32_768 * 1101 + 2 * 2048)
        assert bytemodel.batch_step_bytes(synth.LLAMA_1B, 1100, n) == want
    assert bytemodel.batch_step_bytes(synth.LLAMA_1B, 1100, 1) == bytemodel.step_bytes(synth.LLAMA_1B, 1100, logits=False)
    assert (bytemodel.batch_step_bytes(synth.LLAMA_1B, 1100, 4, logits=True)
            - bytemodel.batch_step_bytes(synth.LLAMA_1B, 1100, 4)) == 4 * 4 * 128256
