"""Pins of the CPU oracle's primitives against closed forms, invariants and
library routines (no GPU). Each test is built so that a plausible slip in the
oracle (a dropped term, a wrong sign or index, a transposed operand, a missing
scale) fails it."""
import math
import os

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
PRECS = (32, 64)


def bits(x) -> np.ndarray:
    """float array -> bf16 bit patterns, rounded by torch (round to nearest even)."""
    t = torch.as_tensor(np.asarray(x, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def widen(b) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint32) << 16).view(np.float32).astype(np.float64)


# ---- bf16 conversions ---------------------------------------------------------

def test_to_bf16_matches_torch_rounding():
    rng = np.random.default_rng(0)
    x = rng.standard_normal(4000).astype(np.float32) * np.float32(3.0)
    # exact ties between two bf16 neighbours: low 16 bits 0x8000
    ties = (rng.integers(0x3000, 0x4800, 200, dtype=np.uint32) << 16) | 0x8000
    x = np.concatenate([x, ties.view(np.float32), np.float32([0.0, -0.0, 1.0, -2.5])])
    want = bits(x)
    for p in PRECS:
        got = oracle.to_bf16(x.astype(np.float64) if p == 64 else x, prec=p)
        np.testing.assert_array_equal(got, want)


def test_to_bf16_double_rounds_once():
    # 1 + 2^-8 + 2^-30 lies just above the midpoint of 1 and 1 + 2^-7, so a single
    # rounding gives 1 + 2^-7 (0x3F81); rounding through float first would give 1.0.
    x = 1.0 + 2.0 ** -8 + 2.0 ** -30
    assert int(oracle.to_bf16([x], prec=64)[0]) == 0x3F81
    assert int(oracle.to_bf16([1.0 + 2.0 ** -8], prec=64)[0]) == 0x3F80  # exact tie: even


def test_from_bf16_exact():
    b = np.array([0x3F80, 0xBF80, 0x4049, 0x0000, 0x8000, 0x3C23, 0x7F7F], dtype=np.uint16)
    for p in PRECS:
        np.testing.assert_array_equal(oracle.from_bf16(b, prec=p), widen(b))


# ---- RMSNorm ------------------------------------------------------------------

@pytest.mark.parametrize("p", PRECS)
def test_rmsnorm_unit_rms_closed_form(p):
    rng = np.random.default_rng(1)
    x = rng.standard_normal(257) * 3.0
    eps = 1e-5
    out = oracle.rmsnorm(x, bits(np.ones(257)), eps, prec=p)
    ms = np.mean(x ** 2)
    want_rms = math.sqrt(ms / (ms + eps))
    assert abs(math.sqrt(np.mean(out.astype(np.float64) ** 2)) - want_rms) < (1e-6 if p == 32 else 1e-13)
    # direction is x's
    np.testing.assert_allclose(out, x / math.sqrt(ms + eps), rtol=1e-6 if p == 32 else 1e-13)


@pytest.mark.parametrize("p", PRECS)
def test_rmsnorm_scale_invariant_and_gain_elementwise(p):
    rng = np.random.default_rng(2)
    x = rng.standard_normal(64)
    g = np.ones(64)
    a = oracle.rmsnorm(x, bits(g), 0.0, prec=p)
    b = oracle.rmsnorm(x * 7.25, bits(g), 0.0, prec=p)
    np.testing.assert_allclose(a, b, rtol=1e-5 if p == 32 else 1e-12)
    g2 = np.zeros(64)
    g2[3], g2[10] = 2.0, -0.5
    c = oracle.rmsnorm(x, bits(g2), 0.0, prec=p)
    want = np.zeros(64)
    want[3], want[10] = 2.0 * a[3], -0.5 * a[10]
    np.testing.assert_allclose(c, want, rtol=1e-6 if p == 32 else 1e-13, atol=0)


# ---- matrix-vector product ------------------------------------------------------

@pytest.mark.parametrize("p", PRECS)
def test_matvec_identity_onehot_and_library(p):
    rng = np.random.default_rng(3)
    x = rng.standard_normal(48)
    eye = bits(np.eye(48))
    np.testing.assert_array_equal(oracle.matvec(eye, x, prec=p), x.astype(oracle._dtype(p)))
    w = np.zeros((5, 48))
    w[0, 7] = 1.0
    w[3, 47] = -2.0
    y = oracle.matvec(bits(w), x, prec=p)
    np.testing.assert_allclose(y, [x[7], 0, 0, -2 * x[47], 0], rtol=1e-7)
    # a non-square product against numpy's matmul on the widened weights: catches a
    # transposed operand or a wrong row stride
    wb = bits(rng.standard_normal((37, 48)) * 0.1)
    got = oracle.matvec(wb, x, prec=p)
    want = widen(wb) @ x.astype(oracle._dtype(p)).astype(np.float64)
    np.testing.assert_allclose(got, want, rtol=1e-5 if p == 32 else 1e-12, atol=1e-6 if p == 32 else 1e-13)


# ---- RoPE -------------------------------------------------------------------------

def _golden_rope():
    rows, cur = [], None
    with open(os.path.join(GOLDEN, "rope_hd4_pos1_theta10000.txt")) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            tag, *vals = line.split()
            if tag == "in":
                cur = [float(v) for v in vals]
            else:
                rows.append((cur, [float(v) for v in vals]))
    return rows


@pytest.mark.parametrize("p", PRECS)
def test_rope_worked_example(p):
    for x, y in _golden_rope():
        got = oracle.rope(x, pos=1, theta=10000.0, prec=p)
        np.testing.assert_allclose(got, y, rtol=0, atol=1e-6 if p == 32 else 1e-14)


@pytest.mark.parametrize("p", PRECS)
def test_rope_identity_norm_and_relative_position(p):
    rng = np.random.default_rng(4)
    hd, theta = 64, 500000.0
    q = rng.standard_normal(hd)
    k = rng.standard_normal(hd)
    tol = 1e-4 if p == 32 else 1e-11
    np.testing.assert_array_equal(oracle.rope(q, 0, theta, prec=p), q.astype(oracle._dtype(p)))
    r = oracle.rope(q, 77, theta, prec=p).astype(np.float64)
    # each (i, i + hd/2) pair keeps its length
    np.testing.assert_allclose(r[:32] ** 2 + r[32:] ** 2, q[:32] ** 2 + q[32:] ** 2, rtol=tol * 10)
    # <R_a q, R_b k> depends only on a - b
    d1 = np.dot(oracle.rope(q, 40, theta, prec=p), oracle.rope(k, 13, theta, prec=p))
    d2 = np.dot(oracle.rope(q, 1027, theta, prec=p), oracle.rope(k, 1000, theta, prec=p))
    assert abs(d1 - d2) < tol * 50


@pytest.mark.parametrize("p", PRECS)
def test_rope_equals_complex_rotation(p):
    # The rotate-half pairing is multiplication of z_i = x_i + i x_{i+hd/2} by
    # exp(i * pos * theta^(-2i/hd)).
    rng = np.random.default_rng(5)
    hd, pos, theta = 128, 513, 500000.0
    x = rng.standard_normal(hd)
    z = (x[: hd // 2] + 1j * x[hd // 2:]) * np.exp(1j * pos * theta ** (-2.0 * np.arange(hd // 2) / hd))
    got = oracle.rope(x, pos, theta, prec=p)
    np.testing.assert_allclose(got, np.concatenate([z.real, z.imag]), atol=1e-5 if p == 32 else 1e-12)


# ---- SiLU ---------------------------------------------------------------------------

@pytest.mark.parametrize("p", PRECS)
def test_silu_closed_forms(p):
    tol = 1e-7 if p == 32 else 1e-15
    assert oracle.silu(0.0, prec=p) == 0.0
    assert abs(oracle.silu(1.0, prec=p) - 1.0 / (1.0 + math.exp(-1.0))) < tol
    assert abs(oracle.silu(30.0, prec=p) - 30.0) < 1e-5
    assert abs(oracle.silu(-30.0, prec=p)) < 1e-10
    for z in (0.3, 1.7, 4.2):  # silu(z) - silu(-z) = z
        assert abs(oracle.silu(z, prec=p) - oracle.silu(-z, prec=p) - z) < 4 * tol * (1 + z)


# ---- attention ------------------------------------------------------------------------

@pytest.mark.parametrize("p", PRECS)
def test_attention_single_entry_returns_v(p):
    rng = np.random.default_rng(6)
    q = rng.standard_normal(64) * 5
    k = bits(rng.standard_normal((1, 64)))
    v = bits(rng.standard_normal((1, 64)))
    np.testing.assert_array_equal(oracle.attention(q, k, v, prec=p), widen(v[0]).astype(oracle._dtype(p)))


@pytest.mark.parametrize("p", PRECS)
def test_attention_zero_query_is_mean_of_v(p):
    rng = np.random.default_rng(7)
    k = bits(rng.standard_normal((37, 64)))
    v = bits(rng.standard_normal((37, 64)))
    got = oracle.attention(np.zeros(64), k, v, prec=p)
    np.testing.assert_allclose(got, widen(v).mean(axis=0), rtol=1e-5 if p == 32 else 1e-12, atol=1e-6)


@pytest.mark.parametrize("p", PRECS)
def test_attention_two_entries_closed_form_scale(p):
    # hd = 4, k0 = 0, k1 = e0, q = a e0: scores 0 and a / sqrt(4), so the weight on
    # entry 1 is sigmoid(a / 2). A missing or wrong 1/sqrt(hd) scale fails this.
    a = 3.0
    q = np.array([a, 0, 0, 0])
    k = bits([[0, 0, 0, 0], [1, 0, 0, 0]])
    v = bits([[1, 2, 0, -1], [-3, 0.5, 4, 2]])
    w1 = 1.0 / (1.0 + math.exp(-a / 2.0))
    want = (1 - w1) * widen(v[0]) + w1 * widen(v[1])
    np.testing.assert_allclose(oracle.attention(q, k, v, prec=p), want, rtol=1e-6 if p == 32 else 1e-14)


@pytest.mark.parametrize("p", PRECS)
def test_attention_onehot_score_and_permutation(p):
    rng = np.random.default_rng(8)
    n, hd = 20, 64
    k = rng.standard_normal((n, hd)) * 0.01
    k[11] = 0
    k[11, 5] = 1.0
    q = np.zeros(hd)
    q[5] = 400.0  # score of entry 11 is 50 above the rest
    kb, vb = bits(k), bits(rng.standard_normal((n, hd)))
    np.testing.assert_allclose(oracle.attention(q, kb, vb, prec=p), widen(vb[11]), rtol=1e-6, atol=1e-6)
    perm = rng.permutation(n)
    q2 = rng.standard_normal(hd)
    a = oracle.attention(q2, kb, vb, prec=p)
    b = oracle.attention(q2, kb[perm].copy(), vb[perm].copy(), prec=p)
    np.testing.assert_allclose(a, b, rtol=1e-5 if p == 32 else 1e-12, atol=1e-6)


# ---- argmax -----------------------------------------------------------------------------

@pytest.mark.parametrize("p", PRECS)
def test_argmax_lowest_index_on_ties(p):
    assert oracle.argmax([0.5, 2.0, -1.0, 2.0, 1.9], prec=p) == 1
    assert oracle.argmax([3.0, 3.0], prec=p) == 0
    assert oracle.argmax([-5.0, -4.0, -4.5], prec=p) == 1
