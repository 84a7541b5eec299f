"""Pins for the oracle's per-head RMSNorm + RoPE (CPU).

RoPE convention: "unsloth: compare main...flex-moe-qwen3" ·
flex_gemma4_moe.py · Rotary helpers (rotate_half = cat(-x2, x1);
x*cos + rotate_half(x)*sin).
"""
import math

import numpy as np

import oracle


def test_rope_hand_values_pin_frequencies_and_sign():
    # D=4, theta=100: inv_freq = [100^0, 100^(-2/4)] = [1, 0.1]
    x = np.array([[[1.0, 2.0, 0.0, 0.0]]])          # pairs (x0, x2), (x1, x3)
    out = oracle.rope(x, [10.0], 100.0)[0, 0]
    # pair 0 rotates by 10 rad, pair 1 by 1 rad; rotate_half gives
    # out_i = x_i cos - x_{i+2} sin, out_{i+2} = x_{i+2} cos + x_i sin
    exp = [math.cos(10.0), 2 * math.cos(1.0), math.sin(10.0), 2 * math.sin(1.0)]
    assert np.allclose(out, exp, atol=1e-15)
    assert np.allclose(oracle.inv_freq(4, 100.0), [1.0, 0.1], rtol=1e-15)


def test_rope_equals_complex_rotation():
    # rotate-half pairing (i, i + D/2) is multiplication of x_i + j x_{i+D/2}
    # by exp(j * pos * f_i), f_i the geometric frequencies from 1 down to
    # theta^(-(D-2)/D) with ratio theta^(-2/D)
    rng = np.random.default_rng(1)
    D, theta = 64, 1e6
    ratio = theta ** (-2.0 / D)
    f = np.array([ratio ** i for i in range(D // 2)])
    x = rng.standard_normal((3, 5, D))
    pos = np.array([0.0, 17.0, 4095.0])
    z = x[..., : D // 2] + 1j * x[..., D // 2:]
    zr = z * np.exp(1j * pos[:, None, None] * f)
    out = oracle.rope(x, pos, theta)
    assert np.allclose(out[..., : D // 2], zr.real, atol=1e-9)
    assert np.allclose(out[..., D // 2:], zr.imag, atol=1e-9)


def test_rope_invariants():
    rng = np.random.default_rng(2)
    x = rng.standard_normal((4, 3, 128))
    p = np.array([1.0, 5.0, 100.0, 1023.0])
    y = oracle.rope(x, p, 5e5)
    assert np.allclose(np.linalg.norm(y, axis=-1), np.linalg.norm(x, axis=-1), rtol=1e-12)
    assert np.allclose(oracle.rope(y, -p, 5e5), x, atol=1e-12)
    assert np.allclose(oracle.rope(oracle.rope(x, p, 5e5), 2 * p, 5e5),
                       oracle.rope(x, 3 * p, 5e5), atol=1e-9)
    assert np.array_equal(oracle.rope(x, np.zeros(4), 5e5), x)


def test_rms_norm_closed_forms():
    # constant input c with unit gain -> c / sqrt(c^2 + eps)
    for c in (-3.0, 0.5, 2.0):
        y = oracle.rms_norm(np.full((1, 8), c), None, 1e-6)
        assert np.allclose(y, c / math.sqrt(c * c + 1e-6), rtol=1e-15)
    # [3, 4]: mean square 12.5 -> y = x / sqrt(12.5 + eps) * gamma
    y = oracle.rms_norm(np.array([3.0, 4.0]), np.array([2.0, -1.0]), 0.0)
    assert np.allclose(y, [6 / math.sqrt(12.5), -4 / math.sqrt(12.5)], rtol=1e-15)
    # eps inside the root: all-zero input stays zero, tiny input is damped
    assert not oracle.rms_norm(np.zeros((2, 4)), None, 1e-6).any()
    y = oracle.rms_norm(np.full(4, 1e-3), None, 1e-6)
    assert np.allclose(y, 1e-3 / math.sqrt(1e-6 + 1e-6), rtol=1e-12)
    # scale invariance (eps=0) and unit mean square with unit gain
    rng = np.random.default_rng(3)
    x = rng.standard_normal((5, 64))
    assert np.allclose(oracle.rms_norm(7.5 * x, None, 0.0), oracle.rms_norm(x, None, 0.0))
    assert np.allclose(np.mean(oracle.rms_norm(x, None, 0.0) ** 2, -1), 1.0)


def test_norm_then_rope_order_and_pos_zero():
    rng = np.random.default_rng(4)
    q = rng.standard_normal((2, 4, 32))
    k = rng.standard_normal((2, 2, 32))
    gq = 1 + 0.1 * rng.standard_normal(32)
    gk = 1 + 0.1 * rng.standard_normal(32)
    q0, k0 = oracle.qk_norm_rope(q, k, gq, gk, [0, 0], 1e4, 1e-6)
    assert np.allclose(q0, oracle.rms_norm(q, gq, 1e-6), atol=0)
    assert np.allclose(k0, oracle.rms_norm(k, gk, 1e-6), atol=0)
    # norm before rotation: with a non-uniform gain the two orders differ
    q1, _ = oracle.qk_norm_rope(q, k, gq, gk, [3, 9], 1e4, 1e-6)
    other = oracle.rms_norm(oracle.rope(q, [3, 9], 1e4), gq, 1e-6)
    assert not np.allclose(q1, other)
    # without the norm branch only the rotation is applied
    q2, k2 = oracle.qk_norm_rope(q, k, None, None, [3, 9], 1e4, 1e-6, norm=False)
    assert np.allclose(q2, oracle.rope(q, [3, 9], 1e4), atol=0)


# ------------------------------------------------ Gemma-4 variants
def test_proportional_rope_hand_values_and_pass_through():
    """Partial (proportional) RoPE: only the leading rotary_dims rotate, with the
    full-dimension frequencies; the tail pairs see inv_freq 0 (cos 1, sin 0)."""
    # D=8, theta=100, rotary_dims=4: inv_freq = [1, 100^(-2/8), 0, 0]
    f = oracle.inv_freq(8, 100.0, 4)
    assert np.allclose(f, [1.0, 100.0 ** -0.25, 0.0, 0.0], rtol=1e-15)
    x = np.arange(1.0, 9.0)[None, :]           # x1 = [1,2,3,4], x2 = [5,6,7,8]
    p = 0.5
    y = oracle.rope(x, [p], 100.0, 4)[0]
    a0, a1 = p * 1.0, p * 100.0 ** -0.25
    want = [1 * math.cos(a0) - 5 * math.sin(a0), 2 * math.cos(a1) - 6 * math.sin(a1), 3.0, 4.0,
            5 * math.cos(a0) + 1 * math.sin(a0), 6 * math.cos(a1) + 2 * math.sin(a1), 7.0, 8.0]
    assert np.allclose(y, want, rtol=1e-13)
    rng = np.random.default_rng(10)
    x = rng.standard_normal((3, 2, 512))
    pos = np.array([7.0, 300.0, 2047.0])
    y = oracle.rope(x, pos, 1e6, 128)
    # pairs 64..255 (dims 64..255 and 320..511) pass through exactly
    assert np.array_equal(y[..., 64:256], x[..., 64:256])
    assert np.array_equal(y[..., 320:], x[..., 320:])
    # the rotated part equals the full rope's first 64 pairs (same frequencies)
    full = oracle.rope(x, pos, 1e6)
    assert np.allclose(y[..., :64], full[..., :64], atol=0)
    assert np.allclose(y[..., 256:320], full[..., 256:320], atol=0)
    # norm preserved, inverse rotation, and the two ends of the range
    assert np.allclose(np.linalg.norm(y, axis=-1), np.linalg.norm(x, axis=-1), rtol=1e-12)
    assert np.allclose(oracle.rope(y, -pos, 1e6, 128), x, atol=1e-12)
    assert np.array_equal(oracle.rope(x, pos, 1e6, 0), x)
    assert np.array_equal(oracle.rope(x, pos, 1e6, 512), full)


def test_v_norm_is_rms_norm_without_gain():
    # constant vector c -> c / sqrt(c^2 + eps); [3, 4] with eps 0 -> x / sqrt(12.5)
    for c in (-2.0, 0.25):
        assert np.allclose(oracle.v_norm(np.full((1, 1, 6), c), 1e-6),
                           c / math.sqrt(c * c + 1e-6), rtol=1e-15)
    assert np.allclose(oracle.v_norm(np.array([3.0, 4.0]), 0.0),
                       [3 / math.sqrt(12.5), 4 / math.sqrt(12.5)], rtol=1e-15)
    rng = np.random.default_rng(11)
    v = rng.standard_normal((4, 2, 256))
    y = oracle.v_norm(v, 0.0)
    assert np.allclose(np.mean(y * y, -1), 1.0)                 # unit mean square
    assert np.allclose(oracle.v_norm(-3.0 * v, 0.0), -y)         # scale-free, sign kept
    # with K=V the value is the raw k normalised without a gain: it differs from the key
    # (which also carries gamma_k and the rotation)
    gk = 1 + 0.1 * rng.standard_normal(256)
    _, k = oracle.qk_norm_rope(v, v, gk, gk, [5, 9, 11, 13], 1e6, 1e-6, rotary_dims=64)
    assert not np.allclose(oracle.v_norm(v, 1e-6), k)
