"""Pins of the oracle's decode attention and RoPE.

Attention is the plain definition (nalar.dev "Kuantisasi KV Cache dengan Error
Budget yang Eksplisit": s_i = q.k_i / sqrt(D); output = sum_i p_i v_i).  The
pins are closed forms and identities from that page, not a second copy of the
formula.  RoPE is split-half (lehuy.net "NexusQuant", section "Cac mo hinh
duoc ho tro"), applied to keys stored pre-RoPE (troisinh.com "KV Cache
Quantization", "RoPE - Cai bay tinh vi").
"""

import math

import numpy as np
import pytest

from oracle import kvq_oracle as O


def test_single_token_returns_its_value():
    rng = np.random.default_rng(0)
    q, k, v = rng.standard_normal((3, 128))
    assert np.array_equal(O.attention_f64(q, k[None], v[None]), v)


def test_empty_cache_gives_zero():
    out = O.attention_f64(np.ones(128), np.zeros((0, 128)), np.zeros((0, 128)))
    assert np.array_equal(out, np.zeros(128))


def test_identical_keys_average_values():
    rng = np.random.default_rng(1)
    q, k = rng.standard_normal((2, 64))
    V = rng.standard_normal((37, 64))
    out = O.attention_f64(q, np.tile(k, (37, 1)), V)
    assert np.allclose(out, V.mean(axis=0), atol=1e-14)


def test_two_tokens_closed_form_with_sqrt_d():
    """q = a e_0, k_i = b_i e_0: s_i = a b_i / sqrt(D) and the output is
    v_1 sigmoid(s_1 - s_2) + v_2 sigmoid(s_2 - s_1)."""
    D = 128
    a, b1, b2 = 3.0, 2.0, -1.5
    q = np.zeros(D); q[0] = a
    K = np.zeros((2, D)); K[0, 0] = b1; K[1, 0] = b2
    rng = np.random.default_rng(2)
    V = rng.standard_normal((2, D))
    s1, s2 = a * b1 / math.sqrt(D), a * b2 / math.sqrt(D)
    assert np.allclose(O.scores_f64(q, K), [s1, s2], atol=1e-15)
    sig = 1.0 / (1.0 + math.exp(-(s1 - s2)))
    assert np.allclose(O.attention_f64(q, K, V), sig * V[0] + (1 - sig) * V[1], atol=1e-14)


def test_shift_and_permutation_invariance():
    rng = np.random.default_rng(3)
    D, T = 128, 50
    q = rng.standard_normal(D)
    K, V = rng.standard_normal((2, T, D))
    base = O.attention_f64(q, K, V)
    # adding u with q.u = c to every key shifts every score by the same constant
    u = 5.0 * q / np.dot(q, q)
    assert np.allclose(O.attention_f64(q, K + u, V), base, atol=1e-13)
    perm = rng.permutation(T)
    assert np.allclose(O.attention_f64(q, K[perm], V[perm]), base, atol=1e-13)


def test_dominant_key_selects_its_value():
    rng = np.random.default_rng(4)
    D, T = 128, 20
    q = rng.standard_normal(D)
    K, V = rng.standard_normal((2, T, D))
    K[7] = q / np.linalg.norm(q) * 60.0 * math.sqrt(D) / np.linalg.norm(q)
    out = O.attention_f64(q, K, V)
    assert np.allclose(out, V[7], atol=1e-12)


def test_key_error_identity():
    """k_i + e_i gives s_i' = s_i + q.e_i / sqrt(D) (nalar.dev, key error)."""
    rng = np.random.default_rng(5)
    D, T = 128, 40
    q = rng.standard_normal(D)
    K, E = rng.standard_normal((2, T, D))
    E *= 0.01
    lhs = O.scores_f64(q, K + E)
    rhs = O.scores_f64(q, K) + (E @ q) / math.sqrt(D)
    assert np.max(np.abs(lhs - rhs)) < 1e-12


def test_value_error_identity():
    """With the probabilities fixed, v_i + r_i moves the output by sum_i p_i r_i
    (nalar.dev, value error)."""
    rng = np.random.default_rng(6)
    D, T = 128, 40
    q = rng.standard_normal(D)
    K, V, Rr = rng.standard_normal((3, T, D))
    Rr *= 0.05
    p = O.softmax_f64(O.scores_f64(q, K))
    delta = O.attention_f64(q, K, V + Rr) - O.attention_f64(q, K, V)
    assert np.max(np.abs(delta - p @ Rr)) < 1e-12


def test_brute_force_loops_tiny():
    rng = np.random.default_rng(7)
    D, T = 4, 6
    q = rng.standard_normal(D)
    K, V = rng.standard_normal((2, T, D))
    w = [math.exp(sum(q[d] * K[t][d] for d in range(D)) / math.sqrt(D)) for t in range(T)]
    z = sum(w)
    ref = [sum(w[t] * V[t][d] for t in range(T)) / z for d in range(D)]
    assert np.allclose(O.attention_f64(q, K, V), ref, atol=1e-14)


def test_rope_identity_at_zero_and_norm():
    rng = np.random.default_rng(8)
    k = rng.standard_normal((5, 128))
    assert np.allclose(O.rope_f64(k, np.zeros(5), 1e4), k, atol=0)
    r = O.rope_f64(k, np.arange(5) * 1000, 1e4)
    h = 64
    assert np.allclose(r[:, :h] ** 2 + r[:, h:] ** 2, k[:, :h] ** 2 + k[:, h:] ** 2, rtol=1e-12)


def test_rope_is_complex_rotation_of_split_halves():
    rng = np.random.default_rng(9)
    D = 128
    k = rng.standard_normal((7, D))
    t = np.array([0, 1, 5, 100, 4095, 31000, 32767])
    z = (k[:, :64] + 1j * k[:, 64:]) * np.exp(1j * t[:, None] * 10000.0 ** (-np.arange(64) * 2.0 / D))
    r = O.rope_f64(k, t, 1e4)
    assert np.allclose(r[:, :64], z.real, atol=1e-12)
    assert np.allclose(r[:, 64:], z.imag, atol=1e-12)
    # frequency 0 turns by exactly t radians
    assert np.allclose(np.arctan2(r[1, 64], r[1, 0]) - np.arctan2(k[1, 64], k[1, 0]),
                       1.0, atol=1e-12)


def test_rope_relative_position():
    rng = np.random.default_rng(10)
    q, k = rng.standard_normal((2, 128))
    a, b = 37, 1290
    lhs = np.dot(O.rope_f64(q[None], [a], 1e4)[0], O.rope_f64(k[None], [b], 1e4)[0])
    rhs = np.dot(q, O.rope_f64(k[None], [b - a], 1e4)[0])
    assert abs(lhs - rhs) < 1e-11


def test_gqa_head_mapping():
    """Query head h reads kv head h // (H_q / H_kv)."""
    cfg = O.Config(L=1, H_kv=2, H_q=4, D=128, batch=1, max_T=8, k_fmt=O.Fmt(8, 32), v_fmt=O.Fmt(8, 32),
                   residual_window=8)
    rng = np.random.default_rng(11)
    k = rng.standard_normal((3, 2, 128)).astype(np.float16)
    v = np.zeros((3, 2, 128), np.float16)
    v[:, 0] = 1.0
    v[:, 1] = -2.0
    bufs = O.new_buffers(cfg)
    O.append(cfg, bufs, 0, k.view(np.uint16), v.view(np.uint16), [3], [0])
    q = rng.standard_normal((1, 1, 4, 128)).astype(np.float16).view(np.uint16)
    out = O.decode_attention(cfg, bufs, 0, 1, q, [3])
    assert np.allclose(out[0, 0, :2], 1.0) and np.allclose(out[0, 0, 2:], -2.0)
