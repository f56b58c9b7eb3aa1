"""Pins of the oracle's softmax attention (arXiv 2601.22156, Section 5.1
"Attention Logits Scaling", Eq. 11; Appendix A "Attention Layers", Eq. 17)
against closed forms and hand-computed cases, independent of its code."""
import math

import numpy as np
import pytest

import oracle


def rand(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


def test_single_token_attends_to_itself():
    # T = 1: the only key gets weight 1, so o_0 = v_0 whatever q, k and a are
    q, k, v, g = rand((2, 1, 4, 8), 1), rand((2, 1, 2, 8), 2), rand((2, 1, 2, 8), 3), rand((2, 1, 4, 8), 4)
    _, o = oracle.attention(q, k, v, g, a=500.0, pos_offset=123)
    for h in range(4):
        np.testing.assert_allclose(o[:, 0, h], v[:, 0, h // 2], rtol=0, atol=1e-15)


def test_identical_keys_average_the_values():
    # every key equal: all logits of a row are equal, so o_t is the mean of v_0..v_t
    T, d = 9, 8
    q, v, g = rand((1, T, 1, d), 5), rand((1, T, 1, d), 6), rand((1, T, 1, d), 7)
    k = np.broadcast_to(rand((1, 1, 1, d), 8), (1, T, 1, d)).copy()
    _, o = oracle.attention(q, k, v, g, a=600.0)
    for t in range(T):
        np.testing.assert_allclose(o[0, t, 0], v[0, :t + 1, 0].mean(axis=0), rtol=0, atol=1e-14)


@pytest.mark.parametrize("pos_offset,s", [(0, 2.0), (4, 3.0)])
def test_hand_computed_two_token_case(pos_offset, s):
    # a = 2: the second token sits at p = pos_offset + 1, so s = log_2(p + 1 + 2),
    # 2 at p = 1 and 3 at p = 5.  With q_1 = (c, 0), k_0 = (1, 0), k_1 = 0 and
    # c = sqrt(2) ln 3 / s the logits are ln 3 and 0: weights 3/4 and 1/4.
    c = math.sqrt(2.0) * math.log(3.0) / s
    q = np.array([[[[0.3, -0.2]], [[c, 0.0]]]])
    k = np.array([[[[1.0, 0.0]], [[0.0, 0.0]]]])
    v = np.array([[[[1.0, 0.0]], [[0.0, 1.0]]]])
    g = np.zeros((1, 2, 1, 2))
    y, o = oracle.attention(q, k, v, g, a=2.0, pos_offset=pos_offset)
    np.testing.assert_allclose(o[0, 1, 0], [0.75, 0.25], rtol=0, atol=1e-14)
    np.testing.assert_allclose(o[0, 0, 0], [1.0, 0.0], rtol=0, atol=1e-15)
    # output norm and gate: o_1 / RMS(o_1) times sigmoid(0) = 1/2
    rms = math.sqrt((0.75 ** 2 + 0.25 ** 2) / 2 + 1e-6)
    np.testing.assert_allclose(y[0, 1, 0], [0.375 / rms, 0.125 / rms], rtol=1e-14, atol=0)


def test_grouped_heads_share_their_key_value_head():
    # Hq = 4 over Hkv = 2 equals Hq = Hkv = 4 with each key/value head repeated
    B, T, d = 2, 7, 8
    q, g = rand((B, T, 4, d), 9), rand((B, T, 4, d), 10)
    k, v = rand((B, T, 2, d), 11), rand((B, T, 2, d), 12)
    y, o = oracle.attention(q, k, v, g, a=900.0)
    y2, o2 = oracle.attention(q, np.repeat(k, 2, axis=2), np.repeat(v, 2, axis=2), g, a=900.0)
    np.testing.assert_array_equal(o, o2)
    np.testing.assert_array_equal(y, y2)


def test_causal():
    # later tokens change nothing before them
    B, T, d, t0 = 1, 10, 8, 5
    q, k, v, g = rand((B, T, 2, d), 13), rand((B, T, 1, d), 14), rand((B, T, 1, d), 15), rand((B, T, 2, d), 16)
    _, o = oracle.attention(q, k, v, g, a=500.0)
    k2, v2 = k.copy(), v.copy()
    k2[:, t0 + 1:] = rand(k2[:, t0 + 1:].shape, 17)
    v2[:, t0 + 1:] = rand(v2[:, t0 + 1:].shape, 18)
    _, o2 = oracle.attention(q, k2, v2, g, a=500.0)
    np.testing.assert_array_equal(o[:, :t0 + 1], o2[:, :t0 + 1])
    assert not np.allclose(o[:, t0 + 1:], o2[:, t0 + 1:])


def test_a_dominant_key_selects_its_value():
    # key 3 parallel to q and 40 times longer than the others: o_t (t >= 3) is v_3
    T, d = 8, 16
    rng = np.random.default_rng(19)
    q = np.tile(rng.standard_normal(d), (1, T, 1, 1))
    k = 0.01 * rng.standard_normal((1, T, 1, d))
    k[0, 3, 0] = 40.0 * q[0, 0, 0]
    v, g = rng.standard_normal((1, T, 1, d)), rng.standard_normal((1, T, 1, d))
    _, o = oracle.attention(q, k, v, g, a=500.0)
    for t in range(3, T):
        np.testing.assert_allclose(o[0, t, 0], v[0, 3, 0], rtol=0, atol=1e-12)
