"""Pins of the oracle's projections around the RNN mixer (arXiv 2601.22156,
Appendix A, Eq. 18: q = Norm(x W_q), k = Norm(x W_k), v = x W_v,
z = sigmoid(x W_z), y = (Norm(o) . z) W_o^T) and of its saved-feature
quantities, each against something other than the oracle itself: hand-computed
products, identity weights, linearity and the closed forms of the feature map."""
import numpy as np
import pytest

import oracle


def test_matmul_nt_hand_computed():
    # out[m, n] = sum_k a[m, k] w[n, k]: [1 2] against rows [3 4] and [5 6]
    # (the untransposed product x W would give [13 16])
    assert np.array_equal(oracle.matmul_nt([[1.0, 2.0]], [[3.0, 4.0], [5.0, 6.0]]), [[11.0, 17.0]])
    # two rows, three inner terms: [[1,0,2],[0,1,-1]] x [[1,1,1],[2,0,1]]^T
    got = oracle.matmul_nt([[1.0, 0.0, 2.0], [0.0, 1.0, -1.0]], [[1.0, 1.0, 1.0], [2.0, 0.0, 1.0]])
    assert np.array_equal(got, [[3.0, 4.0], [0.0, -1.0]])


def identity_blocks(H, d):
    """w_qkvz with W_j,h = (j + 1) times the selector of head h's slice of x."""
    D = H * d
    w = np.zeros((H, 4, d, D))
    for h in range(H):
        for j in range(4):
            for c in range(d):
                w[h, j, c, h * d + c] = j + 1.0
    return w


def test_project_in_block_and_head_order():
    """Identity weights scaled 1, 2, 3, 4 for q, k, v, z: the outputs are x,
    2x, 3x, 4x cut into heads in order (a swapped block or head fails)."""
    rng = np.random.default_rng(0)
    B, T, H, d = 2, 3, 3, 4
    x = rng.standard_normal((B, T, H * d))
    q, k, v, g = oracle.project_in(x, identity_blocks(H, d))
    xh = x.reshape(B, T, H, d)
    assert np.array_equal(q, xh)
    assert np.array_equal(k, 2 * xh)
    assert np.array_equal(v, 3 * xh)
    assert np.array_equal(g, 4 * xh)


def test_identity_projections_reduce_to_the_mixer():
    """With W_q = W_k = W_v = W_z = identity the layer is the mixer on x."""
    rng = np.random.default_rng(1)
    B, T, H, d = 1, 9, 2, 8
    x = rng.standard_normal((B, T, H * d))
    w = identity_blocks(H, d) / np.arange(1, 5).reshape(1, 4, 1, 1)  # all four = I
    q, k, v, g = oracle.project_in(x, w)
    gam = oracle.gamma(H)
    y1, _, s1 = oracle.prefill(q, k, v, g, gam, base=1e4)
    xh = x.reshape(B, T, H, d)
    y2, _, s2 = oracle.prefill(xh, xh, xh, xh, gam, base=1e4)
    assert np.array_equal(y1, y2) and np.array_equal(s1, s2)


def test_project_out_hand_computed_head_order():
    """Two heads of width 1 with u = (1, 2) against W_o = [3 4]: 1*3 + 2*4 = 11
    (heads concatenated in order; reversed heads would give 10)."""
    u = np.array([1.0, 2.0]).reshape(1, 1, 2, 1)
    assert np.array_equal(oracle.project_out(u, [[3.0, 4.0]]), np.array([[[11.0]]]))
    # two output features, heads of width 2
    u = np.array([1.0, -1.0, 2.0, 0.5]).reshape(1, 1, 2, 2)
    w = [[1.0, 0.0, 0.0, 0.0], [0.0, 1.0, 1.0, 2.0]]  # feature 0 = u[0,0]; feature 1 = u01 + u10 + 2 u11
    assert np.array_equal(oracle.project_out(u, w), np.array([[[1.0, 2.0]]]))


def test_projections_are_linear_in_x():
    rng = np.random.default_rng(2)
    B, T, H, d, D = 1, 5, 2, 4, 6
    w = rng.standard_normal((H, 4, d, D))
    x1, x2 = rng.standard_normal((B, T, D)), rng.standard_normal((B, T, D))
    a, b = 0.75, -2.0
    lhs = oracle.project_in(a * x1 + b * x2, w)
    for l, r1, r2 in zip(lhs, oracle.project_in(x1, w), oracle.project_in(x2, w)):
        assert np.allclose(l, a * r1 + b * r2, rtol=0, atol=1e-12)
    wo = rng.standard_normal((D, H * d))
    u1, u2 = rng.standard_normal((B, T, H, d)), rng.standard_normal((B, T, H, d))
    assert np.allclose(oracle.project_out(a * u1 + b * u2, wo),
                       a * oracle.project_out(u1, wo) + b * oracle.project_out(u2, wo), atol=1e-12)


def test_saved_features_closed_forms():
    """q~ . k~ = (q . k) / (RMS(q) RMS(k) sqrt(d)) because RoPE rotates both rows
    by the same angle; |q~|^2 = d mean(q^2) / (mean(q^2) + eps); 1/RMS by its
    definition on a row of constant magnitude."""
    rng = np.random.default_rng(3)
    B, T, H, d, eps = 1, 4, 2, 8, 1e-6
    q, k = rng.standard_normal((B, T, H, d)), rng.standard_normal((B, T, H, d))
    qt, kt, rq, rk, diag = oracle.features(q, k, pos_offset=1000, base=1e4, eps=eps)
    for t in range(T):
        for h in range(H):
            mq, mk = np.mean(q[0, t, h] ** 2), np.mean(k[0, t, h] ** 2)
            want = np.dot(q[0, t, h], k[0, t, h]) / np.sqrt((mq + eps) * (mk + eps) * d)
            assert diag[0, h, t] == pytest.approx(want, rel=1e-12, abs=1e-14)
            assert np.dot(qt[0, t, h], qt[0, t, h]) == pytest.approx(d * mq / (mq + eps), rel=1e-12)
    row = np.full((1, 1, 1, d), -3.0)
    _, _, rq1, _, _ = oracle.features(row, row, eps=0.0)
    assert rq1[0, 0, 0] == pytest.approx(1.0 / 3.0, rel=1e-15)
