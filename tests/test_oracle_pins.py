"""Pins for the fp64 oracle against facts the paper and mathematics fix.

Source: arXiv 2601.22156 ("Hybrid Linear Attention Done Right"), Appendix A,
Eq. 18 (RNN layer) and Eq. 19 with its printed gamma table; the zero-state
unrolled (closed) form of the recurrence and the decay horizon
tau_h = 1/(-ln gamma_h) = 2^(8h/H) from the same paper's reading notes
("Lightning Attention 如何提供局部时序表示", section 2.5).  Appendix G, Table 10
places plain linear attention (gamma = 1) in the same family.

Each pin is independent of the oracle's own code path: printed values, a
closed form evaluated with plain numpy sums, the textbook 2-D rotation, finite
differences, or an invariant of the mathematics.
"""
import math
import os

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def rnd(rng, *shape):
    return rng.standard_normal(shape)


def make(rng, B, T, H, d, with_state=False):
    q, k, v, g = (rnd(rng, B, T, H, d) for _ in range(4))
    s0 = rnd(rng, B, H, d, d) * 0.3 if with_state else None
    return q, k, v, g, s0


def features(x, pos_offset, base, eps, scale):
    """Oracle q~ / k~ rows for every (b, t, h)."""
    B, T, H, d = x.shape
    out = np.zeros_like(x)
    for b in range(B):
        for t in range(T):
            for h in range(H):
                out[b, t, h] = oracle.feature(x[b, t, h], pos_offset + t, base, eps, scale)
    return out


# --------------------------------------------------------------------------- Eq. 19


def test_gamma_matches_printed_table():
    """Appendix A prints gamma_h for H = 32 as shortest decimal strings of fp32
    numbers.  Eq. 19 in fp64, rounded to fp32, must land on the printed fp32
    value or its neighbour (the paper evaluated Eq. 19 in fp32, which moves
    one of the 32 entries, h = 7, by one fp32 ulp)."""
    rows = [l.strip() for l in open(os.path.join(GOLDEN, "gamma_H32.txt"))
            if l.strip() and not l.startswith("#")]
    assert len(rows) == 32
    gam = oracle.gamma(32)
    exact = 0
    for h, txt in enumerate(rows):
        printed = np.float32(float(txt))
        mine = np.float32(gam[h])
        ulp = np.spacing(printed)
        assert abs(float(mine) - float(printed)) <= float(ulp), (h, gam[h], txt)
        exact += int(mine == printed)
    assert exact >= 31


@pytest.mark.parametrize("H", [2, 16, 32])
def test_gamma_decay_horizon(H):
    """tau_h = 1/(-ln gamma_h) = 2^(8h/H); the slowest head has tau = 256 and
    decays to e^-16 ~ 1.13e-7 over 4096 tokens."""
    gam = oracle.gamma(H)
    for h in range(H):
        tau = 1.0 / (-math.log(gam[h]))
        assert tau == pytest.approx(2.0 ** (8.0 * (h + 1) / H), rel=1e-12)
    assert 1.0 / (-math.log(gam[-1])) == pytest.approx(256.0, rel=1e-12)
    assert gam[-1] ** 4096 == pytest.approx(math.exp(-16.0), rel=1e-9)
    assert gam[-1] ** 4096 == pytest.approx(1.13e-7, rel=5e-3)
    assert np.all(np.diff(gam) > 0) and gam[0] > 0 and gam[-1] < 1


# --------------------------------------------------------------------------- Norm / RoPE


def test_feature_two_dim_rotation():
    """d = 2: the single RoPE frequency is base^0 = 1, so RoPE_p is the plane
    rotation by p radians applied to the RMS-normalised row."""
    x = np.array([3.0, 4.0])
    r = 1.0 / math.sqrt((9.0 + 16.0) / 2.0)
    a, b = 3.0 * r, 4.0 * r
    for p in [0, 1, 7, 123456]:
        got = oracle.feature(x, p, 1e6, eps=0.0, scale=1.0)
        want = [a * math.cos(p) - b * math.sin(p), a * math.sin(p) + b * math.cos(p)]
        np.testing.assert_allclose(got, want, rtol=0, atol=1e-12)


def test_feature_pairing_and_frequencies():
    """d = 4, rotate-half pairing: (x0, x2) turns by p, (x1, x3) by p * base^(-1/2)."""
    x = np.array([1.0, -2.0, 0.5, 3.0])
    base, p = 100.0, 5
    r = 1.0 / math.sqrt(np.mean(x * x))
    n = x * r
    got = oracle.feature(x, p, base, eps=0.0, scale=0.5)
    th = [p * 1.0, p * base ** -0.5]
    want = np.zeros(4)
    for i in range(2):
        c, s = math.cos(th[i]), math.sin(th[i])
        want[i] = n[i] * c - n[i + 2] * s
        want[i + 2] = n[i] * s + n[i + 2] * c
    np.testing.assert_allclose(got, 0.5 * want, atol=1e-13)


def test_feature_unit_rms_and_norm_preserving():
    rng = np.random.default_rng(3)
    for d in [64, 128]:
        x = rng.standard_normal(d) * 7.0
        f = oracle.feature(x, 4097, 1e6, eps=0.0, scale=1.0)
        assert np.sqrt(np.mean(f * f)) == pytest.approx(1.0, abs=1e-13)
        fk = oracle.feature(x, 4097, 1e6, eps=0.0, scale=1.0 / math.sqrt(d))
        assert np.linalg.norm(fk) == pytest.approx(1.0, abs=1e-13)


def test_feature_relative_position():
    """RoPE: <RoPE_p a, RoPE_p' b> depends only on p - p'."""
    rng = np.random.default_rng(4)
    a, b = rng.standard_normal(128), rng.standard_normal(128)
    ref = oracle.feature(a, 10, 1e6) @ oracle.feature(b, 3, 1e6)
    for s in [1, 1000, 524288]:
        got = oracle.feature(a, 10 + s, 1e6) @ oracle.feature(b, 3 + s, 1e6)
        assert got == pytest.approx(ref, abs=1e-9)


# --------------------------------------------------------------------------- Eq. 18 recurrence


def closed_form(qt, kt, v, gam, s0):
    """o_t = gamma^{t+1} q~_t S_0 + sum_{s<=t} gamma^{t-s} (q~_t . k~_s) v_s and
    S_T = gamma^T S_0 + sum_s gamma^{T-1-s} k~_s^T v_s, by brute-force sums."""
    B, T, H, d = qt.shape
    o = np.zeros_like(qt)
    S = np.zeros((B, H, d, d))
    for b in range(B):
        for h in range(H):
            gm = gam[h]
            init = s0[b, h] if s0 is not None else np.zeros((d, d))
            for t in range(T):
                acc = gm ** (t + 1) * (qt[b, t, h] @ init)
                for s in range(t + 1):
                    acc = acc + gm ** (t - s) * float(qt[b, t, h] @ kt[b, s, h]) * v[b, s, h]
                o[b, t, h] = acc
            st = gm ** T * init
            for s in range(T):
                st = st + gm ** (T - 1 - s) * np.outer(kt[b, s, h], v[b, s, h])
            S[b, h] = st
    return o, S


@pytest.mark.parametrize("B,T,H,d,with_state", [
    (1, 17, 2, 8, False), (2, 33, 2, 4, True), (1, 64, 32, 8, True), (1, 9, 3, 64, True)])
def test_recurrence_equals_closed_form(B, T, H, d, with_state):
    rng = np.random.default_rng(10 + T)
    q, k, v, g, s0 = make(rng, B, T, H, d, with_state)
    gam = oracle.gamma(H)
    base, eps, off = 1e4, 1e-6, 5
    y, o, st = oracle.prefill(q, k, v, g, gam, s0, pos_offset=off, base=base, eps=eps)
    qt = features(q, off, base, eps, 1.0)
    kt = features(k, off, base, eps, 1.0 / math.sqrt(d))
    o_ref, s_ref = closed_form(qt, kt, v, gam, s0)
    scale = max(1.0, np.abs(o_ref).max())
    np.testing.assert_allclose(o, o_ref, rtol=0, atol=1e-12 * scale)
    np.testing.assert_allclose(st, s_ref, rtol=0, atol=1e-12 * max(1.0, np.abs(s_ref).max()))


def test_gamma_one_is_causal_linear_attention():
    """gamma = 1 (Table 10's linear attention row): O = tril(Q~ K~^T) V."""
    rng = np.random.default_rng(11)
    B, T, H, d = 1, 40, 2, 16
    q, k, v, g, _ = make(rng, B, T, H, d)
    gam = np.ones(H)
    _, o, st = oracle.prefill(q, k, v, g, gam, None, base=1e4)
    qt = features(q, 0, 1e4, 1e-6, 1.0)
    kt = features(k, 0, 1e4, 1e-6, 1.0 / math.sqrt(d))
    for h in range(H):
        A = np.tril(qt[0, :, h] @ kt[0, :, h].T)
        np.testing.assert_allclose(o[0, :, h], A @ v[0, :, h], atol=1e-11)
        np.testing.assert_allclose(st[0, h], kt[0, :, h].T @ v[0, :, h], atol=1e-11)


def test_output_is_rmsnorm_times_sigmoid_gate():
    """y = Norm(o) * sigmoid(g): y / sigmoid(g) has unit RMS and the sign of o."""
    rng = np.random.default_rng(12)
    q, k, v, g, _ = make(rng, 1, 20, 2, 32)
    y, o, _ = oracle.prefill(q, k, v, g, oracle.gamma(2), eps=1e-12)
    n = y * (1.0 + np.exp(-g))
    np.testing.assert_allclose(np.sqrt(np.mean(n * n, axis=-1)), 1.0, atol=1e-9)
    assert np.all(np.sign(n) == np.sign(o))


def test_value_scale_invariance():
    """The output RMSNorm makes y invariant to v -> alpha v (alpha > 0) when eps = 0."""
    rng = np.random.default_rng(13)
    q, k, v, g, _ = make(rng, 1, 30, 2, 16)
    gam = oracle.gamma(2)
    y1, _, _ = oracle.prefill(q, k, v, g, gam, eps=0.0)
    y2, _, _ = oracle.prefill(q, k, 37.5 * v, g, gam, eps=0.0)
    np.testing.assert_allclose(y1, y2, atol=1e-12)


def test_position_shift_invariance():
    """With S_0 = 0 only relative positions enter o (RoPE)."""
    rng = np.random.default_rng(14)
    q, k, v, g, _ = make(rng, 1, 25, 2, 16)
    gam = oracle.gamma(2)
    _, o1, s1 = oracle.prefill(q, k, v, g, gam, pos_offset=0, base=1e6)
    _, o2, _ = oracle.prefill(q, k, v, g, gam, pos_offset=524288, base=1e6)
    np.testing.assert_allclose(o1, o2, atol=1e-9)


@pytest.mark.parametrize("T,chunk", [(100, 64), (128, 64), (100, 16), (37, 7), (5, 64)])
def test_chunked_equals_recurrent(T, chunk):
    rng = np.random.default_rng(15 + T)
    q, k, v, g, s0 = make(rng, 2, T, 3, 16, with_state=True)
    gam = oracle.gamma(3)
    y1, o1, s1 = oracle.prefill(q, k, v, g, gam, s0, pos_offset=3)
    y2, o2, s2 = oracle.prefill_chunked(q, k, v, g, gam, chunk, s0, pos_offset=3)
    np.testing.assert_allclose(o2, o1, atol=1e-12 * np.abs(o1).max())
    np.testing.assert_allclose(y2, y1, atol=1e-11)
    np.testing.assert_allclose(s2, s1, atol=1e-12 * np.abs(s1).max())


def test_split_prefill_then_decode_equals_one_shot():
    rng = np.random.default_rng(16)
    B, T1, n, H, d = 2, 20, 6, 4, 16
    q, k, v, g, s0 = make(rng, B, T1 + n, H, d, with_state=True)
    gam = oracle.gamma(H)
    y_all, _, s_all = oracle.prefill(q, k, v, g, gam, s0, pos_offset=0)
    # prefill T1 then prefill the rest from the handed-off state
    ya, _, sa = oracle.prefill(q[:, :T1], k[:, :T1], v[:, :T1], g[:, :T1], gam, s0)
    yb, _, sb = oracle.prefill(q[:, T1:], k[:, T1:], v[:, T1:], g[:, T1:], gam, sa, pos_offset=T1)
    np.testing.assert_allclose(np.concatenate([ya, yb], 1), y_all, atol=1e-12)
    np.testing.assert_allclose(sb, s_all, atol=1e-12 * np.abs(s_all).max())
    # prefill T1 then n decode steps
    st = sa
    for i in range(n):
        t = T1 + i
        yt, _, st = oracle.decode_step(q[:, t:t + 1], k[:, t:t + 1], v[:, t:t + 1], g[:, t:t + 1],
                                       gam, np.full(B, t), st)
        np.testing.assert_allclose(yt[:, 0], y_all[:, t], atol=1e-12)
    np.testing.assert_allclose(st, s_all, atol=1e-12 * np.abs(s_all).max())


def test_decode_positions_per_sequence():
    """Each sequence of a decode batch is rotated at its own position."""
    rng = np.random.default_rng(17)
    B, H, d = 3, 2, 8
    q, k, v, g, s0 = make(rng, B, 1, H, d, with_state=True)
    gam = oracle.gamma(H)
    pos = np.array([0, 99, 4096])
    y, o, st = oracle.decode_step(q, k, v, g, gam, pos, s0)
    for b in range(B):
        yb, ob, sb = oracle.prefill(q[b:b + 1], k[b:b + 1], v[b:b + 1], g[b:b + 1], gam,
                                    s0[b:b + 1], pos_offset=int(pos[b]))
        np.testing.assert_allclose(y[b], yb[0], atol=1e-13)
        np.testing.assert_allclose(st[b], sb[0], atol=1e-13)


def test_impulse_decays_with_horizon():
    """A single write k~_0^T v_0 followed by silent tokens (v = 0) decays as
    gamma^t: after tau_h tokens it is e^-1 of its size."""
    rng = np.random.default_rng(18)
    H, d = 4, 8
    gam = oracle.gamma(H)
    T = 300
    q, k, v, g, _ = make(rng, 1, T, H, d)
    v[:, 1:] = 0.0
    _, _, s_full = oracle.prefill(q, k, v, g, gam)
    _, _, s_one = oracle.prefill(q[:, :1], k[:, :1], v[:, :1], g[:, :1], gam)
    for h in range(H):
        ratio = np.linalg.norm(s_full[0, h]) / np.linalg.norm(s_one[0, h])
        assert ratio == pytest.approx(math.exp(-(T - 1) / 2.0 ** (8.0 * (h + 1) / H)), rel=1e-10)


# --------------------------------------------------------------------------- backward


def _loss(q, k, v, g, s0, gam, dy, dso, off, base, eps):
    y, _, st = oracle.prefill(q, k, v, g, gam, s0, pos_offset=off, base=base, eps=eps)
    return float(np.sum(dy * y) + np.sum(dso * st))


@pytest.mark.parametrize("d,H", [(8, 2), (4, 3)])
def test_backward_matches_finite_differences(d, H):
    rng = np.random.default_rng(19 + d)
    B, T = 2, 7
    q, k, v, g, s0 = make(rng, B, T, H, d, with_state=True)
    dy = rnd(rng, B, T, H, d)
    dso = rnd(rng, B, H, d, d)
    gam = oracle.gamma(H)
    off, base, eps = 11, 1e4, 1e-6
    grads = oracle.backward(q, k, v, g, gam, dy, s0, dso, pos_offset=off, base=base, eps=eps)
    names = ["q", "k", "v", "g", "s0"]
    arrays = [q, k, v, g, s0]
    step = 1e-6
    for name, arr, grad in zip(names, arrays, grads):
        fd = np.zeros_like(arr)
        it = np.nditer(arr, flags=["multi_index"])
        for _ in it:
            idx = it.multi_index
            args = [a.copy() for a in arrays]
            j = names.index(name)
            args[j][idx] += step
            lp = _loss(*args[:4], args[4], gam, dy, dso, off, base, eps)
            args[j][idx] -= 2 * step
            lm = _loss(*args[:4], args[4], gam, dy, dso, off, base, eps)
            fd[idx] = (lp - lm) / (2 * step)
        err = np.abs(fd - grad).max() / max(1e-3, np.abs(fd).max())
        assert err < 1e-6, (name, err)


def test_backward_without_state_terms():
    """dstate_out = None means zero upstream state gradient, S_0 = None zero state."""
    rng = np.random.default_rng(21)
    q, k, v, g, _ = make(rng, 1, 9, 2, 8)
    dy = rnd(rng, 1, 9, 2, 8)
    gam = oracle.gamma(2)
    a = oracle.backward(q, k, v, g, gam, dy)
    b = oracle.backward(q, k, v, g, gam, dy, np.zeros((1, 2, 8, 8)), np.zeros((1, 2, 8, 8)))
    for x, y_ in zip(a, b):
        np.testing.assert_array_equal(x, y_)
