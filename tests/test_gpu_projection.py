"""GPU parity of the projections around the RNN mixer (Appendix A, Eq. 18)
against the fp64 oracle: hla_project_in (x W_q,k,v,z with the feature map in
its epilogue), hla_prefill_features (the mixer from those features),
hla_project_out (u W_o^T) and the backward from the features, alone and
chained into one layer.  Shapes span several 128-row and 256-column tiles,
ragged row tails and K rings that wrap many times."""
import numpy as np
import pytest
import torch

import oracle
from rnn_sequence_mixer_gb300 import api, inputs
from parity_util import f64, max_rel_err

pytestmark = pytest.mark.gpu
TOL = 2e-2


@pytest.fixture(scope="module")
def dev():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return torch.device("cuda:0")


def split_features(feat, B, T, H, d):
    """The saved layout as (q~, k~ [B, T, H, d], rq, rk, diag [B, H, T]) in fp64."""
    n = B * T * H * d
    q = feat[: 2 * n].view(torch.float16).view(B, T, H, d)
    k = feat[2 * n: 4 * n].view(torch.float16).view(B, T, H, d)
    sc = feat[4 * n: 4 * n + 12 * B * T * H].view(torch.float32).view(3, B, H, T)
    return f64(q), f64(k), f64(sc[0]), f64(sc[1]), f64(sc[2])


@pytest.mark.parametrize("B,T,D,H,pos", [
    (2, 300, 256, 2, 0),        # 600 rows: 5 row tiles, the last of 88 rows
    (1, 1000, 2048, 4, 12345),  # 32 K blocks per tile
    (3, 77, 64, 1, 7),          # one K block, 231 rows
])
def test_project_in_matches_oracle(dev, B, T, D, H, pos):
    d = 128
    w = inputs.layer_inputs(B, T, D, H, d, 100 + T, device=dev)
    feat, v, gate = api.project_in(w["x"], w["w_qkvz"], pos_offset=pos, rope_base=1e6)
    torch.cuda.synchronize()
    q, k, rv, rg = oracle.project_in(f64(w["x"]), f64(w["w_qkvz"]))
    rqt, rkt, rrq, rrk, rdiag = oracle.features(q, k, pos_offset=pos, base=1e6)
    gq, gk, grq, grk, gdiag = split_features(feat, B, T, H, d)
    assert max_rel_err(f64(v), rv) <= TOL
    assert max_rel_err(f64(gate), rg) <= TOL
    assert max_rel_err(gq, rqt) <= TOL
    assert max_rel_err(gk, rkt) <= TOL
    for got, want in ((grq, rrq), (grk, rrk), (gdiag, rdiag)):
        assert max_rel_err(got[..., None], want[..., None], head_axes=(0, 1)) <= TOL


@pytest.mark.parametrize("M,n_in,D", [(600, 256, 256), (1000, 2048, 384), (5, 64, 128)])
def test_project_out_matches_oracle(dev, M, n_in, D):
    gen = inputs.generator(7 + M, dev)
    u = inputs.normal((M, n_in), torch.bfloat16, gen, dev)
    w_o = (torch.randn((D, n_in), generator=gen, device=dev) / n_in ** 0.5).to(torch.bfloat16)
    out = api.project_out(u, w_o)
    torch.cuda.synchronize()
    ref = oracle.matmul_nt(f64(u), f64(w_o))
    # rows as [1, M, 1, D] so the slice is the whole matrix
    assert max_rel_err(f64(out)[None, :, None, :], ref[None, :, None, :]) <= TOL


@pytest.mark.parametrize("B,T,D,H,chunk,with_state", [
    (1, 700, 256, 2, 128, False),
    (2, 300, 512, 3, 64, True),
])
def test_layer_forward_and_backward_from_features(dev, B, T, D, H, chunk, with_state):
    """x -> project_in -> prefill_features -> project_out against the oracle's
    chain, and the backward from the same features (q = k = None) against the
    oracle's gradients of the projected q, k, v and gate."""
    d = 128
    w = inputs.layer_inputs(B, T, D, H, d, 200 + T, device=dev, with_dy=True)
    g = oracle.gamma(H).astype(np.float32)
    s0 = inputs.state(B, H, d, 201, 0.1, device=dev) if with_state else None
    feat, v, gate = api.project_in(w["x"], w["w_qkvz"], rope_base=1e6)
    y, o, st = api.prefill_features(feat, v, gate, torch.from_numpy(g), s0, chunk=chunk,
                                    rope_base=1e6, want_o=True)
    out = api.project_out(y, w["w_o"])
    dq, dk, dv, dg, dsi = api.prefill_backward(None, None, v, gate, torch.from_numpy(g), w["dy"], s0,
                                               chunk=chunk, rope_base=1e6, saved=feat,
                                               want_dstate_in=True)
    torch.cuda.synchronize()
    q, k, rv, rg = oracle.project_in(f64(w["x"]), f64(w["w_qkvz"]))
    s0h = None if s0 is None else f64(s0)
    ry, ro, rs = oracle.prefill(q, k, rv, rg, g.astype(np.float64), s0h, base=1e6)
    assert max_rel_err(f64(o), ro) <= TOL
    assert max_rel_err(f64(y), ry) <= TOL
    assert max_rel_err(f64(st), rs, head_axes=(0, 1)) <= TOL
    rout = oracle.project_out(f64(y), f64(w["w_o"]))  # the projection of the GPU's own y
    assert max_rel_err(f64(out)[:, :, None, :], rout[:, :, None, :]) <= TOL
    rout_chain = oracle.project_out(ry, f64(w["w_o"]))  # and of the oracle's y
    assert max_rel_err(f64(out)[:, :, None, :], rout_chain[:, :, None, :]) <= TOL
    ref = oracle.backward(q, k, rv, rg, g.astype(np.float64), f64(w["dy"]), s0h, base=1e6)
    for got, want in zip((dq, dk, dv, dg), ref[:4]):
        assert max_rel_err(f64(got), want) <= TOL
    assert max_rel_err(f64(dsi), ref[4], head_axes=(0, 1)) <= TOL
    # the same backward from the layer's y: prefill_features wrote 1/RMS(o) into
    # the features, and the dq pass takes the normalized output from y
    from_y = api.prefill_backward(None, None, v, gate, torch.from_numpy(g), w["dy"], s0,
                                  chunk=chunk, rope_base=1e6, saved=feat, y=y,
                                  want_dstate_in=True)
    torch.cuda.synchronize()
    for got, want in zip(from_y[:4], ref[:4]):
        assert max_rel_err(f64(got), want) <= TOL
    assert max_rel_err(f64(from_y[4]), ref[4], head_axes=(0, 1)) <= TOL


def test_prefill_features_matches_the_saving_prefill(dev):
    """The features an hla_prefill call saves, given back to
    hla_prefill_features, reproduce that call's outputs (both against the
    oracle)."""
    B, T, H, d = 1, 1500, 4, 128
    inp = inputs.mixer_inputs(B, T, H, d, torch.bfloat16, 31, device=dev)
    g = oracle.gamma(H).astype(np.float32)
    gt = torch.from_numpy(g)
    shape = api.make_shape(B, T, H, d, chunk=128, rope_base=1e6)
    saved = torch.empty(api.saved_bytes(shape), dtype=torch.uint8, device=dev)
    y1, _, s1 = api.prefill(inp["q"], inp["k"], inp["v"], inp["gate"], gt, chunk=128,
                            rope_base=1e6, saved=saved)
    y2, _, s2 = api.prefill_features(saved, inp["v"], inp["gate"], gt, chunk=128, rope_base=1e6)
    torch.cuda.synchronize()
    ry, _, rs = oracle.prefill(f64(inp["q"]), f64(inp["k"]), f64(inp["v"]), f64(inp["gate"]),
                               g.astype(np.float64), base=1e6)
    for y, s in ((y1, s1), (y2, s2)):
        assert max_rel_err(f64(y), ry) <= TOL
        assert max_rel_err(f64(s), rs, head_axes=(0, 1)) <= TOL
    assert max_rel_err(f64(y2), f64(y1)) <= 1e-2
