"""The tensor-core prefill in one launch (hla_shape.passes = 1): every output
CTA forms the state entering its segment from the decay window before it
(weights whose tail beyond it sums to at most 2^-40; every earlier token when
gamma = 1), with no local-state pass, no scan and no CTA waiting for another.
Checked against the oracle at shapes with several segments, ragged tails,
state in, chunk 64 and 128, gamma = 1 and gamma near 0 heads; against the
three-pass path; with saved features for the backward; from given features;
and through the backward reading its workspace."""
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


def gammas(H, special=True):
    g = oracle.gamma(H).astype(np.float32)
    if special and H >= 3:
        g[0], g[1] = 1.0, 1e-6
    return g


@pytest.mark.parametrize("B,T,H,chunk,pos,with_state", [
    (1, 2500, 16, 64, 0, False),      # 8 segments of 320 tokens
    (2, 3001, 3, 128, 77, True),      # ragged tail, gamma = 1 and gamma = 1e-6 heads
    (1, 9000, 4, 128, 123456, True),  # long windows for the slow heads
    (3, 700, 5, 64, 5, True),
])
def test_one_launch_matches_oracle(dev, B, T, H, chunk, pos, with_state):
    d = 128
    g = gammas(H)
    gt = torch.from_numpy(g)
    inp = inputs.mixer_inputs(B, T, H, d, torch.bfloat16, 300 + T, device=dev)
    s0 = inputs.state(B, H, d, 301, 0.1, device=dev) if with_state else None
    shape = api.make_shape(B, T, H, d, chunk=chunk, passes=1)
    assert api.prefill_launches(shape, g) == 1
    y, o, st = api.prefill(inp["q"], inp["k"], inp["v"], inp["gate"], gt, s0, chunk=chunk,
                           pos_offset=pos, rope_base=1e6, want_o=True, passes=1)
    y3, o3, st3 = api.prefill(inp["q"], inp["k"], inp["v"], inp["gate"], gt, s0, chunk=chunk,
                              pos_offset=pos, rope_base=1e6, want_o=True, passes=3)
    torch.cuda.synchronize()
    ry, ro, rs = oracle.prefill(f64(inp["q"]), f64(inp["k"]), f64(inp["v"]), f64(inp["gate"]),
                                g.astype(np.float64), None if s0 is None else f64(s0),
                                pos_offset=pos, base=1e6)
    assert max_rel_err(f64(o), ro) <= TOL
    assert max_rel_err(f64(y), ry) <= TOL
    assert max_rel_err(f64(st), rs, head_axes=(0, 1)) <= TOL
    # the two launch plans agree with each other as closely as each with the oracle
    assert max_rel_err(f64(o), f64(o3)) <= TOL
    assert max_rel_err(f64(st), f64(st3), head_axes=(0, 1)) <= TOL


def test_one_launch_workspace_states_feed_the_backward(dev):
    """The one-launch forward writes the state entering every segment to its
    workspace and saves the features; the backward reading both matches the
    oracle's gradients."""
    B, T, H, d, chunk = 2, 2000, 4, 128, 64
    g = gammas(H)
    gt = torch.from_numpy(g)
    inp = inputs.mixer_inputs(B, T, H, d, torch.bfloat16, 320, device=dev, with_dy=True)
    s0 = inputs.state(B, H, d, 321, 0.1, device=dev)
    shape = api.make_shape(B, T, H, d, chunk=chunk, rope_base=1e6)
    wsf = torch.empty(api.prefill_workspace_size(shape), dtype=torch.uint8, device=dev)
    ws3 = torch.empty_like(wsf)
    sv = torch.empty(api.saved_bytes(shape), dtype=torch.uint8, device=dev)
    api.prefill(inp["q"], inp["k"], inp["v"], inp["gate"], gt, s0, chunk=chunk, rope_base=1e6,
                workspace=ws3, passes=3)
    y, _, _ = api.prefill(inp["q"], inp["k"], inp["v"], inp["gate"], gt, s0, chunk=chunk,
                          rope_base=1e6, workspace=wsf, saved=sv, passes=1)
    grads = api.prefill_backward(inp["q"], inp["k"], inp["v"], inp["gate"], gt, inp["dy"], s0,
                                 chunk=chunk, rope_base=1e6, want_dstate_in=True,
                                 fwd_workspace=wsf, saved=sv)
    torch.cuda.synchronize()
    # the entering states of the two plans (fp32 [B, H, nseg, d, d] at the start)
    n = (wsf.numel() - 256) // 4
    nseg = n // (B * H * d * d)
    a = wsf[: 4 * B * H * nseg * d * d].view(torch.float32).view(B * H * nseg, d, d)
    b = ws3[: 4 * B * H * nseg * d * d].view(torch.float32).view(B * H * nseg, d, d)
    assert max_rel_err(f64(a)[None], f64(b)[None], head_axes=(0, 1)) <= TOL
    ry, _, _ = oracle.prefill(f64(inp["q"]), f64(inp["k"]), f64(inp["v"]), f64(inp["gate"]),
                              g.astype(np.float64), f64(s0), base=1e6)
    assert max_rel_err(f64(y), ry) <= TOL
    ref = oracle.backward(f64(inp["q"]), f64(inp["k"]), f64(inp["v"]), f64(inp["gate"]),
                          g.astype(np.float64), f64(inp["dy"]), f64(s0), base=1e6)
    for got, want in zip(grads[:4], ref[:4]):
        assert max_rel_err(f64(got), want) <= TOL
    assert max_rel_err(f64(grads[4]), ref[4], head_axes=(0, 1)) <= TOL


def test_one_launch_from_given_features(dev):
    """prefill_features in one launch (the window's k~ read from the features)."""
    B, T, D, H, d = 1, 3000, 256, 4, 128
    w = inputs.layer_inputs(B, T, D, H, d, 330, device=dev)
    g = gammas(H)
    feat, v, gate = api.project_in(w["x"], w["w_qkvz"], rope_base=1e6)
    y, o, st = api.prefill_features(feat, v, gate, torch.from_numpy(g), chunk=128, rope_base=1e6,
                                    want_o=True, passes=1)
    torch.cuda.synchronize()
    q, k, rv, rg = oracle.project_in(f64(w["x"]), f64(w["w_qkvz"]))
    ry, ro, rs = oracle.prefill(q, k, rv, rg, g.astype(np.float64), base=1e6)
    assert max_rel_err(f64(o), ro) <= TOL
    assert max_rel_err(f64(y), ry) <= TOL
    assert max_rel_err(f64(st), rs, head_axes=(0, 1)) <= TOL
