"""Long segments: the tensor-core local-state passes read only the tiles
within the decay horizon (the weights beyond it sum to at most 2^-40), cut
into pieces of at most 48 tiles whose partial sums are added before the scan.  With 76 heads of 18000
tokens every head is two segments of 71 tiles (two pieces when every tile
counts); the forward pass sums the first segment and the state-gradient pass
the second.  Sampled heads, among them gamma = 1 (every tile, all pieces) and
gamma = 1e-6 (one tile), are checked in full against the oracle: outputs,
final state and gradients."""
import numpy as np
import pytest
import torch

import oracle
from rnn_sequence_mixer_gb300 import api, inputs
from parity_util import f64, max_rel_err

pytestmark = pytest.mark.gpu

B, T, H, D = 1, 18000, 76, 128
HEADS = [0, 1, 2, 30, 60, 75]  # gamma = 1, gamma = 1e-6, then the schedule


@pytest.fixture(scope="module")
def case():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    dev = torch.device("cuda:0")
    g = oracle.gamma(H).astype(np.float32)
    g[0], g[1] = 1.0, 1e-6
    inp = inputs.mixer_inputs(B, T, H, D, torch.bfloat16, 91, device=dev, with_dy=True)
    s0 = inputs.state(B, H, D, 92, 0.1, device=dev)
    return g, inp, s0


def _sel(t):
    return f64(torch.stack([t[0, :, h, :] for h in HEADS], dim=1).unsqueeze(0))


def test_forward_with_pieces(case):
    g, inp, s0 = case
    y, o, st = api.prefill(inp["q"], inp["k"], inp["v"], inp["gate"], torch.from_numpy(g), s0,
                           chunk=128, rope_base=1e6, want_o=True)
    torch.cuda.synchronize()
    gg = g[HEADS].astype(np.float64)
    s0h = f64(torch.stack([s0[0, h] for h in HEADS]).unsqueeze(0))
    ry, ro, rs = oracle.prefill(_sel(inp["q"]), _sel(inp["k"]), _sel(inp["v"]), _sel(inp["gate"]),
                                gg, s0h, base=1e6)
    assert max_rel_err(_sel(y), ry) <= 2e-2
    assert max_rel_err(_sel(o), ro) <= 2e-2
    sth = f64(torch.stack([st[0, h] for h in HEADS]).unsqueeze(0))
    assert max_rel_err(sth, rs, head_axes=(0, 1)) <= 2e-2


def test_backward_with_pieces(case):
    g, inp, s0 = case
    out = api.prefill_backward(inp["q"], inp["k"], inp["v"], inp["gate"], torch.from_numpy(g),
                               inp["dy"], s0, chunk=128, rope_base=1e6, want_dstate_in=True)
    torch.cuda.synchronize()
    gg = g[HEADS].astype(np.float64)
    s0h = f64(torch.stack([s0[0, h] for h in HEADS]).unsqueeze(0))
    ref = oracle.backward(_sel(inp["q"]), _sel(inp["k"]), _sel(inp["v"]), _sel(inp["gate"]), gg,
                          _sel(inp["dy"]), s0h, base=1e6)
    for name, got, want in zip(["dq", "dk", "dv", "dgate"], out[:4], ref[:4]):
        err = max_rel_err(_sel(got), want)
        assert err <= 2e-2, f"{name}: {err:.3e}"
    dsi = f64(torch.stack([out[4][0, h] for h in HEADS]).unsqueeze(0))
    assert max_rel_err(dsi, ref[4], head_axes=(0, 1)) <= 2e-2


def test_arbitrary_gammas_forward_and_backward():
    """Per-head gamma drawn over (0, 1] (not the paper's schedule): each head
    keeps a different number of tiles within its decay horizon, and pieces.  76 heads of
    14000 tokens are two segments of 55 tiles each; sampled heads against the
    oracle."""
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    dev = torch.device("cuda:0")
    B_, T_, H_ = 1, 14000, 76
    rng = np.random.default_rng(7)
    g = np.exp(-10.0 ** rng.uniform(-4.5, 1.0, size=H_)).astype(np.float32)  # 0.99997 .. 4.5e-5
    g[3] = 0.99999
    heads = [0, 3, 30, 50, 75]
    inp = inputs.mixer_inputs(B_, T_, H_, D, torch.bfloat16, 93, device=dev, with_dy=True)
    s0 = inputs.state(B_, H_, D, 94, 0.1, device=dev)
    dso = inputs.state(B_, H_, D, 95, 0.05, device=dev)
    gt = torch.from_numpy(g)
    y, o, st = api.prefill(inp["q"], inp["k"], inp["v"], inp["gate"], gt, s0, chunk=128,
                           rope_base=1e6, want_o=True)
    grads = api.prefill_backward(inp["q"], inp["k"], inp["v"], inp["gate"], gt, inp["dy"], s0, dso,
                                 chunk=128, rope_base=1e6, want_dstate_in=True)
    torch.cuda.synchronize()
    sel = lambda t: f64(torch.stack([t[0, :, h, :] for h in heads], dim=1).unsqueeze(0))
    selst = lambda t: f64(torch.stack([t[0, h] for h in heads]).unsqueeze(0))
    gg = g[heads].astype(np.float64)
    ry, ro, rs = oracle.prefill(sel(inp["q"]), sel(inp["k"]), sel(inp["v"]), sel(inp["gate"]), gg,
                                selst(s0), base=1e6)
    assert max_rel_err(sel(y), ry) <= 2e-2
    assert max_rel_err(sel(o), ro) <= 2e-2
    assert max_rel_err(selst(st), rs, head_axes=(0, 1)) <= 2e-2
    ref = oracle.backward(sel(inp["q"]), sel(inp["k"]), sel(inp["v"]), sel(inp["gate"]), gg,
                          sel(inp["dy"]), selst(s0), selst(dso), base=1e6)
    for name, got, want in zip(["dq", "dk", "dv", "dgate"], grads[:4], ref[:4]):
        err = max_rel_err(sel(got), want)
        assert err <= 2e-2, f"{name}: {err:.3e}"
    assert max_rel_err(selst(grads[4]), ref[4], head_axes=(0, 1)) <= 2e-2
