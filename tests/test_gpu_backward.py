"""GPU parity of hla_prefill_backward against the fp64 oracle's chain rule."""
import numpy as np
import pytest
import torch

import oracle
from rnn_sequence_mixer_gb300 import api, inputs, workloads
from parity_util import f64, max_rel_err, tol_for

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return torch.device("cuda:0")


@pytest.mark.parametrize("B,T,H,d,dtype,chunk,with_state,pos", [
    (1, 1, 2, 64, torch.float32, 64, True, 0),
    (2, 90, 3, 64, torch.float32, 64, True, 11),
    (1, 260, 2, 128, torch.float32, 128, False, 0),
    (2, 200, 4, 128, torch.bfloat16, 64, True, 1000),
    (1, 1500, 16, 128, torch.bfloat16, 64, False, 0),
])
def test_backward_small(dev, B, T, H, d, dtype, chunk, with_state, pos):
    g = oracle.gamma(H).astype(np.float32)
    inp = inputs.mixer_inputs(B, T, H, d, dtype, 50 + T, device=dev, with_dy=True)
    s0 = inputs.state(B, H, d, 51, 0.1, device=dev) if with_state else None
    dso = inputs.state(B, H, d, 52, 0.05, device=dev) if with_state else None
    out = api.prefill_backward(inp["q"], inp["k"], inp["v"], inp["gate"], torch.from_numpy(g),
                               inp["dy"], s0, dso, chunk=chunk, pos_offset=pos, rope_base=1e6,
                               want_dstate_in=True)
    torch.cuda.synchronize()
    ref = oracle.backward(f64(inp["q"]), f64(inp["k"]), f64(inp["v"]), f64(inp["gate"]),
                          g.astype(np.float64), f64(inp["dy"]), None if s0 is None else f64(s0),
                          None if dso is None else f64(dso), pos_offset=pos, base=1e6)
    tol = tol_for(dtype)
    for name, got, want in zip(["dq", "dk", "dv", "dgate"], out[:4], ref[:4]):
        err = max_rel_err(f64(got), want)
        assert err <= tol, f"{name}: {err:.3e}"
    err = max_rel_err(f64(out[4]), ref[4], head_axes=(0, 1))
    assert err <= tol, f"dstate_in: {err:.3e}"


def test_fwd_bwd_workload_sampled(dev):
    """B=8, T=16384, H=32 distillation-shaped backward; sampled heads in full."""
    w = workloads.FWD_BWD_16K
    g = oracle.gamma(w.H).astype(np.float32)
    inp = inputs.mixer_inputs(w.B, w.T, w.H, w.d, w.dtype, w.seed, device=dev, with_dy=True)
    out = api.prefill_backward(inp["q"], inp["k"], inp["v"], inp["gate"], torch.from_numpy(g),
                               inp["dy"], chunk=w.chunk, rope_base=w.rope_base, eps=w.eps)
    torch.cuda.synchronize()
    pairs = [(0, 0), (2, 9), (5, 20), (7, 31)]
    gg = np.array([float(g[h]) for (_, h) in pairs])
    sel = lambda t: f64(torch.stack([t[b, :, h, :] for (b, h) in pairs], dim=1).unsqueeze(0))
    ref = oracle.backward(sel(inp["q"]), sel(inp["k"]), sel(inp["v"]), sel(inp["gate"]), gg,
                          sel(inp["dy"]), base=w.rope_base, eps=w.eps)
    for name, got, want in zip(["dq", "dk", "dv", "dgate"], out[:4], ref[:4]):
        err = max_rel_err(sel(got), want)
        assert err <= 2e-2, f"{name}: {err:.3e}"
