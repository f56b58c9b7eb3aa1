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
    (1, 1000, 4, 128, torch.bfloat16, 128, True, 77),
    (3, 333, 5, 128, torch.bfloat16, 128, True, 5),
    (1, 64, 2, 128, torch.bfloat16, 64, True, 0),
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


def test_backward_gamma_one_head(dev):
    """gamma = 1 (no decay: plain linear attention) next to the fastest head of H = 32."""
    g = oracle.gamma(32)[:2].astype(np.float32).copy()
    g[1] = 1.0
    B, T, H, d = 1, 700, 2, 128
    inp = inputs.mixer_inputs(B, T, H, d, torch.bfloat16, 61, device=dev, with_dy=True)
    out = api.prefill_backward(inp["q"], inp["k"], inp["v"], inp["gate"], torch.from_numpy(g),
                               inp["dy"], chunk=128, rope_base=1e6, want_dstate_in=True)
    torch.cuda.synchronize()
    ref = oracle.backward(f64(inp["q"]), f64(inp["k"]), f64(inp["v"]), f64(inp["gate"]),
                          g.astype(np.float64), f64(inp["dy"]), base=1e6)
    for name, got, want in zip(["dq", "dk", "dv", "dgate"], out[:4], ref[:4]):
        err = max_rel_err(f64(got), want)
        assert err <= 2e-2, f"{name}: {err:.3e}"
    assert max_rel_err(f64(out[4]), ref[4], head_axes=(0, 1)) <= 2e-2


def test_backward_status_word_is_clear(dev):
    """The backward workspace ends with the same device status word as the
    forward's: cleared by the call, 0 when no bounded wait gave up."""
    B, T, H, d = 1, 2000, 4, 128
    inp = inputs.mixer_inputs(B, T, H, d, torch.bfloat16, 62, device=dev, with_dy=True)
    shape = api.make_shape(B, T, H, d, chunk=128, dtype=torch.bfloat16)
    n = api.backward_workspace_size(shape)
    ws = torch.full((n,), 0xAB, dtype=torch.uint8, device=dev)
    api.prefill_backward(inp["q"], inp["k"], inp["v"], inp["gate"],
                         torch.from_numpy(oracle.gamma(H).astype(np.float32)), inp["dy"],
                         chunk=128, workspace=ws)
    torch.cuda.synchronize()
    assert ws[n - 256:n - 252].view(torch.int32).item() == 0


@pytest.mark.parametrize("B,T", [(2, 0), (0, 7)])
def test_backward_of_an_empty_sequence_passes_the_state_gradient(dev, B, T):
    H, d = 2, 128
    inp = inputs.mixer_inputs(B, T, H, d, torch.bfloat16, 8, device=dev, with_dy=True)
    dso = inputs.state(B, H, d, 9, 0.05, device=dev)
    out = api.prefill_backward(inp["q"], inp["k"], inp["v"], inp["gate"],
                               torch.from_numpy(oracle.gamma(H).astype(np.float32)), inp["dy"],
                               None, dso, chunk=128, want_dstate_in=True)
    torch.cuda.synchronize()
    assert torch.equal(out[4], dso)
    assert all(t.numel() == 0 for t in out[:4])


def test_backward_large_magnitudes(dev):
    """The tensor-core backward with q, k, v scaled by 1e2 / 1e2 / 1e3, gates of
    +-20 and a large upstream gradient."""
    B, T, H, d = 1, 600, 4, 128
    g = oracle.gamma(H).astype(np.float32)
    inp = inputs.mixer_inputs(B, T, H, d, torch.float32, 73, device=dev, with_dy=True)
    for k, sc in (("q", 100.0), ("k", 100.0), ("v", 1000.0), ("gate", 20.0), ("dy", 50.0)):
        inp[k] *= sc
    inp = {k: v.to(torch.bfloat16) for k, v in inp.items()}
    out = api.prefill_backward(inp["q"], inp["k"], inp["v"], inp["gate"], torch.from_numpy(g),
                               inp["dy"], chunk=128, rope_base=1e6, want_dstate_in=True)
    torch.cuda.synchronize()
    ref = oracle.backward(f64(inp["q"]), f64(inp["k"]), f64(inp["v"]), f64(inp["gate"]),
                          g.astype(np.float64), f64(inp["dy"]), base=1e6)
    for name, got, want in zip(["dq", "dk", "dv", "dgate"], out[:4], ref[:4]):
        assert torch.isfinite(got.float()).all(), name
        err = max_rel_err(f64(got), want)
        assert err <= 2e-2, f"{name}: {err:.3e}"
    assert max_rel_err(f64(out[4]), ref[4], head_axes=(0, 1)) <= 2e-2


@pytest.mark.parametrize("B,T,H,d,dtype,chunk", [
    (2, 90, 3, 64, torch.float32, 64),       # CUDA-core passes
    (3, 1000, 8, 128, torch.bfloat16, 128),  # tensor-core passes, several segments, ragged tail
])
def test_backward_reads_forward_states(dev, B, T, H, d, dtype, chunk):
    """The backward given the forward's workspace skips recomputing the segment
    states and must give the same gradients, bit for bit, as the one that
    recomputes them (the same kernels produced both), and match the oracle."""
    g = oracle.gamma(H).astype(np.float32)
    gt = torch.from_numpy(g)
    inp = inputs.mixer_inputs(B, T, H, d, dtype, 70 + T, device=dev, with_dy=True)
    s0 = inputs.state(B, H, d, 71, 0.1, device=dev)
    dso = inputs.state(B, H, d, 72, 0.05, device=dev)
    kw = dict(chunk=chunk, pos_offset=3, rope_base=1e6)
    shape = api.make_shape(B, T, H, d, dtype=dtype, **kw)
    wsf = torch.empty(api.prefill_workspace_size(shape), dtype=torch.uint8, device=dev)
    api.prefill(inp["q"], inp["k"], inp["v"], inp["gate"], gt, s0, workspace=wsf, **kw)
    saved = api.prefill_backward(inp["q"], inp["k"], inp["v"], inp["gate"], gt, inp["dy"], s0, dso,
                                 want_dstate_in=True, fwd_workspace=wsf, **kw)
    fresh = api.prefill_backward(inp["q"], inp["k"], inp["v"], inp["gate"], gt, inp["dy"], s0, dso,
                                 want_dstate_in=True, **kw)
    torch.cuda.synchronize()
    for name, a, b in zip(["dq", "dk", "dv", "dgate", "dstate_in"], saved, fresh):
        assert torch.equal(a, b), name
    ref = oracle.backward(f64(inp["q"]), f64(inp["k"]), f64(inp["v"]), f64(inp["gate"]),
                          g.astype(np.float64), f64(inp["dy"]), f64(s0), f64(dso), pos_offset=3,
                          base=1e6)
    tol = tol_for(dtype)
    for name, got, want in zip(["dq", "dk", "dv", "dgate"], saved[:4], ref[:4]):
        err = max_rel_err(f64(got), want)
        assert err <= tol, f"{name}: {err:.3e}"
