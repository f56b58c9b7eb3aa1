"""GPU parity of the saved-feature path: hla_prefill writing q~, k~ and the row
norms for the backward (the `saved` buffer), and hla_prefill_backward reading
them instead of recomputing the feature map, against the fp64 oracle."""
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


def split_saved(sv, B, T, H, d):
    """The documented layout: fp16 q~ and k~ [B, T, H, d], then fp32 [4, B, H, T]."""
    n = B * T * H * d
    qt = sv[:2 * n].view(torch.float16).view(B, T, H, d)
    kt = sv[2 * n:4 * n].view(torch.float16).view(B, T, H, d)
    sc = sv[4 * n:4 * n + 16 * B * T * H].view(torch.float32).view(4, B, H, T)
    return qt, kt, sc


# (B, T, H, chunk, pos_offset): chunk 64 (rows past the chunk in the 128-row
# tiles), several segments with a ragged tail, one exact tile, T below a tile,
# a single token
CASES = [
    (1, 300, 2, 64, 0),
    (2, 1000, 3, 128, 5),
    (1, 128, 2, 128, 0),
    (3, 777, 5, 64, 1000),
    (1, 5, 2, 128, 0),
    (2, 1, 1, 64, 7),
]


@pytest.mark.parametrize("B,T,H,chunk,pos", CASES)
def test_forward_saves_features(dev, B, T, H, chunk, pos):
    """o and the state are bit-identical with and without saving, and y within
    a bf16 step (saving, the gate takes the sigmoid form the backward can
    divide y by again, 1 / (1 + 2^(-z log2 e)), which can round differently
    from 0.5 + 0.5 tanh(z / 2)); every saved row matches the oracle's
    feature map within its fp16 rounding, and
    the norms and the q~ . k~ diagonal match it in fp32, and the output norm's
    1/RMS(o) matches the pass's own fp32 o (and the oracle's o)."""
    d, eps, base = 128, 1e-6, 1e6
    g = torch.from_numpy(oracle.gamma(H).astype(np.float32))
    inp = inputs.mixer_inputs(B, T, H, d, torch.bfloat16, 90 + T, device=dev)
    s0 = inputs.state(B, H, d, 91, 0.1, device=dev)
    kw = dict(chunk=chunk, pos_offset=pos, rope_base=base, eps=eps, want_o=True)
    shape = api.make_shape(B, T, H, d, chunk=chunk, dtype=torch.bfloat16)
    sv = torch.full((api.saved_bytes(shape),), 0xFF, dtype=torch.uint8, device=dev)
    ref_run = api.prefill(inp["q"], inp["k"], inp["v"], inp["gate"], g, s0, **kw)
    run = api.prefill(inp["q"], inp["k"], inp["v"], inp["gate"], g, s0, saved=sv, **kw)
    torch.cuda.synchronize()
    for name, a, b in zip(["o", "state_out"], run[1:], ref_run[1:]):
        assert torch.equal(a, b), name
    assert max_rel_err(f64(run[0]), f64(ref_run[0])) <= 1e-2, "y"
    qt, kt, sc = split_saved(sv, B, T, H, d)
    qt, kt, sc = f64(qt), f64(kt), f64(sc)
    assert np.isfinite(qt).all() and np.isfinite(kt).all() and np.isfinite(sc).all()
    q64, k64 = f64(inp["q"]), f64(inp["k"])
    for b in range(B):
        for t in range(T):
            for h in range(H):
                wq = oracle.feature(q64[b, t, h], pos + t, base, eps)
                wk = oracle.feature(k64[b, t, h], pos + t, base, eps, 1.0 / np.sqrt(d))
                for name, got, want in (("q~", qt[b, t, h], wq), ("k~", kt[b, t, h], wk)):
                    bound = 6e-4 * np.abs(want) + 2e-5 * np.abs(want).max()
                    assert (np.abs(got - want) <= bound).all(), (name, b, t, h)
                # RMSNorm keeps direction: 1 / RMS(x) = |Norm(x)| / |x|
                rq = np.linalg.norm(wq) / np.linalg.norm(q64[b, t, h])
                rk = np.linalg.norm(wk) * np.sqrt(d) / np.linalg.norm(k64[b, t, h])
                assert abs(sc[0, b, h, t] - rq) <= 1e-5 * rq, ("rq", b, t, h)
                assert abs(sc[1, b, h, t] - rk) <= 1e-5 * rk, ("rk", b, t, h)
                scale = np.linalg.norm(wq) * np.linalg.norm(wk)
                assert abs(sc[2, b, h, t] - wq @ wk) <= 2e-5 * scale, ("diag", b, t, h)
    o_gpu = f64(run[1])
    ro_gpu = 1.0 / np.sqrt((o_gpu ** 2).mean(axis=-1) + eps)  # [B, T, H]
    ro_got = sc[3].transpose(0, 2, 1)
    assert np.abs(ro_got - ro_gpu).max() <= 1e-5 * np.abs(ro_gpu).max(), "1/RMS(o)"
    _, o_ref, _ = oracle.prefill(f64(inp["q"]), f64(inp["k"]), f64(inp["v"]), f64(inp["gate"]),
                                 g.numpy().astype(np.float64), f64(s0), pos_offset=pos, base=base,
                                 eps=eps)
    ro_ref = 1.0 / np.sqrt((o_ref ** 2).mean(axis=-1) + eps)
    assert (np.abs(ro_got - ro_ref) <= 2e-2 * ro_ref).all(), "1/RMS(o) against the oracle"


@pytest.mark.parametrize("B,T,H,chunk,pos,with_state", [
    (1, 300, 2, 64, 0, False),
    (2, 1000, 3, 128, 5, True),
    (3, 777, 5, 64, 1000, True),
    (1, 5, 2, 128, 0, True),
    (1, 1500, 16, 128, 0, False),
])
def test_backward_reads_saved_features(dev, B, T, H, chunk, pos, with_state):
    """The backward reading the saved features (and the forward's segment
    states) matches the oracle, as does the one that recomputes them."""
    d = 128
    g = oracle.gamma(H).astype(np.float32)
    gt = torch.from_numpy(g)
    inp = inputs.mixer_inputs(B, T, H, d, torch.bfloat16, 95 + T, device=dev, with_dy=True)
    s0 = inputs.state(B, H, d, 96, 0.1, device=dev) if with_state else None
    dso = inputs.state(B, H, d, 97, 0.05, device=dev) if with_state else None
    kw = dict(chunk=chunk, pos_offset=pos, rope_base=1e6)
    shape = api.make_shape(B, T, H, d, dtype=torch.bfloat16, **kw)
    wsf = torch.empty(api.prefill_workspace_size(shape), dtype=torch.uint8, device=dev)
    sv = torch.empty(api.saved_bytes(shape), dtype=torch.uint8, device=dev)
    api.prefill(inp["q"], inp["k"], inp["v"], inp["gate"], gt, s0, workspace=wsf, saved=sv, **kw)
    with_saved = api.prefill_backward(inp["q"], inp["k"], inp["v"], inp["gate"], gt, inp["dy"], s0,
                                      dso, want_dstate_in=True, fwd_workspace=wsf, saved=sv, **kw)
    saved_only = api.prefill_backward(inp["q"], inp["k"], inp["v"], inp["gate"], gt, inp["dy"], s0,
                                      dso, want_dstate_in=True, saved=sv, **kw)
    torch.cuda.synchronize()
    # the segment states do not depend on where they came from: bit for bit
    for name, a, b in zip(["dq", "dk", "dv", "dgate", "dstate_in"], with_saved, saved_only):
        assert torch.equal(a, b), name
    ref = oracle.backward(f64(inp["q"]), f64(inp["k"]), f64(inp["v"]), f64(inp["gate"]),
                          g.astype(np.float64), f64(inp["dy"]),
                          None if s0 is None else f64(s0), None if dso is None else f64(dso),
                          pos_offset=pos, base=1e6)
    tol = tol_for(torch.bfloat16)
    for name, got, want in zip(["dq", "dk", "dv", "dgate"], with_saved[:4], ref[:4]):
        err = max_rel_err(f64(got), want)
        assert err <= tol, f"{name}: {err:.3e}"
    err = max_rel_err(f64(with_saved[4]), ref[4], head_axes=(0, 1))
    assert err <= tol, f"dstate_in: {err:.3e}"


def test_fwd_bwd_workload_saved_features_sampled(dev):
    """B=8, T=16384, H=32 forward + backward as the benchmark runs it (segment
    states and features saved by the forward); sampled heads in full."""
    w = workloads.FWD_BWD_16K
    g = oracle.gamma(w.H).astype(np.float32)
    gt = torch.from_numpy(g)
    inp = inputs.mixer_inputs(w.B, w.T, w.H, w.d, w.dtype, w.seed, device=dev, with_dy=True)
    kw = dict(chunk=w.chunk, rope_base=w.rope_base, eps=w.eps)
    shape = api.make_shape(w.B, w.T, w.H, w.d, dtype=w.dtype, **kw)
    wsf = torch.empty(api.prefill_workspace_size(shape), dtype=torch.uint8, device=dev)
    sv = torch.empty(api.saved_bytes(shape), dtype=torch.uint8, device=dev)
    api.prefill(inp["q"], inp["k"], inp["v"], inp["gate"], gt, want_state=False, workspace=wsf,
                saved=sv, **kw)
    out = api.prefill_backward(inp["q"], inp["k"], inp["v"], inp["gate"], gt, inp["dy"],
                               fwd_workspace=wsf, saved=sv, **kw)
    torch.cuda.synchronize()
    del sv, wsf
    pairs = [(0, 0), (3, 14), (6, 27), (7, 31)]
    gg = np.array([float(g[h]) for (_, h) in pairs])
    sel = lambda t: f64(torch.stack([t[b, :, h, :] for (b, h) in pairs], dim=1).unsqueeze(0))
    ref = oracle.backward(sel(inp["q"]), sel(inp["k"]), sel(inp["v"]), sel(inp["gate"]), gg,
                          sel(inp["dy"]), base=w.rope_base, eps=w.eps)
    for name, got, want in zip(["dq", "dk", "dv", "dgate"], out[:4], ref[:4]):
        err = max_rel_err(sel(got), want)
        assert err <= 2e-2, f"{name}: {err:.3e}"


@pytest.mark.parametrize("B,T", [(2, 0), (0, 7)])
def test_saved_features_of_an_empty_batch_or_sequence(dev, B, T):
    """No rows: a saved buffer is accepted and nothing is written; the states
    pass through as without one."""
    H, d = 2, 128
    g = torch.from_numpy(oracle.gamma(H).astype(np.float32))
    inp = inputs.mixer_inputs(B, T, H, d, torch.bfloat16, 8, device=dev, with_dy=True)
    s0 = inputs.state(B, H, d, 9, 0.1, device=dev)
    dso = inputs.state(B, H, d, 10, 0.05, device=dev)
    sv = torch.full((16,), 0x5A, dtype=torch.uint8, device=dev)
    _, _, st = api.prefill(inp["q"], inp["k"], inp["v"], inp["gate"], g, s0, chunk=128, saved=sv)
    out = api.prefill_backward(inp["q"], inp["k"], inp["v"], inp["gate"], g, inp["dy"], s0, dso,
                               chunk=128, want_dstate_in=True, saved=sv)
    torch.cuda.synchronize()
    assert torch.equal(st, s0)
    assert torch.equal(out[4], dso)
    assert bool((sv == 0x5A).all())


@pytest.mark.parametrize("B,T,H,chunk,pos,with_state", [
    (1, 300, 2, 64, 0, False),
    (2, 1000, 3, 128, 5, True),
    (3, 777, 5, 64, 1000, True),
    (1, 128, 2, 128, 0, False),
    (1, 1500, 16, 128, 0, False),
    (2, 1, 1, 64, 7, True),
])
def test_backward_from_forward_output(dev, B, T, H, chunk, pos, with_state):
    """Given the forward's y, the dq pass takes the normalized output from y
    (with the saved 1/RMS(o)) instead of recomputing o: the gradients match
    the oracle, and the recomputing path within the bf16 rounding of y."""
    d = 128
    g = oracle.gamma(H).astype(np.float32)
    gt = torch.from_numpy(g)
    inp = inputs.mixer_inputs(B, T, H, d, torch.bfloat16, 190 + T, device=dev, with_dy=True)
    s0 = inputs.state(B, H, d, 191, 0.1, device=dev) if with_state else None
    dso = inputs.state(B, H, d, 192, 0.05, device=dev) if with_state else None
    kw = dict(chunk=chunk, pos_offset=pos, rope_base=1e6)
    shape = api.make_shape(B, T, H, d, dtype=torch.bfloat16, **kw)
    wsf = torch.empty(api.prefill_workspace_size(shape), dtype=torch.uint8, device=dev)
    sv = torch.empty(api.saved_bytes(shape), dtype=torch.uint8, device=dev)
    y, _, _ = api.prefill(inp["q"], inp["k"], inp["v"], inp["gate"], gt, s0, workspace=wsf,
                          saved=sv, **kw)
    from_y = api.prefill_backward(None, None, inp["v"], inp["gate"], gt, inp["dy"], s0, dso,
                                  want_dstate_in=True, fwd_workspace=wsf, saved=sv, y=y, **kw)
    recomp = api.prefill_backward(None, None, inp["v"], inp["gate"], gt, inp["dy"], s0, dso,
                                  want_dstate_in=True, fwd_workspace=wsf, saved=sv, **kw)
    torch.cuda.synchronize()
    ref = oracle.backward(f64(inp["q"]), f64(inp["k"]), f64(inp["v"]), f64(inp["gate"]),
                          g.astype(np.float64), f64(inp["dy"]),
                          None if s0 is None else f64(s0), None if dso is None else f64(dso),
                          pos_offset=pos, base=1e6)
    tol = tol_for(torch.bfloat16)
    for name, got, want in zip(["dq", "dk", "dv", "dgate"], from_y[:4], ref[:4]):
        assert torch.isfinite(got.float()).all(), name
        err = max_rel_err(f64(got), want)
        assert err <= tol, f"{name}: {err:.3e}"
    err = max_rel_err(f64(from_y[4]), ref[4], head_axes=(0, 1))
    assert err <= tol, f"dstate_in: {err:.3e}"
    for name, a, b in zip(["dq", "dk", "dv", "dgate"], from_y[:4], recomp[:4]):
        assert max_rel_err(f64(a), f64(b)) <= 1e-2, name


def test_backward_from_y_rejects_y_without_saved(dev):
    B, T, H, d = 1, 64, 2, 128
    inp = inputs.mixer_inputs(B, T, H, d, torch.bfloat16, 7, device=dev, with_dy=True)
    gt = torch.from_numpy(oracle.gamma(H).astype(np.float32))
    with pytest.raises(ValueError):
        api.prefill_backward(inp["q"], inp["k"], inp["v"], inp["gate"], gt, inp["dy"], chunk=128,
                             y=inp["q"])
