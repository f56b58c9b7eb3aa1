"""GPU parity of hla_prefill against the fp64 oracle (element by element).

Small shapes are compared in full; the 16K workload is compared in full; the
512K workload is compared on sampled heads over time windows whose warm-up
length W makes gamma^W <= 1e-12 (the state of a decaying recurrence forgets
its start: a zero-state oracle run over [t - W, t + M) reproduces outputs in
[t, t + M) to that accuracy)."""
import numpy as np
import pytest
import torch

import oracle
from rnn_sequence_mixer_gb300 import api, inputs, workloads
from parity_util import (f64, gather_heads, gather_state, max_rel_err, oracle_window, tol_for,
                         window_for)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return torch.device("cuda:0")


def gamma32(H):
    """fp32 forget rates from the oracle's Eq. 19 (never from the library)."""
    return oracle.gamma(H).astype(np.float32)


def run_case(dev, B, T, H, d, dtype, chunk, base=1e4, pos_offset=0, with_state=False, seed=0,
             gam=None):
    inp = inputs.mixer_inputs(B, T, H, d, dtype, seed, device=dev)
    g = gamma32(H) if gam is None else np.asarray(gam, dtype=np.float32)
    s0 = inputs.state(B, H, d, seed + 1000, scale=0.1, device=dev) if with_state else None
    y, o, st = api.prefill(inp["q"], inp["k"], inp["v"], inp["gate"], torch.from_numpy(g), s0,
                           chunk=chunk, pos_offset=pos_offset, rope_base=base, eps=1e-6,
                           want_o=True)
    torch.cuda.synchronize()
    ry, ro, rs = oracle.prefill(f64(inp["q"]), f64(inp["k"]), f64(inp["v"]), f64(inp["gate"]),
                                g.astype(np.float64), None if s0 is None else f64(s0),
                                pos_offset=pos_offset, base=base, eps=1e-6)
    return (f64(y), f64(o), f64(st)), (ry, ro, rs)


def assert_close(got, ref, tol, what):
    err = max_rel_err(got, ref)
    assert err <= tol, f"{what}: max rel err {err:.3e} > {tol:.1e}"


def assert_state_close(got, ref, tol, what):
    err = max_rel_err(got, ref, head_axes=(0, 1))
    assert err <= tol, f"{what}: max rel err {err:.3e} > {tol:.1e}"


def test_tiny_fp32_workload(dev):
    w = workloads.TINY_FP32
    (y, o, st), (ry, ro, rs) = run_case(dev, w.B, w.T, w.H, w.d, w.dtype, w.chunk, w.rope_base,
                                        seed=w.seed)
    assert_close(o, ro, 1e-4, "o")
    assert_close(y, ry, 1e-4, "y")
    assert_state_close(st, rs, 1e-4, "state")


@pytest.mark.parametrize("B,T,H,d,dtype,chunk,with_state,pos", [
    (1, 1, 2, 64, torch.float32, 64, False, 0),
    (2, 77, 3, 64, torch.float32, 64, True, 5),
    (1, 300, 2, 128, torch.float32, 128, True, 1000),
    (2, 129, 4, 128, torch.bfloat16, 64, False, 0),
    (1, 1000, 2, 128, torch.bfloat16, 128, True, 123456),
    (3, 64, 5, 64, torch.bfloat16, 64, True, 7),
    (1, 2500, 16, 128, torch.bfloat16, 64, False, 0),
])
def test_small_shapes(dev, B, T, H, d, dtype, chunk, with_state, pos):
    (y, o, st), (ry, ro, rs) = run_case(dev, B, T, H, d, dtype, chunk, 1e6, pos, with_state,
                                        seed=T + H)
    tol = tol_for(dtype)
    assert_close(o, ro, tol, "o")
    assert_close(y, ry, tol, "y")
    assert_state_close(st, rs, tol, "state")


def test_gamma_one_and_fast_heads(dev):
    """gamma = 1 (plain linear attention) next to the fastest-decaying heads of H = 32."""
    g = gamma32(32)[:4].copy()
    g[1] = 1.0
    (y, o, st), (ry, ro, rs) = run_case(dev, 1, 333, 4, 64, torch.float32, 64, 1e4, 0, True,
                                        seed=9, gam=g)
    assert_close(o, ro, 1e-4, "o")
    assert_close(y, ry, 1e-4, "y")
    assert_state_close(st, rs, 1e-4, "state")


def test_chunk_64_and_128_agree(dev):
    inp = inputs.mixer_inputs(1, 700, 4, 128, torch.float32, 31, device=dev)
    g = torch.from_numpy(gamma32(4))
    a = api.prefill(inp["q"], inp["k"], inp["v"], inp["gate"], g, chunk=64, want_o=True)
    b = api.prefill(inp["q"], inp["k"], inp["v"], inp["gate"], g, chunk=128, want_o=True)
    assert max_rel_err(f64(a[1]), f64(b[1])) < 1e-5
    assert max_rel_err(f64(a[2]), f64(b[2]), head_axes=(0, 1)) < 1e-5


def test_state_out_in_place(dev):
    inp = inputs.mixer_inputs(2, 200, 2, 64, torch.float32, 32, device=dev)
    g = torch.from_numpy(gamma32(2))
    s0 = inputs.state(2, 2, 64, 33, 0.1, device=dev)
    ref = api.prefill(inp["q"], inp["k"], inp["v"], inp["gate"], g, s0.clone())[2]
    buf = s0.clone()
    api.prefill(inp["q"], inp["k"], inp["v"], inp["gate"], g, buf, state_out=buf)
    torch.cuda.synchronize()
    assert torch.equal(buf, ref)


def test_prefill_16k_workload_full(dev):
    w = workloads.PREFILL_16K
    (y, o, st), (ry, ro, rs) = run_case(dev, w.B, w.T, w.H, w.d, w.dtype, w.chunk, w.rope_base,
                                        seed=w.seed)
    assert_close(y, ry, 2e-2, "y")
    assert_close(o, ro, 2e-2, "o")
    assert_state_close(st, rs, 2e-2, "state")


def test_prefill_512k_workload_sampled(dev):
    w = workloads.PREFILL_512K
    inp = inputs.mixer_inputs(w.B, w.T, w.H, w.d, w.dtype, w.seed, device=dev)
    g = gamma32(w.H)
    y, _, st = api.prefill(inp["q"], inp["k"], inp["v"], inp["gate"], torch.from_numpy(g),
                           chunk=w.chunk, rope_base=w.rope_base, eps=w.eps)
    torch.cuda.synchronize()
    pairs = [(0, 0), (0, 5), (0, 11), (0, 15)]
    W = window_for(g, pairs)
    M = 384
    for t in (0, 131_072 + 77, 400_000, w.T - M):
        lo = max(0, t - W)
        ry, _, _ = oracle_window(inp, g, pairs, lo, t + M, w.rope_base, w.eps)
        got = gather_heads(y, pairs, t, t + M)
        assert_close(got, ry[:, t - lo:], 2e-2, f"y window at {t}")
    _, _, rs = oracle_window(inp, g, pairs, w.T - W, w.T, w.rope_base, w.eps)
    assert_state_close(gather_state(st, pairs), rs, 2e-2, "final state")
    del inp, y, st
    torch.cuda.empty_cache()


@pytest.mark.parametrize("dtype,d", [(torch.bfloat16, 128), (torch.float32, 64)])
def test_status_word_is_clear(dev, dtype, d):
    """The last 256 bytes of the workspace hold the device status word; it is
    cleared by every call and stays 0 when no bounded wait gave up."""
    B, T, H = 1, 3000, 8
    inp = inputs.mixer_inputs(B, T, H, d, dtype, 77, device=dev)
    shape = api.make_shape(B, T, H, d, chunk=128, dtype=dtype)
    n = api.prefill_workspace_size(shape)
    ws = torch.full((n,), 0xAB, dtype=torch.uint8, device=dev)
    api.prefill(inp["q"], inp["k"], inp["v"], inp["gate"], torch.from_numpy(gamma32(H)),
                chunk=128, workspace=ws)
    torch.cuda.synchronize()
    status = ws[n - 256:n - 252].view(torch.int32).item()
    assert status == 0


def test_streamed_prefill_matches_one_shot_oracle(dev):
    """A sequence fed through hla_prefill in pieces (each piece's final state
    is the next one's state_in, positions continued by pos_offset) equals the
    oracle's single pass; the last piece is ragged."""
    B, T, H, d = 1, 6000, 4, 128
    inp = inputs.mixer_inputs(B, T, H, d, torch.bfloat16, 41, device=dev)
    g = gamma32(H)
    y = torch.empty_like(inp["q"])
    st = torch.empty((B, H, d, d), dtype=torch.float32, device=dev)
    for j, (a, b) in enumerate([(0, 2048), (2048, 4096), (4096, T)]):
        sl = slice(a, b)
        api.prefill(inp["q"][:, sl], inp["k"][:, sl], inp["v"][:, sl], inp["gate"][:, sl],
                    torch.from_numpy(g), st if j else None, chunk=128, pos_offset=a,
                    rope_base=1e6, y=y[:, sl], state_out=st)
    torch.cuda.synchronize()
    ry, _, rs = oracle.prefill(f64(inp["q"]), f64(inp["k"]), f64(inp["v"]), f64(inp["gate"]),
                               g.astype(np.float64), None, base=1e6)
    assert_close(f64(y), ry, 2e-2, "y")
    assert_state_close(f64(st), rs, 2e-2, "state")


@pytest.mark.parametrize("B,T", [(1, 0), (0, 5), (3, 0)])
def test_empty_inputs_pass_the_state_through(dev, B, T):
    """An empty batch or sequence computes nothing: state_out = state_in, or
    zeros without state_in; the status word is cleared."""
    H, d = 3, 128
    inp = inputs.mixer_inputs(B, T, H, d, torch.bfloat16, 5, device=dev)
    g = torch.from_numpy(gamma32(H))
    s0 = inputs.state(B, H, d, 6, 0.1, device=dev)
    _, _, st = api.prefill(inp["q"], inp["k"], inp["v"], inp["gate"], g, s0, chunk=128)
    torch.cuda.synchronize()
    assert torch.equal(st, s0)
    shape = api.make_shape(B, T, H, d, chunk=128, dtype=torch.bfloat16)
    n = api.prefill_workspace_size(shape)
    ws = torch.full((n,), 0xAB, dtype=torch.uint8, device=dev)
    _, _, st0 = api.prefill(inp["q"], inp["k"], inp["v"], inp["gate"], g, chunk=128, workspace=ws)
    torch.cuda.synchronize()
    assert torch.count_nonzero(st0).item() == 0
    assert ws[n - 256:n - 252].view(torch.int32).item() == 0


@pytest.mark.parametrize("case", ["large_magnitudes", "single_token", "tiny_gamma"])
def test_tensor_core_path_edge_inputs(dev, case):
    """bf16 at d = 128 (the tensor-core kernels) away from N(0, 1) inputs: q, k,
    v scaled by 1e2 / 1e2 / 1e3 with gates of +-20 (the fp16 state scaling and
    the norms must absorb them), a single token, and gamma = 1e-6 (every decay
    power underflows after one step)."""
    B, T, H, d = 1, 777, 4, 128
    g = gamma32(H)
    if case == "single_token":
        T = 1
    if case == "tiny_gamma":
        g = np.full(H, 1e-6, dtype=np.float32)
    inp = inputs.mixer_inputs(B, T, H, d, torch.float32, 71, device=dev)
    if case == "large_magnitudes":
        inp["q"] *= 100.0
        inp["k"] *= 100.0
        inp["v"] *= 1000.0
        inp["gate"] *= 20.0
    inp = {k: v.to(torch.bfloat16) for k, v in inp.items()}
    s0 = inputs.state(B, H, d, 72, scale=1.0 if case == "large_magnitudes" else 0.1, device=dev)
    y, o, st = api.prefill(inp["q"], inp["k"], inp["v"], inp["gate"], torch.from_numpy(g), s0,
                           chunk=128, rope_base=1e6, want_o=True)
    torch.cuda.synchronize()
    ry, ro, rs = oracle.prefill(f64(inp["q"]), f64(inp["k"]), f64(inp["v"]), f64(inp["gate"]),
                                g.astype(np.float64), f64(s0), base=1e6)
    assert torch.isfinite(y.float()).all() and torch.isfinite(st).all()
    assert_close(f64(o), ro, 2e-2, "o")
    assert_close(f64(y), ry, 2e-2, "y")
    assert_state_close(f64(st), rs, 2e-2, "state")
