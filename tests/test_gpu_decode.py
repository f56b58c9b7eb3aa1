"""GPU parity of hla_decode_step against the fp64 oracle."""
import numpy as np
import pytest
import torch

import oracle
from rnn_sequence_mixer_gb300 import api, inputs, workloads
from parity_util import elem_rel_err, f64, gather_state, max_rel_err, tol_for

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return torch.device("cuda:0")


@pytest.mark.parametrize("B,H,d,dtype,use_pos,inplace", [
    (3, 4, 64, torch.float32, True, True),
    (2, 2, 128, torch.float32, False, False),
    (5, 3, 128, torch.bfloat16, True, False),
    (1, 32, 64, torch.bfloat16, False, True),
    (16, 32, 128, torch.bfloat16, True, True),
    (9, 40, 64, torch.float32, True, False),
    (1, 16, 128, torch.bfloat16, False, False),
])
@pytest.mark.parametrize("split", [0, 1, 2, 4, 8])
def test_decode_small(dev, B, H, d, dtype, use_pos, inplace, split):
    g = oracle.gamma(H).astype(np.float32)
    inp = inputs.mixer_inputs(B, 1, H, d, dtype, 40 + B, device=dev)
    s0 = inputs.state(B, H, d, 41, scale=0.2, device=dev)
    pos_host = np.array([17 * b + 3 for b in range(B)], dtype=np.int64)
    pos = torch.from_numpy(pos_host).to(dev) if use_pos else None
    st_in = s0.clone()
    st_out = st_in if inplace else torch.empty_like(s0)
    y, o, st = api.decode_step(inp["q"], inp["k"], inp["v"], inp["gate"], torch.from_numpy(g),
                               st_in, pos, pos_offset=9, rope_base=1e6, state_out=st_out,
                               want_o=True, split=split)
    torch.cuda.synchronize()
    rpos = pos_host if use_pos else np.full(B, 9)
    ry, ro, rs = oracle.decode_step(f64(inp["q"]), f64(inp["k"]), f64(inp["v"]), f64(inp["gate"]),
                                    g.astype(np.float64), rpos, f64(s0), base=1e6)
    tol = tol_for(dtype)
    assert max_rel_err(f64(o), ro) <= tol
    assert max_rel_err(f64(y), ry) <= tol
    assert max_rel_err(f64(st), rs, head_axes=(0, 1)) <= tol
    # a single step from a given state also holds element by element (floor
    # 1e-3 of each slice's maximum)
    assert elem_rel_err(f64(o), ro) <= tol
    assert elem_rel_err(f64(y), ry) <= tol
    assert elem_rel_err(f64(st), rs, head_axes=(0, 1)) <= tol
    if not inplace:
        assert torch.equal(st_in, s0), "state_in must be left untouched"


def test_decode_workload_sampled(dev):
    """4096-token prefill builds the state; 256 single-token steps follow.
    Sampled (b, h) heads are checked at every step and at the end."""
    w = workloads.DECODE_B64
    g = oracle.gamma(w.H).astype(np.float32)
    gt = torch.from_numpy(g)
    pre = inputs.mixer_inputs(w.B, w.prefill_T, w.H, w.d, w.dtype, w.seed, device=dev)
    _, _, state = api.prefill(pre["q"], pre["k"], pre["v"], pre["gate"], gt, chunk=w.chunk,
                              rope_base=w.rope_base, eps=w.eps)
    steps = inputs.decode_inputs(w.steps, w.B, w.H, w.d, w.dtype, w.seed + 100, device=dev)
    pos = torch.full((w.B,), w.prefill_T, dtype=torch.int64, device=dev)
    ys = []
    for s in range(w.steps):
        y, _, _ = api.decode_step(steps["q"][s], steps["k"][s], steps["v"][s], steps["gate"][s], gt,
                                  state, pos, rope_base=w.rope_base, eps=w.eps)
        ys.append(y)
        pos += 1
    torch.cuda.synchronize()
    pairs = [(0, 0), (7, 3), (21, 16), (40, 29), (63, 31)]
    gg = np.array([float(g[h]) for (_, h) in pairs])
    sel = lambda t: f64(torch.stack([t[b, :, h, :] for (b, h) in pairs], dim=1).unsqueeze(0))
    _, _, rs = oracle.prefill(sel(pre["q"]), sel(pre["k"]), sel(pre["v"]), sel(pre["gate"]), gg,
                              base=w.rope_base, eps=w.eps)
    worst = 0.0
    for s in range(w.steps):
        row = lambda t: sel(t[s])
        ry, _, rs = oracle.decode_step(row(steps["q"]), row(steps["k"]), row(steps["v"]),
                                       row(steps["gate"]), gg, np.array([w.prefill_T + s]), rs,
                                       base=w.rope_base, eps=w.eps)
        worst = max(worst, max_rel_err(sel(ys[s]), ry))
    assert worst <= 2e-2, worst
    err = max_rel_err(gather_state(state, pairs), rs, head_axes=(0, 1))
    assert err <= 2e-2, err


def test_decode_of_an_empty_batch_is_a_no_op():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    dev = torch.device("cuda:0")
    H, d = 4, 128
    rows = inputs.decode_inputs(1, 0, H, d, torch.bfloat16, 3, device=dev)
    state = torch.empty((0, H, d, d), dtype=torch.float32, device=dev)
    y, _, st = api.decode_step(rows["q"][0], rows["k"][0], rows["v"][0], rows["gate"][0],
                               api.gamma_schedule(H), state)
    torch.cuda.synchronize()
    assert y.numel() == 0 and st.numel() == 0


@pytest.mark.parametrize("B,H,d,dtype", [(1, 16, 128, torch.bfloat16), (2, 8, 64, torch.float32)])
def test_decode_split_state_is_bit_identical(dev, B, H, d, dtype):
    """Every split applies the same per-element update S <- gamma S + k~^T v with
    the same k~ and v, so the new state is bit-identical whichever CTA owns
    which columns; o and y differ only in the order of the q~ S sum."""
    g = torch.from_numpy(oracle.gamma(H).astype(np.float32))
    inp = inputs.mixer_inputs(B, 1, H, d, dtype, 55, device=dev)
    s0 = inputs.state(B, H, d, 56, scale=0.3, device=dev)
    outs = {}
    for split in (1, 2, 4, 8):
        st = s0.clone()
        y, o, st = api.decode_step(inp["q"], inp["k"], inp["v"], inp["gate"], g, st, None,
                                   pos_offset=4096, rope_base=1e6, want_o=True, split=split)
        outs[split] = (y.float(), o, st)
    torch.cuda.synchronize()
    for split in (2, 4, 8):
        assert torch.equal(outs[split][2], outs[1][2]), split
        assert torch.allclose(outs[split][1], outs[1][1], rtol=1e-5, atol=1e-5), split
        assert torch.allclose(outs[split][0], outs[1][0], rtol=1e-2, atol=1e-2), split
