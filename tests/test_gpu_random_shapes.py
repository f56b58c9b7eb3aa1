"""A seeded sweep of random small shapes through the prefill, its backward
(recomputing and with saved features) and the attention layer, against the
fp64 oracle: batch, length (ragged against the tile), heads, chunk, position
offset, initial state and grouped heads drawn from a fixed generator."""
import numpy as np
import pytest
import torch

import oracle
from rnn_sequence_mixer_gb300 import api, inputs
from parity_util import f64, max_rel_err

pytestmark = pytest.mark.gpu

TOL = 2e-2  # bf16


def shapes(n, seed):
    rng = np.random.default_rng(seed)
    out = []
    for _ in range(n):
        out.append(dict(B=int(rng.integers(1, 4)), T=int(rng.integers(1, 700)),
                        H=int(rng.choice([1, 2, 3, 5])), chunk=int(rng.choice([64, 128])),
                        pos=int(rng.choice([0, 1, 4093, 10 ** 6])), state=bool(rng.integers(0, 2))))
    return out


@pytest.fixture(scope="module")
def dev():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return torch.device("cuda:0")


@pytest.mark.parametrize("case", shapes(10, 2024), ids=lambda c: "B{B}T{T}H{H}c{chunk}p{pos}s{state:d}".format(**c))
def test_random_mixer_shapes(dev, case):
    B, T, H, chunk, pos = case["B"], case["T"], case["H"], case["chunk"], case["pos"]
    d = 128
    g = oracle.gamma(H).astype(np.float32)
    gt = torch.from_numpy(g)
    inp = inputs.mixer_inputs(B, T, H, d, torch.bfloat16, 300 + T, device=dev, with_dy=True)
    s0 = inputs.state(B, H, d, 301, 0.1, device=dev) if case["state"] else None
    dso = inputs.state(B, H, d, 302, 0.05, device=dev) if case["state"] else None
    kw = dict(chunk=chunk, pos_offset=pos, rope_base=1e6)
    shape = api.make_shape(B, T, H, d, dtype=torch.bfloat16, **kw)
    sv = torch.empty(api.saved_bytes(shape), dtype=torch.uint8, device=dev)
    y, o, st = api.prefill(inp["q"], inp["k"], inp["v"], inp["gate"], gt, s0, want_o=True, saved=sv,
                           **kw)
    grads = api.prefill_backward(inp["q"], inp["k"], inp["v"], inp["gate"], gt, inp["dy"], s0, dso,
                                 want_dstate_in=True, saved=sv, **kw)
    fresh = api.prefill_backward(inp["q"], inp["k"], inp["v"], inp["gate"], gt, inp["dy"], s0, dso,
                                 want_dstate_in=True, **kw)
    torch.cuda.synchronize()
    h = {k: f64(t) for k, t in inp.items()}
    s0h = None if s0 is None else f64(s0)
    ry, ro, rs = oracle.prefill(h["q"], h["k"], h["v"], h["gate"], g.astype(np.float64), s0h,
                                pos_offset=pos, base=1e6)
    assert max_rel_err(f64(y), ry) <= TOL
    assert max_rel_err(f64(o), ro) <= TOL
    assert max_rel_err(f64(st), rs, head_axes=(0, 1)) <= TOL
    ref = oracle.backward(h["q"], h["k"], h["v"], h["gate"], g.astype(np.float64), h["dy"], s0h,
                          None if dso is None else f64(dso), pos_offset=pos, base=1e6)
    for label, out in (("saved", grads), ("recomputed", fresh)):
        for name, got, want in zip(["dq", "dk", "dv", "dgate"], out[:4], ref[:4]):
            err = max_rel_err(f64(got), want)
            assert err <= TOL, f"{label} {name}: {err:.3e}"
        assert max_rel_err(f64(out[4]), ref[4], head_axes=(0, 1)) <= TOL, label


@pytest.mark.parametrize("case", shapes(6, 77), ids=lambda c: "B{B}T{T}p{pos}".format(**c))
def test_random_attention_shapes(dev, case):
    B, T, pos = case["B"], case["T"], case["pos"]
    rng = np.random.default_rng(T)
    Hkv = int(rng.choice([1, 2]))
    Hq = Hkv * int(rng.choice([1, 2, 4]))
    a = float(rng.choice([500.0, 600.0, 900.0]))
    x = inputs.mixer_inputs(B, T, Hq, 128, torch.bfloat16, 400 + T, device=dev)
    kv = inputs.mixer_inputs(B, T, Hkv, 128, torch.bfloat16, 401 + T, device=dev)
    y, o = api.attention_prefill(x["q"], kv["k"], kv["v"], x["gate"], a, pos_offset=pos, want_o=True)
    torch.cuda.synchronize()
    ry, ro = oracle.attention(f64(x["q"]), f64(kv["k"]), f64(kv["v"]), f64(x["gate"]), a,
                              pos_offset=pos)
    assert max_rel_err(f64(o), ro) <= TOL
    assert max_rel_err(f64(y), ry) <= TOL
