"""hla_prefill_noalloc, the prefill for callers that cannot allocate device
memory (an engine plugin whose host owns every byte of GPU memory, or a serving
loop that must not allocate once it runs): it takes no workspace and keeps its
per-segment states in a fixed scratch array inside the library.

Its results are checked against the fp64 oracle, call after call: the scratch
array keeps the previous call's contents, so two calls in a row with different
inputs check that nothing stale leaks from one call into the next.  hla_prefill
on the same inputs is a second check.  Kept in a file of its own that pytest
collects last.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from rnn_sequence_mixer_gb300 import _lib, api, inputs
from parity_util import f64, max_rel_err, tol_for

pytestmark = pytest.mark.gpu


def noalloc(q, k, v, gate, gamma, state_in, *, chunk, base, eps=1e-6, B=None, T=None,
            H=None, d=None, dtype=None, state_out=True):
    """Call hla_prefill_noalloc through the C ABI; returns (status, y, o, state_out)."""
    if q is not None:
        B, T, H, d = q.shape
        dtype = q.dtype
    shape = api.make_shape(B, T, H, d, chunk=chunk, dtype=dtype, rope_base=base, eps=eps)
    dev = torch.device("cuda:0")
    y = None if q is None else torch.empty_like(q)
    o = None if q is None else torch.empty(q.shape, dtype=torch.float32, device=dev)
    st = torch.empty((B, H, d, d), dtype=torch.float32, device=dev) if state_out else None
    g = torch.as_tensor(gamma, dtype=torch.float32).contiguous()
    gp = ctypes.cast(ctypes.c_void_p(g.data_ptr()), ctypes.POINTER(ctypes.c_float))
    ptr = lambda t: None if t is None else ctypes.c_void_p(t.data_ptr())
    stream = ctypes.c_void_p(torch.cuda.current_stream(dev).cuda_stream)
    status = _lib.load().hla_prefill_noalloc(ctypes.byref(shape), ptr(q), ptr(k), ptr(v),
                                             ptr(gate), gp, ptr(state_in), ptr(st), ptr(y),
                                             ptr(o), stream)
    return status, y, o, st


def test_empty_call_sets_up_the_device_and_passes_the_state_through():
    """The start-up call (B == 0 or T == 0) resolves the scratch array and loads
    the kernels, launches no kernel, and leaves state_out = state_in."""
    assert torch.cuda.is_available(), "GPU test needs a CUDA device"
    dev = torch.device("cuda:0")
    H, d = 4, 128
    gamma = oracle.gamma(H).astype(np.float32)
    s0 = inputs.state(2, H, d, 5, 0.1, device=dev)
    status, _, _, st = noalloc(None, None, None, None, gamma, s0, chunk=64, base=1e6, B=2, T=0,
                               H=H, d=d, dtype=torch.bfloat16)
    assert status == _lib.HLA_OK, _lib.status_string(status)
    torch.cuda.synchronize()
    assert torch.equal(st, s0)
    status, *_ = noalloc(None, None, None, None, gamma, None, chunk=64, base=1e6, B=0, T=16,
                         H=H, d=d, dtype=torch.bfloat16, state_out=False)
    assert status == _lib.HLA_OK, _lib.status_string(status)


@pytest.mark.parametrize("B,T,H,d,dtype,chunk,with_state", [
    (1, 4000, 16, 128, torch.bfloat16, 64, False),
    (3, 300, 100, 128, torch.bfloat16, 64, True),   # 300 heads of d = 128: one segment each
    (1, 3000, 120, 128, torch.bfloat16, 64, True),  # the plan's 5 segments exceed the scratch: capped to 4
    (4, 1000, 128, 128, torch.bfloat16, 128, True), # B * H = 512, the limit: one segment of 1000 tokens
    (2, 517, 4, 64, torch.float32, 128, True),
])
def test_noalloc_matches_oracle_two_calls_in_a_row(B, T, H, d, dtype, chunk, with_state):
    assert torch.cuda.is_available(), "GPU test needs a CUDA device"
    dev = torch.device("cuda:0")
    gamma = oracle.gamma(H).astype(np.float32)
    tol = tol_for(dtype)
    for call in range(2):
        seed = 1000 * call + T + H
        inp = inputs.mixer_inputs(B, T, H, d, dtype, seed, device=dev)
        s0 = inputs.state(B, H, d, seed + 1, 0.1, device=dev) if with_state else None
        status, y, o, st = noalloc(inp["q"], inp["k"], inp["v"], inp["gate"], gamma, s0,
                                   chunk=chunk, base=1e6)
        assert status == _lib.HLA_OK, _lib.status_string(status)
        torch.cuda.synchronize()
        ry, ro, rs = oracle.prefill(f64(inp["q"]), f64(inp["k"]), f64(inp["v"]), f64(inp["gate"]),
                                    gamma.astype(np.float64), None if s0 is None else f64(s0),
                                    base=1e6, eps=1e-6)
        assert max_rel_err(f64(y), ry) <= tol, f"call {call}: y against the oracle"
        assert max_rel_err(f64(o), ro) <= tol, f"call {call}: o against the oracle"
        assert max_rel_err(f64(st), rs, head_axes=(0, 1)) <= tol, f"call {call}: state against the oracle"
        # second check: the workspace entry point on the same inputs
        py, po, ps = api.prefill(inp["q"], inp["k"], inp["v"], inp["gate"], torch.from_numpy(gamma),
                                 s0, chunk=chunk, rope_base=1e6, want_o=True)
        torch.cuda.synchronize()
        assert max_rel_err(f64(y), f64(py)) <= tol, f"call {call}: y against hla_prefill"
        assert max_rel_err(f64(st), f64(ps), head_axes=(0, 1)) <= tol, f"call {call}: state against hla_prefill"


def test_noalloc_rejects_problems_beyond_the_scratch_limit():
    """B * H fp32 d x d states must fit in the fixed scratch; 1024 heads of
    d = 128 need 64 MiB and are refused before anything runs."""
    assert torch.cuda.is_available(), "GPU test needs a CUDA device"
    dev = torch.device("cuda:0")
    B, T, H, d = 16, 8, 64, 128
    inp = inputs.mixer_inputs(B, T, H, d, torch.bfloat16, 3, device=dev)
    status, *_ = noalloc(inp["q"], inp["k"], inp["v"], inp["gate"], np.full(H, 0.9, dtype=np.float32),
                         None, chunk=64, base=1e6)
    assert status == _lib.HLA_ERR_WORKSPACE
