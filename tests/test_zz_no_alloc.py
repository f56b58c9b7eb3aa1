"""hla_prefill_noalloc, the prefill for callers that cannot allocate device
memory (an engine plugin whose host owns every byte of GPU memory, or a serving
loop that must not allocate once it runs): it takes no workspace and keeps its
per-segment states in a fixed scratch array inside the library.

Its results must match hla_prefill's, call after call: the scratch array keeps
the previous call's contents, so two calls in a row with different inputs
check that nothing stale leaks from one call into the next.  Kept in a file of
its own that pytest collects last.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from rnn_sequence_mixer_gb300 import _lib, api, inputs
from parity_util import f64, max_rel_err, tol_for

pytestmark = pytest.mark.gpu


def noalloc(inp, gamma, state_in, *, chunk, base, eps=1e-6):
    """Call hla_prefill_noalloc through the C ABI; returns (status, y, o, state_out)."""
    q = inp["q"]
    B, T, H, d = q.shape
    shape = api.make_shape(B, T, H, d, chunk=chunk, dtype=q.dtype, rope_base=base, eps=eps)
    y = torch.empty_like(q)
    o = torch.empty(q.shape, dtype=torch.float32, device=q.device)
    st = torch.empty((B, H, d, d), dtype=torch.float32, device=q.device)
    g = torch.as_tensor(gamma, dtype=torch.float32).contiguous()
    gp = ctypes.cast(ctypes.c_void_p(g.data_ptr()), ctypes.POINTER(ctypes.c_float))
    ptr = lambda t: None if t is None else ctypes.c_void_p(t.data_ptr())
    stream = ctypes.c_void_p(torch.cuda.current_stream(q.device).cuda_stream)
    status = _lib.load().hla_prefill_noalloc(ctypes.byref(shape), ptr(q), ptr(inp["k"]),
                                             ptr(inp["v"]), ptr(inp["gate"]), gp, ptr(state_in),
                                             ptr(st), ptr(y), ptr(o), stream)
    return status, y, o, st


@pytest.mark.parametrize("B,T,H,d,dtype,chunk,with_state", [
    (1, 4000, 16, 128, torch.bfloat16, 64, False),
    (3, 300, 100, 128, torch.bfloat16, 64, True),   # 300 heads of d = 128: one segment each
    (1, 3000, 120, 128, torch.bfloat16, 64, True),  # the plan's 5 segments exceed the scratch: capped to 4
    (2, 517, 4, 64, torch.float32, 128, True),
])
def test_noalloc_matches_prefill_two_calls_in_a_row(B, T, H, d, dtype, chunk, with_state):
    assert torch.cuda.is_available(), "GPU test needs a CUDA device"
    dev = torch.device("cuda:0")
    gamma = oracle.gamma(H).astype(np.float32)
    for call in range(2):
        seed = 1000 * call + T + H
        inp = inputs.mixer_inputs(B, T, H, d, dtype, seed, device=dev)
        s0 = inputs.state(B, H, d, seed + 1, 0.1, device=dev) if with_state else None
        status, y, o, st = noalloc(inp, gamma, s0, chunk=chunk, base=1e6)
        assert status == _lib.HLA_OK, _lib.status_string(status)
        ry, ro, rs = api.prefill(inp["q"], inp["k"], inp["v"], inp["gate"], torch.from_numpy(gamma),
                                 s0, chunk=chunk, rope_base=1e6, want_o=True)
        torch.cuda.synchronize()
        tol = tol_for(dtype)
        assert max_rel_err(f64(y), f64(ry)) <= tol, f"call {call}: y"
        assert max_rel_err(f64(o), f64(ro)) <= tol, f"call {call}: o"
        assert max_rel_err(f64(st), f64(rs), head_axes=(0, 1)) <= tol, f"call {call}: state"


def test_noalloc_rejects_problems_beyond_the_scratch_limit():
    """B * H fp32 d x d states must fit in the fixed scratch; 1024 heads of
    d = 128 need 64 MiB and are refused before anything runs."""
    assert torch.cuda.is_available(), "GPU test needs a CUDA device"
    dev = torch.device("cuda:0")
    B, T, H, d = 16, 8, 64, 128
    inp = inputs.mixer_inputs(B, T, H, d, torch.bfloat16, 3, device=dev)
    status, *_ = noalloc(inp, np.full(H, 0.9, dtype=np.float32), None, chunk=64, base=1e6)
    assert status == _lib.HLA_ERR_WORKSPACE
