"""The bounded waits' expiry path, forced from the host: a prefill whose
output-pass CTAs are given a budget of a few clock cycles for their first
wait (hla_trace.test_wait_cycles) gives up there, drains what it issued and
leaves; the call's status word reports HLA_ERR_TIMEOUT.  The device stays
usable: a normal prefill right after it, on the same stream and workspace,
matches the oracle and reports HLA_OK.  (No GPU fault is involved: the wait
simply runs out, the copies it had issued complete on their own.)"""
import numpy as np
import pytest
import torch

import oracle
from rnn_sequence_mixer_gb300 import _lib, api, inputs
from parity_util import f64, max_rel_err

pytestmark = pytest.mark.gpu


def test_expired_wait_reports_timeout_and_the_device_stays_usable():
    assert torch.cuda.is_available(), "GPU test needs a CUDA device"
    dev = torch.device("cuda:0")
    B, T, H, d, chunk = 1, 512, 152, 128, 128  # one CTA of four tiles per head, one wave
    g = oracle.gamma(H).astype(np.float32)
    gt = torch.from_numpy(g)
    inp = inputs.mixer_inputs(B, T, H, d, torch.bfloat16, 61, device=dev)
    shape = api.make_shape(B, T, H, d, chunk=chunk, rope_base=1e6)
    ws = torch.empty(api.prefill_workspace_size(shape), dtype=torch.uint8, device=dev)
    api.prefill(inp["q"], inp["k"], inp["v"], inp["gate"], gt, chunk=chunk, rope_base=1e6,
                workspace=ws, test_wait_cycles=1)
    torch.cuda.synchronize()
    assert api.workspace_status(ws) == _lib.HLA_ERR_TIMEOUT
    word = int(ws[-256:-252].cpu().view(torch.int32).item())
    assert word & 2, f"the output pass's bit, got {word:#x}"
    # the same stream and workspace, the normal budget: valid again
    y, o, st = api.prefill(inp["q"], inp["k"], inp["v"], inp["gate"], gt, chunk=chunk,
                           rope_base=1e6, want_o=True, workspace=ws)
    torch.cuda.synchronize()
    assert api.workspace_status(ws) == _lib.HLA_OK
    ry, ro, rs = oracle.prefill(f64(inp["q"]), f64(inp["k"]), f64(inp["v"]), f64(inp["gate"]),
                                g.astype(np.float64), base=1e6)
    assert max_rel_err(f64(y), ry) <= 2e-2
    assert max_rel_err(f64(o), ro) <= 2e-2
    assert max_rel_err(f64(st), rs, head_axes=(0, 1)) <= 2e-2


def test_expired_wait_in_the_one_launch_prefill():
    """The same in the prefill as one kernel launch (hla_shape.passes = 1),
    whose CTAs first form the state entering their segment from the decay
    window before it: with two segments per head the second segment's CTAs
    run that window phase to its end, then their first tile-loop wait runs
    out; the status word reports the timeout, and a normal one-launch call on
    the same stream and workspace matches the oracle."""
    assert torch.cuda.is_available(), "GPU test needs a CUDA device"
    dev = torch.device("cuda:0")
    B, T, H, d, chunk = 1, 1024, 76, 128, 128  # two segments of four tiles per head, one wave
    g = oracle.gamma(H).astype(np.float32)
    gt = torch.from_numpy(g)
    # more than one segment per head: the three-pass plan runs its local-state pass
    assert api.prefill_launches(api.make_shape(B, T, H, d, chunk=chunk, passes=3), gt) >= 3
    assert api.prefill_launches(api.make_shape(B, T, H, d, chunk=chunk, passes=1), gt) == 1
    inp = inputs.mixer_inputs(B, T, H, d, torch.bfloat16, 67, device=dev)
    shape = api.make_shape(B, T, H, d, chunk=chunk, rope_base=1e6, passes=1)
    ws = torch.empty(api.prefill_workspace_size(shape), dtype=torch.uint8, device=dev)
    api.prefill(inp["q"], inp["k"], inp["v"], inp["gate"], gt, chunk=chunk, rope_base=1e6,
                workspace=ws, passes=1, test_wait_cycles=1)
    torch.cuda.synchronize()
    assert api.workspace_status(ws) == _lib.HLA_ERR_TIMEOUT
    word = int(ws[-256:-252].cpu().view(torch.int32).item())
    assert word & 2, f"the output pass's bit, got {word:#x}"
    y, o, st = api.prefill(inp["q"], inp["k"], inp["v"], inp["gate"], gt, chunk=chunk,
                           rope_base=1e6, want_o=True, workspace=ws, passes=1)
    torch.cuda.synchronize()
    assert api.workspace_status(ws) == _lib.HLA_OK
    ry, ro, rs = oracle.prefill(f64(inp["q"]), f64(inp["k"]), f64(inp["v"]), f64(inp["gate"]),
                                g.astype(np.float64), base=1e6)
    assert max_rel_err(f64(y), ry) <= 2e-2
    assert max_rel_err(f64(o), ro) <= 2e-2
    assert max_rel_err(f64(st), rs, head_axes=(0, 1)) <= 2e-2
