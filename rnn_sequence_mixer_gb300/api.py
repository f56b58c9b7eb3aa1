"""PyTorch-facing binding of the C ABI (``include/hla.h``).

Each function checks that its tensors are CUDA, contiguous and of one dtype,
allocates outputs and workspace through PyTorch's caching allocator, and calls
the library entry point of the same name on the current CUDA stream.  It does
no arithmetic of the mixer: there is no CPU path and no fallback, and a missing
``libhla.so`` raises.
"""
from __future__ import annotations

import ctypes
from typing import Optional, Sequence

import torch

from . import _lib

_DTYPES = {torch.float32: _lib.HLA_F32, torch.bfloat16: _lib.HLA_BF16}


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _host_gamma(gamma, H: int):
    g = torch.as_tensor(gamma, dtype=torch.float32, device="cpu").contiguous()
    if g.numel() != H:
        raise ValueError(f"gamma must have H={H} entries, got {g.numel()}")
    return g, ctypes.cast(ctypes.c_void_p(g.data_ptr()), ctypes.POINTER(ctypes.c_float))


def _check_acts(*ts: torch.Tensor):
    ref = ts[0]
    if not ref.is_cuda:
        raise ValueError("libhla runs on CUDA tensors only (no CPU path)")
    if ref.dim() != 4:
        raise ValueError("activations must be [B, T, H, d]")
    if ref.dtype not in _DTYPES:
        raise ValueError(f"unsupported dtype {ref.dtype}")
    for t in ts:
        if t.shape != ref.shape or t.dtype != ref.dtype or t.device != ref.device:
            raise ValueError("q, k, v, gate (and dy) must share shape, dtype and device")
        if not t.is_contiguous():
            raise ValueError("activations must be contiguous")


def _check_state(s: Optional[torch.Tensor], B, H, d, device):
    if s is None:
        return
    if s.dtype != torch.float32 or not s.is_contiguous() or s.device != device:
        raise ValueError("states are contiguous fp32 tensors on the activations' device")
    if tuple(s.shape) != (B, H, d, d):
        raise ValueError(f"state must be [B, H, d, d] = {(B, H, d, d)}")


def make_shape(B, T, H, d, *, chunk=64, dtype=torch.bfloat16, pos_offset=0, rope_base=1e4,
               eps=1e-6, decode_split=0, passes=0) -> _lib.HlaShape:
    return _lib.HlaShape(B=B, T=T, H=H, dk=d, dv=d, chunk=chunk, dtype=_DTYPES[dtype],
                         decode_split=int(decode_split),
                         pos_offset=int(pos_offset), rope_base=float(rope_base),
                         norm_eps=float(eps), passes=int(passes))


def gamma_schedule(H: int) -> torch.Tensor:
    """Eq. 19 forget rates for H heads as a host fp32 tensor (hla_gamma_schedule)."""
    out = torch.empty(H, dtype=torch.float32)
    st = _lib.load().hla_gamma_schedule(H, ctypes.cast(ctypes.c_void_p(out.data_ptr()),
                                                       ctypes.POINTER(ctypes.c_float)))
    _lib.check(st, "hla_gamma_schedule")
    return out


def prefill_workspace_size(shape: _lib.HlaShape) -> int:
    return int(_lib.load().hla_prefill_workspace_size(ctypes.byref(shape)))


def workspace_status(workspace: torch.Tensor) -> int:
    """The status of a finished call from its workspace's status word (the
    first uint32 of its last 256 bytes; the caller synchronizes first):
    HLA_OK, or HLA_ERR_TIMEOUT when a bounded device-side wait gave up."""
    word = int(workspace[-256:-252].cpu().view(torch.int32).item())
    return _lib.HLA_OK if word == 0 else _lib.HLA_ERR_TIMEOUT


def prefill_launches(shape: _lib.HlaShape, gamma) -> int:
    """hla_prefill_launches: kernels one prefill call with this shape launches."""
    g_host, g_ptr = _host_gamma(gamma, shape.H)
    return int(_lib.load().hla_prefill_launches(ctypes.byref(shape), g_ptr))


def backward_launches(shape: _lib.HlaShape, gamma, with_fwd_ws: bool) -> int:
    """hla_backward_launches: kernels one prefill_backward call launches."""
    g_host, g_ptr = _host_gamma(gamma, shape.H)
    return int(_lib.load().hla_backward_launches(ctypes.byref(shape), g_ptr, int(bool(with_fwd_ws))))


def saved_bytes(shape: _lib.HlaShape) -> int:
    """hla_saved_bytes: size of the ``saved`` buffer of prefill / prefill_backward
    (0 where the shape cannot save its features)."""
    return int(_lib.load().hla_saved_bytes(ctypes.byref(shape)))


def backward_workspace_size(shape: _lib.HlaShape) -> int:
    return int(_lib.load().hla_backward_workspace_size(ctypes.byref(shape)))


def _check_saved(saved, shape):
    if saved is None:
        return
    need = saved_bytes(shape)
    if saved.dtype != torch.uint8 or not saved.is_cuda or not saved.is_contiguous():
        raise ValueError("saved must be a contiguous uint8 CUDA tensor")
    if need and saved.numel() < need:
        raise ValueError(f"saved holds {saved.numel()} bytes, the shape needs {need}")


def _stream(device) -> ctypes.c_void_p:
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def _trace(events, device, test_wait_cycles=0):
    """hla_trace from a list of torch.cuda.Event (None = no tracing) and the
    testing-only wait budget (hla.h)."""
    if test_wait_cycles:
        tr = _lib.HlaTrace()
        tr.count = 0
        tr.test_wait_cycles = int(test_wait_cycles)
        if events:
            raise ValueError("test_wait_cycles is not combined with trace events")
        return ctypes.byref(tr), tr
    if not events:
        return None
    if len(events) > _lib.HLA_TRACE_MAX:
        raise ValueError(f"at most {_lib.HLA_TRACE_MAX} trace events")
    tr = _lib.HlaTrace()
    stream = torch.cuda.current_stream(device)
    for i, ev in enumerate(events):
        if not ev.cuda_event:  # torch creates the event on its first record
            ev.record(stream)
        tr.events[i] = ev.cuda_event
    tr.count = len(events)
    return ctypes.byref(tr), tr


def prefill(q, k, v, gate, gamma: Sequence[float] | torch.Tensor, state_in=None, *, chunk=64,
            pos_offset=0, rope_base=1e4, eps=1e-6, want_o=False, want_state=True, y=None,
            state_out=None, workspace=None, trace=None, saved=None, passes=0,
            test_wait_cycles=0):
    """hla_prefill.  Returns (y, o or None, state_out or None).  ``trace``: optional
    list of torch.cuda.Event recorded before each pass and after the last.
    ``saved``: optional uint8 CUDA tensor of ``saved_bytes(shape)`` bytes that
    receives the features for ``prefill_backward(..., saved=...)``.  ``passes``:
    0 (the library's choice), 1 (one launch) or 3 (local-state pass, scan,
    output pass)."""
    _check_acts(q, k, v, gate)
    B, T, H, d = q.shape
    _check_state(state_in, B, H, d, q.device)
    shape = make_shape(B, T, H, d, chunk=chunk, dtype=q.dtype, pos_offset=pos_offset,
                       rope_base=rope_base, eps=eps, passes=passes)
    lib = _lib.load()
    g_host, g_ptr = _host_gamma(gamma, H)
    if y is None:
        y = torch.empty_like(q)
    o = torch.empty(q.shape, dtype=torch.float32, device=q.device) if want_o else None
    if want_state and state_out is None:
        state_out = torch.empty((B, H, d, d), dtype=torch.float32, device=q.device)
    if not want_state:
        state_out = None
    ws_bytes = prefill_workspace_size(shape)
    if workspace is None:
        workspace = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device=q.device)
    _check_saved(saved, shape)
    tr = _trace(trace, q.device, test_wait_cycles)
    st = lib.hla_prefill(ctypes.byref(shape), _ptr(q), _ptr(k), _ptr(v), _ptr(gate), g_ptr,
                         _ptr(state_in), _ptr(state_out), _ptr(y), _ptr(o), _ptr(workspace),
                         workspace.numel(), _stream(q.device), tr[0] if tr else None,
                         _ptr(saved))
    _lib.check(st, "hla_prefill")
    del g_host
    return y, o, state_out


def decode_step(q, k, v, gate, gamma, state, pos=None, *, pos_offset=0, rope_base=1e4, eps=1e-6,
                state_out=None, want_o=False, y=None, split=0):
    """hla_decode_step on [B, 1, H, d] rows.  ``state_out`` defaults to ``state``
    (in-place update).  ``pos`` is an optional int64 CUDA tensor [B].  ``split``:
    CTAs per (sequence, head), 1, 2, 4 or 8; 0 lets the library choose."""
    _check_acts(q, k, v, gate)
    B, T, H, d = q.shape
    _check_state(state, B, H, d, q.device)
    if state_out is None:
        state_out = state
    _check_state(state_out, B, H, d, q.device)
    if pos is not None and (pos.dtype != torch.int64 or not pos.is_cuda or pos.numel() != B):
        raise ValueError("pos must be an int64 CUDA tensor with B entries")
    shape = make_shape(B, T, H, d, dtype=q.dtype, pos_offset=pos_offset, rope_base=rope_base,
                       eps=eps, decode_split=split)
    lib = _lib.load()
    g_host, g_ptr = _host_gamma(gamma, H)
    if y is None:
        y = torch.empty_like(q)
    o = torch.empty(q.shape, dtype=torch.float32, device=q.device) if want_o else None
    st = lib.hla_decode_step(ctypes.byref(shape), _ptr(q), _ptr(k), _ptr(v), _ptr(gate), g_ptr,
                             _ptr(pos), _ptr(state), _ptr(state_out), _ptr(y), _ptr(o),
                             _stream(q.device))
    _lib.check(st, "hla_decode_step")
    del g_host
    return y, o, state_out


def prefill_features(features, v, gate, gamma, state_in=None, *, chunk=64, pos_offset=0,
                     rope_base=1e4, eps=1e-6, want_o=False, want_state=True, y=None,
                     state_out=None, workspace=None, trace=None, passes=0):
    """hla_prefill_features: the forward from q~, k~ features (``features``: a
    uint8 CUDA tensor of ``saved_bytes(shape)`` bytes, e.g. from
    ``project_in``) and raw v, gate [B, T, H, d] bf16.  Returns
    (y, o or None, state_out or None)."""
    _check_acts(v, gate)
    B, T, H, d = v.shape
    _check_state(state_in, B, H, d, v.device)
    shape = make_shape(B, T, H, d, chunk=chunk, dtype=v.dtype, pos_offset=pos_offset,
                       rope_base=rope_base, eps=eps, passes=passes)
    _check_saved(features, shape)
    lib = _lib.load()
    g_host, g_ptr = _host_gamma(gamma, H)
    if y is None:
        y = torch.empty_like(v)
    o = torch.empty(v.shape, dtype=torch.float32, device=v.device) if want_o else None
    if want_state and state_out is None:
        state_out = torch.empty((B, H, d, d), dtype=torch.float32, device=v.device)
    if not want_state:
        state_out = None
    if workspace is None:
        workspace = torch.empty(max(prefill_workspace_size(shape), 16), dtype=torch.uint8,
                                device=v.device)
    tr = _trace(trace, v.device)
    st = lib.hla_prefill_features(ctypes.byref(shape), _ptr(features), _ptr(v), _ptr(gate), g_ptr,
                                  _ptr(state_in), _ptr(state_out), _ptr(y), _ptr(o),
                                  _ptr(workspace), workspace.numel(), _stream(v.device),
                                  tr[0] if tr else None)
    _lib.check(st, "hla_prefill_features")
    del g_host
    return y, o, state_out


def prefill_backward(q, k, v, gate, gamma, dy, state_in=None, dstate_out=None, *, chunk=64,
                     pos_offset=0, rope_base=1e4, eps=1e-6, want_dstate_in=False,
                     workspace=None, trace=None, fwd_workspace=None, saved=None, y=None):
    """hla_prefill_backward.  Returns (dq, dk, dv, dgate, dstate_in or None).
    ``fwd_workspace``: the ``workspace`` of a ``prefill`` call on the same
    shape, inputs, gamma and state_in, enqueued earlier on this stream; the
    backward then reads the forward's segment states instead of recomputing
    them.  ``saved``: the ``saved`` buffer of such a call (or the features of
    ``project_in``); the backward reads the q / k features from it, and q and
    k may then be None.  ``y``: with ``saved``, the output of the forward call
    that wrote it; the dq pass then takes the normalized output from y
    instead of recomputing o."""
    if saved is not None and q is None and k is None:
        _check_acts(v, gate, dy)
        ref = v
    else:
        _check_acts(q, k, v, gate, dy)
        ref = q
    B, T, H, d = ref.shape
    _check_state(state_in, B, H, d, ref.device)
    _check_state(dstate_out, B, H, d, ref.device)
    shape = make_shape(B, T, H, d, chunk=chunk, dtype=ref.dtype, pos_offset=pos_offset,
                       rope_base=rope_base, eps=eps)
    lib = _lib.load()
    g_host, g_ptr = _host_gamma(gamma, H)
    dq, dk, dv, dg = (torch.empty_like(ref) for _ in range(4))
    dsi = torch.empty((B, H, d, d), dtype=torch.float32, device=ref.device) if want_dstate_in else None
    ws_bytes = backward_workspace_size(shape)
    if workspace is None:
        workspace = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device=ref.device)
    _check_saved(saved, shape)
    if y is not None:
        if saved is None:
            raise ValueError("y is used only with saved features")
        _check_acts(y)
        if tuple(y.shape) != (B, T, H, d) or y.dtype != ref.dtype:
            raise ValueError("y must be the forward's output, shaped like v")
    tr = _trace(trace, ref.device)
    st = lib.hla_prefill_backward(ctypes.byref(shape), _ptr(q), _ptr(k), _ptr(v), _ptr(gate), g_ptr,
                                  _ptr(state_in), _ptr(dy), _ptr(dstate_out), _ptr(dq), _ptr(dk),
                                  _ptr(dv), _ptr(dg), _ptr(dsi), _ptr(workspace), workspace.numel(),
                                  _stream(ref.device), tr[0] if tr else None, _ptr(fwd_workspace),
                                  _ptr(saved), _ptr(y))
    _lib.check(st, "hla_prefill_backward")
    del g_host
    return dq, dk, dv, dg, dsi


def make_attn_shape(B, T, Hq, Hkv, d, *, a, dtype=torch.bfloat16, pos_offset=0,
                    eps=1e-6) -> _lib.HlaAttnShape:
    return _lib.HlaAttnShape(B=B, T=T, Hq=Hq, Hkv=Hkv, d=d, dtype=_DTYPES[dtype],
                             pos_offset=int(pos_offset), a=float(a), norm_eps=float(eps))


def attention_workspace_size(shape: _lib.HlaAttnShape) -> int:
    return int(_lib.load().hla_attention_workspace_size(ctypes.byref(shape)))


def attention_prefill(q, k, v, gate, a: float, *, pos_offset=0, eps=1e-6, want_o=False, y=None,
                      workspace=None):
    """hla_attention_prefill: causal softmax attention with the logit scale
    log_a(p + 1 + a), output norm and gate.  q, gate [B, T, Hq, d]; k, v
    [B, T, Hkv, d] (Hkv divides Hq).  Returns (y, o or None)."""
    _check_acts(q, gate)
    _check_acts(k, v)
    B, T, Hq, d = q.shape
    Hkv = k.shape[2]
    if k.shape[:2] != (B, T) or k.shape[3] != d or k.dtype != q.dtype or k.device != q.device:
        raise ValueError("k, v must be [B, T, Hkv, d] with q's B, T, d, dtype and device")
    shape = make_attn_shape(B, T, Hq, Hkv, d, a=a, dtype=q.dtype, pos_offset=pos_offset, eps=eps)
    lib = _lib.load()
    if y is None:
        y = torch.empty_like(q)
    o = torch.empty(q.shape, dtype=torch.float32, device=q.device) if want_o else None
    if workspace is None:
        workspace = torch.empty(max(attention_workspace_size(shape), 16), dtype=torch.uint8,
                                device=q.device)
    st = lib.hla_attention_prefill(ctypes.byref(shape), _ptr(q), _ptr(k), _ptr(v), _ptr(gate),
                                   _ptr(y), _ptr(o), _ptr(workspace), workspace.numel(),
                                   _stream(q.device))
    _lib.check(st, "hla_attention_prefill")
    return y, o


def project_workspace_size() -> int:
    return int(_lib.load().hla_project_workspace_size())


def project_in(x, w_qkvz, *, pos_offset=0, rope_base=1e4, eps=1e-6, chunk=64, features=None,
               v=None, gate=None, workspace=None):
    """hla_project_in: x [B, T, D] bf16 and w_qkvz [H, 4, d, D] bf16 (per head the
    transposes of W_q, W_k, W_v, W_z).  Returns (features, v, gate): features a
    uint8 tensor in the saved layout (q~, k~ fp16 and the fp32 scalars), v and
    gate bf16 [B, T, H, d]."""
    if not (x.is_cuda and w_qkvz.is_cuda) or x.dtype != torch.bfloat16 or w_qkvz.dtype != torch.bfloat16:
        raise ValueError("x and w_qkvz are bf16 CUDA tensors (no CPU path)")
    if x.dim() != 3 or w_qkvz.dim() != 4 or w_qkvz.shape[1] != 4 or w_qkvz.shape[3] != x.shape[2]:
        raise ValueError("x must be [B, T, D] and w_qkvz [H, 4, d, D]")
    if not (x.is_contiguous() and w_qkvz.is_contiguous()):
        raise ValueError("x and w_qkvz must be contiguous")
    B, T, Dm = x.shape
    H, _, d, _ = w_qkvz.shape
    shape = make_shape(B, T, H, d, chunk=chunk, dtype=torch.bfloat16, pos_offset=pos_offset,
                       rope_base=rope_base, eps=eps)
    lib = _lib.load()
    if features is None:
        features = torch.empty(max(saved_bytes(shape), 16), dtype=torch.uint8, device=x.device)
    _check_saved(features, shape)
    if v is None:
        v = torch.empty((B, T, H, d), dtype=torch.bfloat16, device=x.device)
    if gate is None:
        gate = torch.empty((B, T, H, d), dtype=torch.bfloat16, device=x.device)
    if workspace is None:
        workspace = torch.empty(project_workspace_size(), dtype=torch.uint8, device=x.device)
    st = lib.hla_project_in(ctypes.byref(shape), Dm, _ptr(x), _ptr(w_qkvz), _ptr(features),
                            _ptr(v), _ptr(gate), _ptr(workspace), workspace.numel(),
                            _stream(x.device))
    _lib.check(st, "hla_project_in")
    return features, v, gate


def project_out(u, w_o, *, out=None, workspace=None):
    """hla_project_out: u [..., n_in] bf16 (e.g. y [B, T, H, d] with n_in = H d
    folded), w_o [D, n_in] bf16.  Returns out [rows, D] shaped like u's leading
    dimensions plus D."""
    if not (u.is_cuda and w_o.is_cuda) or u.dtype != torch.bfloat16 or w_o.dtype != torch.bfloat16:
        raise ValueError("u and w_o are bf16 CUDA tensors (no CPU path)")
    if not (u.is_contiguous() and w_o.is_contiguous()) or w_o.dim() != 2:
        raise ValueError("u and w_o must be contiguous, w_o [D, n_in]")
    Dm, n_in = w_o.shape
    if u.dim() == 4:  # [B, T, H, d]
        lead = u.shape[:2]
        if u.shape[2] * u.shape[3] != n_in:
            raise ValueError("u's heads times d must equal w_o's columns")
    else:
        lead = u.shape[:-1]
        if u.shape[-1] != n_in:
            raise ValueError("u's last dimension must equal w_o's columns")
    M = u.numel() // n_in
    lib = _lib.load()
    if out is None:
        out = torch.empty(tuple(lead) + (Dm,), dtype=torch.bfloat16, device=u.device)
    if workspace is None:
        workspace = torch.empty(project_workspace_size(), dtype=torch.uint8, device=u.device)
    st = lib.hla_project_out(M, n_in, Dm, _ptr(u), _ptr(w_o), _ptr(out), _ptr(workspace),
                             workspace.numel(), _stream(u.device))
    _lib.check(st, "hla_project_out")
    return out
