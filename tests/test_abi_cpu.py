"""Host-side checks of the C ABI that need no GPU: the library loads, exports
every entry point include/hla.h declares, computes the Eq. 19 schedule, and
rejects bad arguments with the documented status before any launch.

Every call below carries at least one invalid argument, so validation returns
before the library touches the CUDA runtime; the fake device addresses are
never dereferenced."""
import ctypes
import os
import re
import subprocess

import numpy as np
import pytest
import torch

import oracle
from rnn_sequence_mixer_gb300 import _lib, api, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "hla.h")
FAKE = 0x7F0000000000  # 16-byte aligned, never dereferenced


@pytest.fixture(scope="module")
def lib():
    return _lib.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(hla_[a-z_]+)\s*\(", text)))


def test_header_declares_the_binding_exports():
    assert declared_functions() == sorted(_lib.EXPORTS)


def test_library_exports_every_declared_symbol(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", build.LIB], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r"\bT (hla_\w+)", out))
    missing = set(declared_functions()) - exported
    assert not missing, missing
    for name in declared_functions():
        assert hasattr(lib, name)


def test_abi_version_and_status_strings(lib):
    assert lib.hla_abi_version() == 7
    for code in range(6):
        assert _lib.status_string(code).startswith("HLA_")
    assert "UNKNOWN" in _lib.status_string(99)


def test_gamma_schedule_matches_oracle_and_table(lib):
    for H in (1, 2, 16, 32, 256):
        mine = api.gamma_schedule(H).numpy()
        ref = oracle.gamma(H).astype(np.float32)
        assert np.max(np.abs(mine - ref) / np.spacing(ref)) <= 1.0
    rows = [float(l) for l in open(os.path.join(ROOT, "tests", "golden", "gamma_H32.txt"))
            if l.strip() and not l.startswith("#")]
    table = np.array(rows, dtype=np.float32)
    assert np.max(np.abs(api.gamma_schedule(32).numpy() - table) / np.spacing(table)) <= 1.0
    assert lib.hla_gamma_schedule(0, None) == _lib.HLA_ERR_INVALID_ARG


def shape(**kw):
    base = dict(B=1, T=128, H=2, d=64, chunk=64, dtype=torch.bfloat16, pos_offset=0,
                rope_base=1e4, eps=1e-6)
    base.update(kw)
    return api.make_shape(base.pop("B"), base.pop("T"), base.pop("H"), base.pop("d"), **base)


def test_workspace_sizes():
    s = shape(B=1, T=524288, H=16, d=128)
    n = api.prefill_workspace_size(s)
    assert n > 256 and (n - 256) % (128 * 128 * 4) == 0
    bw = api.backward_workspace_size(s)
    # the backward holds what the forward does (segment states and the local-state
    # pass's partial sums), a second set of segment states and an fp32-sized dO region
    assert bw >= (n - 256) + 16 * 128 * 128 * 4 + 524288 * 16 * 128 * 4
    bad = shape(d=96)
    assert api.prefill_workspace_size(bad) == 0
    assert api.backward_workspace_size(bad) == 0
    # one segment state per (b, h, segment), at least one segment per (b, h)
    tiny = shape(B=1, T=1, H=1, d=64)
    assert api.prefill_workspace_size(tiny) == 64 * 64 * 4 + 256
    # an empty sequence or batch needs only the status word
    for empty in (shape(T=0), shape(B=0), shape(B=0, T=0)):
        assert api.prefill_workspace_size(empty) == 256
        assert api.backward_workspace_size(empty) == 256


def _gamma(H, value=0.9):
    arr = (ctypes.c_float * H)(*([value] * H))
    return ctypes.cast(arr, ctypes.POINTER(ctypes.c_float)), arr


def call_prefill(lib, s, gamma=None, q=FAKE, y=FAKE, ws=FAKE, ws_bytes=1 << 40, saved=None):
    gp, keep = _gamma(s.H) if gamma is None else gamma
    return lib.hla_prefill(ctypes.byref(s), q, FAKE, FAKE, FAKE, gp, None, None, y, None, ws,
                           ws_bytes, None, None, saved)


@pytest.mark.parametrize("kw,code", [
    (dict(d=96), _lib.HLA_ERR_UNSUPPORTED),
    (dict(chunk=32), _lib.HLA_ERR_UNSUPPORTED),
    (dict(T=-1), _lib.HLA_ERR_INVALID_ARG),
    (dict(B=-1), _lib.HLA_ERR_INVALID_ARG),
    (dict(H=257), _lib.HLA_ERR_UNSUPPORTED),
    (dict(pos_offset=-1), _lib.HLA_ERR_INVALID_ARG),
    (dict(rope_base=0.0), _lib.HLA_ERR_INVALID_ARG),
    (dict(eps=float("nan")), _lib.HLA_ERR_INVALID_ARG),
])
def test_prefill_rejects_bad_shapes(lib, kw, code):
    assert call_prefill(lib, shape(**kw)) == code


def test_prefill_rejects_bad_pointers_gamma_and_workspace(lib):
    s = shape()
    assert lib.hla_prefill(None, FAKE, FAKE, FAKE, FAKE, _gamma(2)[0], None, None, FAKE, None,
                           FAKE, 1 << 40, None, None, None) == _lib.HLA_ERR_INVALID_ARG
    bad_trace = _lib.HlaTrace()
    bad_trace.count = _lib.HLA_TRACE_MAX + 1
    assert lib.hla_prefill(ctypes.byref(s), FAKE, FAKE, FAKE, FAKE, _gamma(2)[0], None, None, FAKE,
                           None, FAKE, 1 << 40, None,
                           ctypes.byref(bad_trace), None) == _lib.HLA_ERR_INVALID_ARG
    assert call_prefill(lib, s, q=None) == _lib.HLA_ERR_INVALID_ARG
    assert call_prefill(lib, s, q=FAKE + 8) == _lib.HLA_ERR_INVALID_ARG
    assert call_prefill(lib, s, y=FAKE + 2) == _lib.HLA_ERR_INVALID_ARG
    for bad in (0.0, -0.5, 1.0001, float("nan"), float("inf")):
        assert call_prefill(lib, s, gamma=_gamma(2, bad)) == _lib.HLA_ERR_INVALID_ARG
    need = api.prefill_workspace_size(s)
    assert call_prefill(lib, s, ws=None) == _lib.HLA_ERR_WORKSPACE
    assert call_prefill(lib, s, ws_bytes=need - 1) == _lib.HLA_ERR_WORKSPACE
    assert call_prefill(lib, s, ws=FAKE + 4) == _lib.HLA_ERR_WORKSPACE
    r = s
    r.decode_split = 1  # a decode-step field: must be 0 for the prefill
    assert call_prefill(lib, r) == _lib.HLA_ERR_INVALID_ARG


def call_noalloc(lib, s, gamma=None, q=FAKE, k=FAKE, y=FAKE, state_in=None, state_out=None, o=None):
    gp, keep = _gamma(s.H) if gamma is None else gamma
    return lib.hla_prefill_noalloc(ctypes.byref(s), q, k, FAKE, FAKE, gp, state_in, state_out, y,
                                   o, None)


@pytest.mark.parametrize("kw,code", [
    (dict(d=96), _lib.HLA_ERR_UNSUPPORTED),
    (dict(chunk=32), _lib.HLA_ERR_UNSUPPORTED),
    (dict(T=-1), _lib.HLA_ERR_INVALID_ARG),
    (dict(B=-1), _lib.HLA_ERR_INVALID_ARG),
    (dict(H=257), _lib.HLA_ERR_UNSUPPORTED),
    (dict(pos_offset=-1), _lib.HLA_ERR_INVALID_ARG),
    (dict(rope_base=float("inf")), _lib.HLA_ERR_INVALID_ARG),
])
def test_noalloc_rejects_bad_shapes(lib, kw, code):
    assert call_noalloc(lib, shape(**kw)) == code


def test_noalloc_rejects_bad_pointers_and_gamma(lib):
    """Every check of hla_prefill_noalloc runs before its per-device set-up,
    so none of these calls touches the CUDA runtime."""
    s = shape()
    gp, keep = _gamma(2)
    assert lib.hla_prefill_noalloc(None, FAKE, FAKE, FAKE, FAKE, gp, None, None, FAKE, None,
                                   None) == _lib.HLA_ERR_INVALID_ARG
    assert call_noalloc(lib, s, q=None) == _lib.HLA_ERR_INVALID_ARG
    assert call_noalloc(lib, s, k=FAKE + 8) == _lib.HLA_ERR_INVALID_ARG
    assert call_noalloc(lib, s, y=None) == _lib.HLA_ERR_INVALID_ARG
    assert call_noalloc(lib, s, y=FAKE + 2) == _lib.HLA_ERR_INVALID_ARG
    assert call_noalloc(lib, s, state_in=FAKE + 4) == _lib.HLA_ERR_INVALID_ARG
    assert call_noalloc(lib, s, state_out=FAKE + 12) == _lib.HLA_ERR_INVALID_ARG
    assert call_noalloc(lib, s, o=FAKE + 1) == _lib.HLA_ERR_INVALID_ARG
    for bad in (0.0, -0.5, 1.0001, float("nan"), float("inf")):
        assert call_noalloc(lib, s, gamma=_gamma(2, bad)) == _lib.HLA_ERR_INVALID_ARG
    assert lib.hla_prefill_noalloc(ctypes.byref(s), FAKE, FAKE, FAKE, FAKE, None, None, None, FAKE,
                                   None, None) == _lib.HLA_ERR_INVALID_ARG
    # an empty call may pass NULL tensors, but not misaligned ones
    assert call_noalloc(lib, shape(B=0), q=FAKE + 4) == _lib.HLA_ERR_INVALID_ARG
    assert call_noalloc(lib, shape(T=0), state_out=FAKE + 4) == _lib.HLA_ERR_INVALID_ARG
    # more heads than the scratch array holds states for: refused before the set-up
    assert call_noalloc(lib, shape(B=16, T=8, H=64, d=128)) == _lib.HLA_ERR_WORKSPACE


def test_decode_rejects_bad_arguments(lib):
    gp, keep = _gamma(2)
    s = shape(T=2)
    assert lib.hla_decode_step(ctypes.byref(s), FAKE, FAKE, FAKE, FAKE, gp, None, FAKE, FAKE, FAKE,
                               None, None) == _lib.HLA_ERR_INVALID_ARG
    s = shape(T=1)
    # state buffers overlapping without being the same buffer
    assert lib.hla_decode_step(ctypes.byref(s), FAKE, FAKE, FAKE, FAKE, gp, None, FAKE, FAKE + 256,
                               FAKE, None, None) == _lib.HLA_ERR_INVALID_ARG
    assert lib.hla_decode_step(ctypes.byref(s), FAKE, FAKE, FAKE, FAKE, gp, FAKE + 4, FAKE, FAKE,
                               FAKE, None, None) == _lib.HLA_ERR_INVALID_ARG
    assert lib.hla_decode_step(ctypes.byref(s), FAKE, FAKE, FAKE, FAKE, gp, None, None, FAKE, FAKE,
                               None, None) == _lib.HLA_ERR_INVALID_ARG
    assert lib.hla_decode_step(ctypes.byref(shape(T=1, d=32)), FAKE, FAKE, FAKE, FAKE, gp, None,
                               FAKE, FAKE, FAKE, None, None) == _lib.HLA_ERR_UNSUPPORTED
    # CTAs per (sequence, head): 0 (library's choice), 1, 2, 4 or 8
    for bad in (-1, 3, 5, 6, 16):
        r = shape(T=1)
        r.decode_split = bad
        assert lib.hla_decode_step(ctypes.byref(r), FAKE, FAKE, FAKE, FAKE, gp, None, FAKE, FAKE,
                                   FAKE, None, None) == _lib.HLA_ERR_INVALID_ARG


def test_backward_rejects_bad_arguments(lib):
    gp, keep = _gamma(2)
    s = shape()
    need = api.backward_workspace_size(s)
    args = lambda **kw: [kw.get(n, FAKE) for n in ("q", "k", "v", "g")]
    assert lib.hla_prefill_backward(ctypes.byref(s), *args(), gp, None, FAKE, None, FAKE, FAKE,
                                    FAKE, FAKE, None, FAKE, need - 16,
                                    None, None, None, None, None) == _lib.HLA_ERR_WORKSPACE
    assert lib.hla_prefill_backward(ctypes.byref(s), *args(), gp, None, None, None, FAKE, FAKE,
                                    FAKE, FAKE, None, FAKE, need, None,
                                    None, None, None, None) == _lib.HLA_ERR_INVALID_ARG
    assert lib.hla_prefill_backward(ctypes.byref(s), *args(), gp, None, FAKE, None, FAKE, FAKE,
                                    FAKE, FAKE + 1, None, FAKE, need,
                                    None, None, None, None, None) == _lib.HLA_ERR_INVALID_ARG
    # a misaligned forward workspace
    assert lib.hla_prefill_backward(ctypes.byref(s), *args(), gp, None, FAKE, None, FAKE, FAKE,
                                    FAKE, FAKE, None, FAKE, need, None, None,
                                    FAKE + 4, None, None) == _lib.HLA_ERR_INVALID_ARG
    # saved features: misaligned, and on a shape that cannot save them
    assert lib.hla_prefill_backward(ctypes.byref(s), *args(), gp, None, FAKE, None, FAKE, FAKE,
                                    FAKE, FAKE, None, FAKE, need, None, None, None,
                                    FAKE + 4, None) == _lib.HLA_ERR_INVALID_ARG
    s64 = shape(d=64)
    assert lib.hla_prefill_backward(ctypes.byref(s64), *args(), gp, None, FAKE, None, FAKE, FAKE,
                                    FAKE, FAKE, None, FAKE, 1 << 40, None, None, None,
                                    FAKE, None) == _lib.HLA_ERR_UNSUPPORTED
    # the forward's y: only with saved features, and 16-byte aligned
    s128 = shape(d=128)
    need128 = api.backward_workspace_size(s128)
    assert lib.hla_prefill_backward(ctypes.byref(s128), *args(), gp, None, FAKE, None, FAKE, FAKE,
                                    FAKE, FAKE, None, FAKE, need128, None, None, None,
                                    None, FAKE) == _lib.HLA_ERR_INVALID_ARG
    assert lib.hla_prefill_backward(ctypes.byref(s128), *args(), gp, None, FAKE, None, FAKE, FAKE,
                                    FAKE, FAKE, None, FAKE, need128, None, None, None,
                                    FAKE, FAKE + 2) == _lib.HLA_ERR_INVALID_ARG


def test_saved_feature_bytes_and_checks(lib):
    # fp16 q~ and k~ plus four fp32 scalars per row, on the tensor-core path only
    s = shape(B=2, T=1000, H=3, d=128)
    assert api.saved_bytes(s) == 2 * 1000 * 3 * (4 * 128 + 16)
    assert api.saved_bytes(shape(B=2, T=1000, H=3, d=64)) == 0
    assert api.saved_bytes(shape(B=2, T=1000, H=3, d=128, dtype=torch.float32)) == 0
    assert api.saved_bytes(shape(d=96)) == 0
    assert api.saved_bytes(shape(B=0, d=128)) == 0
    assert call_prefill(lib, s, saved=FAKE + 8) == _lib.HLA_ERR_INVALID_ARG
    assert call_prefill(lib, shape(d=64), saved=FAKE) == _lib.HLA_ERR_UNSUPPORTED
    assert call_prefill(lib, shape(d=128, dtype=torch.float32), saved=FAKE) == _lib.HLA_ERR_UNSUPPORTED


def test_python_api_has_no_cpu_path():
    x = torch.zeros(1, 4, 2, 64)
    with pytest.raises(ValueError):
        api.prefill(x, x, x, x, [0.5, 0.5])
    with pytest.raises(ValueError):
        api.decode_step(x[:, :1], x[:, :1], x[:, :1], x[:, :1], [0.5, 0.5],
                        torch.zeros(1, 2, 64, 64))


def attn_shape(**kw):
    base = dict(B=1, T=256, Hq=4, Hkv=2, d=128, a=500.0, dtype=torch.bfloat16, pos_offset=0,
                eps=1e-6)
    base.update(kw)
    return api.make_attn_shape(base.pop("B"), base.pop("T"), base.pop("Hq"), base.pop("Hkv"),
                               base.pop("d"), **base)


def call_attention(lib, s, q=FAKE, y=FAKE, o=None, ws=FAKE, ws_bytes=256):
    return lib.hla_attention_prefill(ctypes.byref(s), q, FAKE, FAKE, FAKE, y, o, ws, ws_bytes, None)


def test_attention_workspace_and_argument_checks(lib):
    assert api.attention_workspace_size(attn_shape()) == 256
    assert api.attention_workspace_size(attn_shape(Hkv=3)) == 0
    for kw, code in [(dict(Hkv=3), _lib.HLA_ERR_INVALID_ARG),     # Hkv must divide Hq
                     (dict(a=1.0), _lib.HLA_ERR_INVALID_ARG),     # log base a > 1
                     (dict(a=float("nan")), _lib.HLA_ERR_INVALID_ARG),
                     (dict(T=-1), _lib.HLA_ERR_INVALID_ARG),
                     (dict(pos_offset=-5), _lib.HLA_ERR_INVALID_ARG),
                     (dict(d=64), _lib.HLA_ERR_UNSUPPORTED),
                     (dict(dtype=torch.float32), _lib.HLA_ERR_UNSUPPORTED),
                     (dict(Hq=512, Hkv=2), _lib.HLA_ERR_UNSUPPORTED)]:
        assert call_attention(lib, attn_shape(**kw)) == code, kw
    s = attn_shape()
    assert lib.hla_attention_prefill(None, FAKE, FAKE, FAKE, FAKE, FAKE, None, FAKE, 256,
                                     None) == _lib.HLA_ERR_INVALID_ARG
    assert call_attention(lib, s, q=None) == _lib.HLA_ERR_INVALID_ARG
    assert call_attention(lib, s, y=FAKE + 2) == _lib.HLA_ERR_INVALID_ARG
    assert call_attention(lib, s, o=FAKE + 4) == _lib.HLA_ERR_INVALID_ARG
    assert call_attention(lib, s, ws=None) == _lib.HLA_ERR_WORKSPACE
    assert call_attention(lib, s, ws_bytes=255) == _lib.HLA_ERR_WORKSPACE


def test_projection_and_feature_entry_points_reject_bad_arguments(lib):
    """hla_project_in / hla_project_out / hla_prefill_features validate before
    touching the GPU (the fake addresses are never used)."""
    ws = api.project_workspace_size()
    assert ws == 256
    s = shape(B=1, T=128, H=2, d=128)
    pin = lambda s, d_model=256, x=FAKE, w=FAKE, f=FAKE, ws_bytes=ws: lib.hla_project_in(
        ctypes.byref(s), d_model, x, w, f, FAKE, FAKE, FAKE, ws_bytes, None)
    assert pin(s, d_model=0) == _lib.HLA_ERR_INVALID_ARG
    assert pin(s, d_model=96) == _lib.HLA_ERR_UNSUPPORTED       # not a multiple of 64
    assert pin(shape(d=64)) == _lib.HLA_ERR_UNSUPPORTED          # tensor cores: d = 128 only
    assert pin(shape(d=128, dtype=torch.float32)) == _lib.HLA_ERR_UNSUPPORTED
    assert pin(s, x=None) == _lib.HLA_ERR_INVALID_ARG
    assert pin(s, w=FAKE + 8) == _lib.HLA_ERR_INVALID_ARG
    assert pin(s, f=FAKE + 4) == _lib.HLA_ERR_INVALID_ARG
    assert pin(s, ws_bytes=255) == _lib.HLA_ERR_WORKSPACE
    pout = lambda M=100, n_in=256, D=256, u=FAKE, ws_bytes=ws: lib.hla_project_out(
        M, n_in, D, u, FAKE, FAKE, FAKE, ws_bytes, None)
    assert pout(M=-1) == _lib.HLA_ERR_INVALID_ARG
    assert pout(n_in=0) == _lib.HLA_ERR_INVALID_ARG
    assert pout(n_in=100) == _lib.HLA_ERR_UNSUPPORTED
    assert pout(D=192) == _lib.HLA_ERR_UNSUPPORTED
    assert pout(u=FAKE + 2) == _lib.HLA_ERR_INVALID_ARG
    assert pout(ws_bytes=0) == _lib.HLA_ERR_WORKSPACE
    gp, keep = _gamma(2)
    pf = lambda s, f=FAKE, ws_bytes=1 << 40: lib.hla_prefill_features(
        ctypes.byref(s), f, FAKE, FAKE, gp, None, None, FAKE, None, FAKE, ws_bytes, None, None)
    assert pf(s, f=None) == _lib.HLA_ERR_INVALID_ARG
    assert pf(s, f=FAKE + 4) == _lib.HLA_ERR_INVALID_ARG
    assert pf(shape(d=64)) == _lib.HLA_ERR_UNSUPPORTED
    assert pf(s, ws_bytes=16) == _lib.HLA_ERR_WORKSPACE


def test_launch_counts():
    """The library's choice is three passes (one launch on request)."""
    g16 = api.gamma_schedule(16)
    big = api.make_shape(1, 524288, 16, 128, chunk=128)
    assert api.prefill_launches(big, g16) == 4  # local-state pass, its piece sums, scan, outputs
    assert api.prefill_launches(api.make_shape(1, 524288, 16, 128, chunk=128, passes=1), g16) == 1
    assert api.prefill_launches(api.make_shape(1, 524288, 16, 128, chunk=128, passes=3), g16) >= 3
    short = api.make_shape(1, 16384, 16, 128, chunk=64)
    assert api.prefill_launches(short, g16) >= 2
    assert api.prefill_launches(api.make_shape(1, 16384, 16, 128, chunk=64, passes=1), g16) == 1
    assert api.prefill_launches(api.make_shape(1, 100, 2, 64, chunk=64, dtype=torch.float32),
                                api.gamma_schedule(2)) == 3
    assert api.prefill_launches(api.make_shape(0, 100, 2, 128, chunk=64), api.gamma_schedule(2)) == 0
    # bad arguments
    assert api.prefill_launches(api.make_shape(1, 100, 2, 96, chunk=64), api.gamma_schedule(2)) == -1
    assert api.prefill_launches(api.make_shape(1, 100, 2, 128, chunk=64, passes=2),
                                api.gamma_schedule(2)) == -1


def test_trace_rejects_a_negative_test_wait_budget(lib):
    tr = _lib.HlaTrace()
    tr.test_wait_cycles = -1
    s = shape()
    assert lib.hla_prefill(ctypes.byref(s), FAKE, FAKE, FAKE, FAKE, _gamma(2)[0], None, None, FAKE,
                           None, FAKE, 1 << 40, None, ctypes.byref(tr), None) == _lib.HLA_ERR_INVALID_ARG
