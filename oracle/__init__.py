"""fp64 CPU oracle of the Lightning Attention RNN mixer (ctypes wrapper).

TEST INFRASTRUCTURE ONLY: the test suite, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` are the only
callers.  The product package never imports this module and shares no code with
it.  The arithmetic lives in ``hla_oracle.c`` (plain C, fp64, OpenMP over the
independent (b, h) recurrences); this file only compiles it with gcc and
marshals numpy arrays.

Every function follows arXiv 2601.22156 ("Hybrid Linear Attention Done
Right"), Appendix A, Eq. 18 (RNN layers) and Eq. 19 (forget gate).  Arrays are
float64, C-contiguous, activations [B, T, H, d], state [B, H, d, d]
(d_k rows, d_v fastest).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import tempfile

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "hla_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "libhla_oracle.so")
_lib = None

_dp = ctypes.POINTER(ctypes.c_double)
_i64p = ctypes.POINTER(ctypes.c_int64)


def build(force: bool = False) -> str:
    """Compile hla_oracle.c into a shared library (gcc -O2 -fopenmp)."""
    os.makedirs(_BUILD, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    fd, tmp = tempfile.mkstemp(suffix=".so", dir=_BUILD)
    os.close(fd)
    cmd = ["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is not None:
        return _lib
    lib = ctypes.CDLL(build())
    i, d64, dbl = ctypes.c_int, ctypes.c_int64, ctypes.c_double
    lib.hla_oracle_threads.restype = i
    lib.hla_oracle_set_threads.argtypes = [i]
    lib.hla_oracle_gamma.argtypes = [i, _dp]
    lib.hla_oracle_feature.argtypes = [i, _dp, d64, dbl, dbl, dbl, _dp]
    lib.hla_oracle_prefill.argtypes = [i, i, i, i, _dp, _dp, _dp, _dp, _dp, _dp, d64, dbl, dbl,
                                       _dp, _dp, _dp]
    lib.hla_oracle_prefill.restype = i
    lib.hla_oracle_prefill_chunked.argtypes = [i, i, i, i, i, _dp, _dp, _dp, _dp, _dp, _dp, d64,
                                               dbl, dbl, _dp, _dp, _dp]
    lib.hla_oracle_prefill_chunked.restype = i
    lib.hla_oracle_decode.argtypes = [i, i, i, _dp, _dp, _dp, _dp, _dp, _i64p, _dp, dbl, dbl,
                                      _dp, _dp, _dp]
    lib.hla_oracle_decode.restype = i
    lib.hla_oracle_backward.argtypes = [i, i, i, i, _dp, _dp, _dp, _dp, _dp, _dp, _dp, _dp, d64,
                                        dbl, dbl, _dp, _dp, _dp, _dp, _dp]
    lib.hla_oracle_backward.restype = i
    lib.hla_oracle_attention.argtypes = [i, i, i, i, i, _dp, _dp, _dp, _dp, dbl, d64, dbl, _dp,
                                         _dp]
    lib.hla_oracle_attention.restype = i
    lib.hla_oracle_matmul_nt.argtypes = [i, i, i, _dp, _dp, _dp]
    lib.hla_oracle_matmul_nt.restype = i
    _lib = lib
    return lib


def _f64(x):
    if x is None:
        return None
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _ptr(x):
    if x is None:
        return ctypes.cast(None, _dp)
    return x.ctypes.data_as(_dp)


def threads() -> int:
    """OpenMP threads the oracle uses (all host cores unless OMP_NUM_THREADS)."""
    return int(_load().hla_oracle_threads())


def set_threads(n: int) -> None:
    """Use n OpenMP threads for the following calls (timing on fewer cores)."""
    _load().hla_oracle_set_threads(int(n))


def gamma(H: int) -> np.ndarray:
    """Eq. 19 forget rates gamma_h = exp(-2^(-8(h+1)/H)), 0-based head h, fp64."""
    out = np.zeros(H, dtype=np.float64)
    _load().hla_oracle_gamma(H, _ptr(out))
    return out


def feature(x, pos: int, base: float, eps: float = 1e-6, scale: float = 1.0) -> np.ndarray:
    """Norm(x), rotated by RoPE at position ``pos``, times ``scale`` (one row)."""
    x = _f64(x)
    out = np.zeros_like(x)
    _load().hla_oracle_feature(x.shape[-1], _ptr(x), int(pos), float(base), float(eps),
                               float(scale), _ptr(out))
    return out


def _dims(q):
    if q.ndim != 4:
        raise ValueError("activations must be [B, T, H, d]")
    return q.shape


def prefill(q, k, v, g, gam, state_in=None, pos_offset=0, base=1e4, eps=1e-6):
    """Per-timestep recurrence of Eq. 18.  Returns (y, o, state_out)."""
    q, k, v, g, gam, state_in = map(_f64, (q, k, v, g, gam, state_in))
    B, T, H, d = _dims(q)
    y, o = np.zeros_like(q), np.zeros_like(q)
    st = np.zeros((B, H, d, d), dtype=np.float64)
    rc = _load().hla_oracle_prefill(B, T, H, d, _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(gam),
                                    _ptr(state_in), int(pos_offset), float(base), float(eps),
                                    _ptr(y), _ptr(o), _ptr(st))
    if rc:
        raise RuntimeError(f"oracle prefill failed ({rc})")
    return y, o, st


def prefill_chunked(q, k, v, g, gam, chunk, state_in=None, pos_offset=0, base=1e4, eps=1e-6):
    """Block (chunked) evaluation of the same mixer.  Returns (y, o, state_out)."""
    q, k, v, g, gam, state_in = map(_f64, (q, k, v, g, gam, state_in))
    B, T, H, d = _dims(q)
    y, o = np.zeros_like(q), np.zeros_like(q)
    st = np.zeros((B, H, d, d), dtype=np.float64)
    rc = _load().hla_oracle_prefill_chunked(B, T, H, d, int(chunk), _ptr(q), _ptr(k), _ptr(v),
                                            _ptr(g), _ptr(gam), _ptr(state_in), int(pos_offset),
                                            float(base), float(eps), _ptr(y), _ptr(o), _ptr(st))
    if rc:
        raise RuntimeError(f"oracle chunked prefill failed ({rc})")
    return y, o, st


def decode_step(q, k, v, g, gam, pos, state_in, base=1e4, eps=1e-6):
    """One token per sequence ([B, 1, H, d]); pos[b] is its RoPE position."""
    q, k, v, g, gam, state_in = map(_f64, (q, k, v, g, gam, state_in))
    B, T, H, d = _dims(q)
    if T != 1:
        raise ValueError("decode takes T == 1")
    pos = np.ascontiguousarray(np.asarray(pos, dtype=np.int64).reshape(B))
    y, o = np.zeros_like(q), np.zeros_like(q)
    st = np.zeros((B, H, d, d), dtype=np.float64)
    rc = _load().hla_oracle_decode(B, H, d, _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(gam),
                                   pos.ctypes.data_as(_i64p), _ptr(state_in), float(base),
                                   float(eps), _ptr(y), _ptr(o), _ptr(st))
    if rc:
        raise RuntimeError(f"oracle decode failed ({rc})")
    return y, o, st


def backward(q, k, v, g, gam, dy, state_in=None, dstate_out=None, pos_offset=0, base=1e4,
             eps=1e-6):
    """Chain-rule gradients.  Returns (dq, dk, dv, dg, dstate_in)."""
    q, k, v, g, gam, dy, state_in, dstate_out = map(
        _f64, (q, k, v, g, gam, dy, state_in, dstate_out))
    B, T, H, d = _dims(q)
    dq, dk, dv, dg = (np.zeros_like(q) for _ in range(4))
    dst = np.zeros((B, H, d, d), dtype=np.float64)
    rc = _load().hla_oracle_backward(B, T, H, d, _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(gam),
                                     _ptr(state_in), _ptr(dy), _ptr(dstate_out), int(pos_offset),
                                     float(base), float(eps), _ptr(dq), _ptr(dk), _ptr(dv),
                                     _ptr(dg), _ptr(dst))
    if rc:
        raise RuntimeError(f"oracle backward failed ({rc})")
    return dq, dk, dv, dg, dst


def attention(q, k, v, g, a, pos_offset=0, eps=1e-6):
    """Causal NoPE softmax attention with logit scaling s = log_a(p + 1 + a)
    (Section 5.1, Eq. 11; Appendix A, Eq. 17), output norm and gate.
    q, g [B, T, Hq, d]; k, v [B, T, Hkv, d].  Returns (y, o)."""
    q, k, v, g = map(_f64, (q, k, v, g))
    B, T, Hq, d = _dims(q)
    Hkv = k.shape[2]
    if k.shape != (B, T, Hkv, d) or v.shape != k.shape or g.shape != q.shape:
        raise ValueError("q, g [B, T, Hq, d] and k, v [B, T, Hkv, d]")
    y, o = np.zeros_like(q), np.zeros_like(q)
    rc = _load().hla_oracle_attention(B, T, Hq, Hkv, d, _ptr(q), _ptr(k), _ptr(v), _ptr(g),
                                      float(a), int(pos_offset), float(eps), _ptr(y), _ptr(o))
    if rc:
        raise RuntimeError(f"oracle attention failed ({rc})")
    return y, o


def matmul_nt(a, w) -> np.ndarray:
    """a [M, K] times w [N, K] transposed: out[m, n] = sum_k a[m, k] w[n, k]."""
    a, w = _f64(a), _f64(w)
    if a.ndim != 2 or w.ndim != 2 or a.shape[1] != w.shape[1]:
        raise ValueError("matmul_nt needs a [M, K] and w [N, K]")
    out = np.zeros((a.shape[0], w.shape[0]), dtype=np.float64)
    if _load().hla_oracle_matmul_nt(a.shape[0], w.shape[0], a.shape[1], _ptr(a), _ptr(w),
                                    _ptr(out)) != 0:
        raise ValueError("bad shape")
    return out


def project_in(x, w_qkvz):
    """The input projections of an RNN layer (Appendix A, Eq. 18): per head h
    q = x W_q,h, k = x W_k,h, v = x W_v,h and the gate logit x W_z,h, before
    the norms and the sigmoid.  x [B, T, D]; w_qkvz [H, 4, d, D] holds, for
    head h, the transposes of (W_q, W_k, W_v, W_z) in that order (row c of
    w_qkvz[h, j] is column c of the paper's d x d_h matrix).  Returns q, k, v,
    g as [B, T, H, d]."""
    x, w = _f64(x), _f64(w_qkvz)
    B, T, Dm = x.shape
    H, four, d, Dw = w.shape
    if four != 4 or Dw != Dm:
        raise ValueError("w_qkvz must be [H, 4, d, D]")
    out = matmul_nt(x.reshape(B * T, Dm), w.reshape(H * 4 * d, Dm)).reshape(B, T, H, 4, d)
    return tuple(np.ascontiguousarray(out[:, :, :, j, :]) for j in range(4))


def project_out(u, w_o):
    """The output projection (Appendix A, Eq. 18: y_t = u_t W_o^T), over all
    heads at once: u [B, T, H, d] (the gated, normalized mixer rows, heads
    concatenated), w_o [D, H d] (the paper's W_o of every head side by side:
    column h d + c belongs to head h).  Returns [B, T, D]."""
    u, w = _f64(u), _f64(w_o)
    B, T, H, d = u.shape
    if w.shape[1] != H * d:
        raise ValueError("w_o must be [D, H d]")
    return matmul_nt(u.reshape(B * T, H * d), w).reshape(B, T, w.shape[0])


def features(q, k, pos_offset=0, base=1e4, eps=1e-6):
    """The saved-feature quantities of a prefill (Appendix A, Eq. 18), per
    (b, t, h): q~ = RoPE(Norm(q)), k~ = RoPE(Norm(k)) / sqrt(d), 1 / RMS(q),
    1 / RMS(k) and q~ . k~.  Returns (q~, k~ [B, T, H, d], rq, rk, diag
    [B, H, T])."""
    q, k = _f64(q), _f64(k)
    B, T, H, d = _dims(q)
    qt = np.zeros_like(q)
    kt = np.zeros_like(k)
    sc = np.zeros((3, B, H, T), dtype=np.float64)
    for b in range(B):
        for t in range(T):
            for h in range(H):
                p = pos_offset + t
                qt[b, t, h] = feature(q[b, t, h], p, base, eps)
                kt[b, t, h] = feature(k[b, t, h], p, base, eps, 1.0 / np.sqrt(d))
                sc[0, b, h, t] = 1.0 / np.sqrt(np.mean(q[b, t, h] ** 2) + eps)
                sc[1, b, h, t] = 1.0 / np.sqrt(np.mean(k[b, t, h] ** 2) + eps)
                sc[2, b, h, t] = float(np.dot(qt[b, t, h], kt[b, t, h]))
    return qt, kt, sc[0], sc[1], sc[2]
