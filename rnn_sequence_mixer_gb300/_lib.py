"""ctypes binding of libhla.so: the C structs, the status codes and the raw
entry points with the same names as ``include/hla.h``.  Argument marshalling
only; every step of the mixer runs in the library's CUDA kernels."""
from __future__ import annotations

import ctypes
import os

from . import build as _build

HLA_OK = 0
HLA_ERR_INVALID_ARG = 1
HLA_ERR_UNSUPPORTED = 2
HLA_ERR_WORKSPACE = 3
HLA_ERR_CUDA = 4
HLA_ERR_TIMEOUT = 5

HLA_F32 = 0
HLA_BF16 = 1

# Every symbol include/hla.h declares (checked by the ABI tests).
EXPORTS = (
    "hla_abi_version",
    "hla_status_string",
    "hla_gamma_schedule",
    "hla_prefill_workspace_size",
    "hla_prefill_launches",
    "hla_backward_launches",
    "hla_saved_bytes",
    "hla_prefill",
    "hla_decode_step",
    "hla_backward_workspace_size",
    "hla_prefill_backward",
    "hla_prefill_features",
    "hla_prefill_noalloc",
    "hla_attention_workspace_size",
    "hla_attention_prefill",
    "hla_project_workspace_size",
    "hla_project_in",
    "hla_project_out",
)


class HlaShape(ctypes.Structure):
    _fields_ = [
        ("B", ctypes.c_int32),
        ("T", ctypes.c_int32),
        ("H", ctypes.c_int32),
        ("dk", ctypes.c_int32),
        ("dv", ctypes.c_int32),
        ("chunk", ctypes.c_int32),
        ("dtype", ctypes.c_int32),
        ("decode_split", ctypes.c_int32),
        ("pos_offset", ctypes.c_int64),
        ("rope_base", ctypes.c_double),
        ("norm_eps", ctypes.c_float),
        ("passes", ctypes.c_int32),
    ]


class HlaAttnShape(ctypes.Structure):
    _fields_ = [
        ("B", ctypes.c_int32),
        ("T", ctypes.c_int32),
        ("Hq", ctypes.c_int32),
        ("Hkv", ctypes.c_int32),
        ("d", ctypes.c_int32),
        ("dtype", ctypes.c_int32),
        ("pos_offset", ctypes.c_int64),
        ("a", ctypes.c_double),
        ("norm_eps", ctypes.c_float),
    ]


HLA_TRACE_MAX = 16


class HlaTrace(ctypes.Structure):
    _fields_ = [("events", ctypes.c_void_p * HLA_TRACE_MAX), ("count", ctypes.c_int32),
                ("test_wait_cycles", ctypes.c_int64)]


class HlaError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_string(status)}")


_lib = None


def lib_path() -> str:
    return _build.LIB


def load(build_if_missing: bool = True) -> ctypes.CDLL:
    """Load libhla.so (building it first if needed).  Raises if it cannot."""
    global _lib
    if _lib is not None:
        return _lib
    if build_if_missing and not _build.up_to_date():
        _build.build()
    if not os.path.exists(_build.LIB):
        raise RuntimeError("libhla.so is not built; run rnn_sequence_mixer_gb300.build.build()")
    lib = ctypes.CDLL(_build.LIB)
    vp, sz, f32p, i64p = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p, ctypes.c_void_p
    shp = ctypes.POINTER(HlaShape)
    lib.hla_abi_version.restype = ctypes.c_int
    lib.hla_status_string.restype = ctypes.c_char_p
    lib.hla_status_string.argtypes = [ctypes.c_int]
    lib.hla_gamma_schedule.restype = ctypes.c_int
    lib.hla_gamma_schedule.argtypes = [ctypes.c_int32, ctypes.POINTER(ctypes.c_float)]
    lib.hla_prefill_workspace_size.restype = sz
    lib.hla_prefill_workspace_size.argtypes = [shp]
    fp = ctypes.POINTER(ctypes.c_float)
    lib.hla_prefill_launches.restype = ctypes.c_int32
    lib.hla_prefill_launches.argtypes = [shp, fp]
    lib.hla_backward_launches.restype = ctypes.c_int32
    lib.hla_backward_launches.argtypes = [shp, fp, ctypes.c_int32]
    lib.hla_saved_bytes.restype = sz
    lib.hla_saved_bytes.argtypes = [shp]
    lib.hla_backward_workspace_size.restype = sz
    lib.hla_backward_workspace_size.argtypes = [shp]
    lib.hla_prefill.restype = ctypes.c_int
    trp = ctypes.POINTER(HlaTrace)
    lib.hla_prefill.argtypes = [shp, vp, vp, vp, vp, ctypes.POINTER(ctypes.c_float), f32p, f32p, vp,
                                f32p, vp, sz, vp, trp, vp]
    lib.hla_decode_step.restype = ctypes.c_int
    lib.hla_decode_step.argtypes = [shp, vp, vp, vp, vp, ctypes.POINTER(ctypes.c_float), i64p,
                                    f32p, f32p, vp, f32p, vp]
    lib.hla_prefill_backward.restype = ctypes.c_int
    lib.hla_prefill_backward.argtypes = [shp, vp, vp, vp, vp, ctypes.POINTER(ctypes.c_float), f32p,
                                         vp, f32p, vp, vp, vp, vp, f32p, vp, sz, vp, trp, vp, vp, vp]
    lib.hla_prefill_features.restype = ctypes.c_int
    lib.hla_prefill_features.argtypes = [shp, vp, vp, vp, ctypes.POINTER(ctypes.c_float), f32p,
                                         f32p, vp, f32p, vp, sz, vp, trp]
    lib.hla_project_workspace_size.restype = sz
    lib.hla_project_workspace_size.argtypes = []
    lib.hla_project_in.restype = ctypes.c_int
    lib.hla_project_in.argtypes = [shp, ctypes.c_int32, vp, vp, vp, vp, vp, vp, sz, vp]
    lib.hla_project_out.restype = ctypes.c_int
    lib.hla_project_out.argtypes = [ctypes.c_int64, ctypes.c_int32, ctypes.c_int32, vp, vp, vp, vp,
                                    sz, vp]
    lib.hla_prefill_noalloc.restype = ctypes.c_int
    lib.hla_prefill_noalloc.argtypes = [shp, vp, vp, vp, vp, ctypes.POINTER(ctypes.c_float), f32p,
                                        f32p, vp, f32p, vp]
    ashp = ctypes.POINTER(HlaAttnShape)
    lib.hla_attention_workspace_size.restype = sz
    lib.hla_attention_workspace_size.argtypes = [ashp]
    lib.hla_attention_prefill.restype = ctypes.c_int
    lib.hla_attention_prefill.argtypes = [ashp, vp, vp, vp, vp, vp, f32p, vp, sz, vp]
    _lib = lib
    return lib


def status_string(status: int) -> str:
    return load().hla_status_string(int(status)).decode()


def check(status: int, where: str) -> None:
    if status != HLA_OK:
        raise HlaError(status, where)
