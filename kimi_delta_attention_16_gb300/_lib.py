"""ctypes declarations of libkda.so's C ABI (include/kda.h).  Marshalling only."""
from __future__ import annotations

import ctypes
import os
import threading

from . import build as _build

_lock = threading.Lock()
_lib = None

KDA_OK = 0
KDA_ERR_INVALID_ARG = 1
KDA_ERR_UNSUPPORTED = 2
KDA_ERR_WORKSPACE = 3
KDA_ERR_CUDA = 4
KDA_ERR_TIMEOUT = 5
KDA_ERR_DEVICE_ARG = 6
KDA_BF16 = 0
KDA_FP32 = 1
KDA_FLAG_FORCE_SIMT = 1
KDA_FLAG_NO_RECURRENT = 2
KDA_FLAG_TEST_DROP_STAGING = 4
KDA_PATH_SIMT, KDA_PATH_TENSOR_CORE, KDA_PATH_RECURRENT = 0, 1, 2
KDA_RECURRENT_MAX_LEN = 8
KDA_MAX_SEGMENTS = 16
KDA_EPI_NONE, KDA_EPI_DECAY, KDA_EPI_SIGMOID = 0, 1, 2
ABI_VERSION = 10401  # kda_backward with chunk records in its workspace

# Every symbol include/kda.h declares.
EXPORTED = ("kda_status_string", "kda_last_error", "kda_version", "kda_short_conv",
            "kda_prefill_workspace_size", "kda_prefill", "kda_prefill_plan", "kda_prefill_noalloc",
            "kda_decode_step", "kda_gemm", "kda_backward_workspace_size", "kda_backward")
NOALLOC_SCRATCH_BYTES = 64 << 20  # KDA_NOALLOC_SCRATCH_BYTES in include/kda.h

_vp = ctypes.c_void_p
_i64 = ctypes.c_int64
_int = ctypes.c_int
_f = ctypes.c_float


class PrefillArgs(ctypes.Structure):
    """Mirror of kda_prefill_args."""
    _fields_ = [
        ("N", _int), ("H", _int), ("D", _int), ("chunk", _int),
        ("T_total", _i64),
        ("io", _int), ("out_dtype", _int),
        ("cu_seqlens", _vp), ("cu_seqlens_host", _vp),
        ("q", _vp), ("k", _vp), ("v", _vp),
        ("qkv_row_stride", _i64),
        ("conv_w", _vp), ("conv_state_in", _vp), ("conv_state_out", _vp),
        ("g", _vp), ("beta", _vp), ("gate", _vp), ("rms_w", _vp),
        ("eps_l2", _f), ("eps_rms", _f), ("scale", _f),
        ("initial_state", _vp), ("final_state", _vp), ("out", _vp),
        ("workspace", _vp), ("workspace_bytes", ctypes.c_size_t),
        ("d_status", _vp), ("flags", _int), ("segments", _int),
    ]


class DecodeArgs(ctypes.Structure):
    """Mirror of kda_decode_args."""
    _fields_ = [
        ("N", _int), ("H", _int), ("D", _int),
        ("io", _int), ("out_dtype", _int),
        ("q", _vp), ("k", _vp), ("v", _vp),
        ("qkv_row_stride", _i64),
        ("gate", _vp), ("g", _vp), ("beta", _vp), ("conv_w", _vp), ("rms_w", _vp),
        ("eps_l2", _f), ("eps_rms", _f), ("scale", _f),
        ("state", _vp), ("conv_state", _vp), ("out", _vp), ("d_status", _vp),
    ]


class GemmArgs(ctypes.Structure):
    """Mirror of kda_gemm_args."""
    _fields_ = [
        ("M", _int), ("N", _int), ("K", _int),
        ("A", _vp), ("lda", _i64), ("W", _vp), ("ldw", _i64), ("C", _vp), ("ldc", _i64),
        ("c_dtype", _int), ("epilogue", _int), ("d_status", _vp),
    ]


class BackwardArgs(ctypes.Structure):
    """Mirror of kda_backward_args."""
    _fields_ = [
        ("fwd", PrefillArgs), ("dy", _vp), ("d_final_state", _vp),
        ("dq", _vp), ("dk", _vp), ("dv", _vp), ("dconv_w", _vp), ("dg", _vp), ("dbeta", _vp),
        ("dgate", _vp), ("drms_w", _vp), ("dinitial_state", _vp), ("dconv_state_in", _vp),
    ]


def lib_path() -> str:
    return _build.SO


def load(auto_build: bool = True) -> ctypes.CDLL:
    """Loads libkda.so (building it first if it is missing or stale and nvcc exists).

    Raises if the library cannot be produced: there is no fallback path.
    """
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = _build.SO
        if auto_build:
            try:
                path = _build.build()
            except RuntimeError:
                if not os.path.exists(path):
                    raise
        if not os.path.exists(path):
            raise RuntimeError(f"libkda.so is not built ({path}); run kimi_delta_attention_16_gb300.build")
        lib = ctypes.CDLL(path)
        lib.kda_status_string.restype = ctypes.c_char_p
        lib.kda_status_string.argtypes = [_int]
        lib.kda_last_error.restype = ctypes.c_char_p
        lib.kda_last_error.argtypes = []
        lib.kda_version.restype = _int
        lib.kda_version.argtypes = []
        if lib.kda_version() < ABI_VERSION:
            raise RuntimeError(f"{path} has ABI version {lib.kda_version()}, this binding needs "
                               f">= {ABI_VERSION}; rebuild it")
        lib.kda_short_conv.restype = _int
        lib.kda_short_conv.argtypes = [_vp, _i64, _vp, _vp, _vp, _int, _i64, _int, _int, _vp, _vp,
                                       _vp, _i64, _int, _f, _int, _vp, _vp]
        lib.kda_prefill_workspace_size.restype = _int
        lib.kda_prefill_workspace_size.argtypes = [ctypes.POINTER(PrefillArgs),
                                                   ctypes.POINTER(ctypes.c_size_t)]
        lib.kda_prefill.restype = _int
        lib.kda_prefill.argtypes = [ctypes.POINTER(PrefillArgs), _vp]
        lib.kda_prefill_plan.restype = _int
        lib.kda_prefill_plan.argtypes = [ctypes.POINTER(PrefillArgs), ctypes.POINTER(_int),
                                         ctypes.POINTER(_int)]
        lib.kda_prefill_noalloc.restype = _int
        lib.kda_prefill_noalloc.argtypes = [ctypes.POINTER(PrefillArgs), _vp]
        lib.kda_decode_step.restype = _int
        lib.kda_decode_step.argtypes = [ctypes.POINTER(DecodeArgs), _vp]
        lib.kda_gemm.restype = _int
        lib.kda_gemm.argtypes = [ctypes.POINTER(GemmArgs), _vp]
        lib.kda_backward_workspace_size.restype = _int
        lib.kda_backward_workspace_size.argtypes = [ctypes.POINTER(BackwardArgs),
                                                    ctypes.POINTER(ctypes.c_size_t)]
        lib.kda_backward.restype = _int
        lib.kda_backward.argtypes = [ctypes.POINTER(BackwardArgs), _vp]
        _lib = lib
        return lib
