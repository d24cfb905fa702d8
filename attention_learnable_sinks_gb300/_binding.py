"""ctypes binding of libsinkattn.so (C ABI in include/sinkattn.h).

Argument marshalling only: torch tensors are turned into device pointers,
sizes and strides, and every step of the computation runs in the library's
CUDA kernels. There is no fallback: if the library is missing or cannot be
loaded, every entry point raises.
"""

from __future__ import annotations

import ctypes
import os
import threading

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libsinkattn.so")

_c_void_p = ctypes.c_void_p


class FwdParams(ctypes.Structure):
    _fields_ = [
        ("q", _c_void_p), ("k", _c_void_p), ("v", _c_void_p),
        ("sinks", _c_void_p), ("cu_seqlens", _c_void_p),
        ("o", _c_void_p), ("lse", _c_void_p),
        ("workspace", _c_void_p), ("workspace_bytes", ctypes.c_size_t),
        ("timing_events", _c_void_p * 2),
        ("q_row_stride", ctypes.c_int64), ("k_row_stride", ctypes.c_int64),
        ("v_row_stride", ctypes.c_int64),
        ("nseq", ctypes.c_int32), ("total", ctypes.c_int32), ("max_seqlen", ctypes.c_int32),
        ("Hq", ctypes.c_int32), ("Hkv", ctypes.c_int32), ("head_dim", ctypes.c_int32),
        ("causal", ctypes.c_int32), ("window", ctypes.c_int32),
        ("softmax_scale", ctypes.c_float),
        ("bwd_workspace", _c_void_p), ("bwd_workspace_bytes", ctypes.c_size_t),
    ]


class BwdParams(ctypes.Structure):
    _fields_ = [
        ("fwd", FwdParams),
        ("dout", _c_void_p), ("dq", _c_void_p), ("dk", _c_void_p), ("dv", _c_void_p),
        ("dsinks", _c_void_p),
        ("workspace", _c_void_p), ("workspace_bytes", ctypes.c_size_t),
        ("timing_events", _c_void_p * 2),
        ("accumulate_dsinks", ctypes.c_int32),
        ("deterministic", ctypes.c_int32),
        ("timing_events_dq", _c_void_p * 2),
        ("workspace_cleared", ctypes.c_int32),
    ]


class DecodeParams(ctypes.Structure):
    _fields_ = [
        ("q", _c_void_p), ("k_cache", _c_void_p), ("v_cache", _c_void_p),
        ("block_table", _c_void_p), ("seqlens", _c_void_p), ("sinks", _c_void_p),
        ("o", _c_void_p), ("lse", _c_void_p),
        ("workspace", _c_void_p), ("workspace_bytes", ctypes.c_size_t),
        ("nseq", ctypes.c_int32), ("num_blocks", ctypes.c_int32), ("block_size", ctypes.c_int32),
        ("max_blocks_per_seq", ctypes.c_int32), ("Hq", ctypes.c_int32), ("Hkv", ctypes.c_int32),
        ("head_dim", ctypes.c_int32), ("window", ctypes.c_int32), ("num_splits", ctypes.c_int32),
        ("softmax_scale", ctypes.c_float),
    ]


# Every symbol include/sinkattn.h declares: (name, restype, argtypes).
SYMBOLS = [
    ("sinkattn_fwd_workspace_size", ctypes.c_size_t, [ctypes.c_int32] * 5),
    ("sinkattn_bwd_workspace_size", ctypes.c_size_t, [ctypes.c_int32] * 5),
    ("sinkattn_bwd_workspace_size_mode", ctypes.c_size_t, [ctypes.c_int32] * 6),
    ("sinkattn_fwd", ctypes.c_int, [ctypes.POINTER(FwdParams), _c_void_p]),
    ("sinkattn_bwd", ctypes.c_int, [ctypes.POINTER(BwdParams), _c_void_p]),
    ("sinkattn_bwd_static_workspace", ctypes.c_int, [ctypes.POINTER(BwdParams), _c_void_p]),
    ("sinkattn_decode_workspace_size", ctypes.c_size_t, [ctypes.c_int32] * 3),
    ("sinkattn_decode", ctypes.c_int, [ctypes.POINTER(DecodeParams), _c_void_p]),
    ("sinkattn_decode_exact", ctypes.c_int, [ctypes.POINTER(DecodeParams), _c_void_p]),
    ("sinkattn_status_string", ctypes.c_char_p, [ctypes.c_int32]),
    ("sinkattn_last_error_message", ctypes.c_char_p, []),
    ("sinkattn_device_error", ctypes.c_int32, [ctypes.c_int32]),
    ("sinkattn_launch_count", ctypes.c_uint64, []),
    ("sinkattn_decode_workspace_size_d", ctypes.c_size_t,
     [ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32]),
    ("sinkattn_params_size", ctypes.c_size_t, [ctypes.c_int32]),
    ("sinkattn_set_wait_limit_ns", None, [ctypes.c_uint64]),
    ("sinkattn_test_withhold_copies", None, [ctypes.c_int32]),
]

STATUS = {0: "SINKATTN_OK", 1: "SINKATTN_ERR_INVALID_ARG", 2: "SINKATTN_ERR_UNSUPPORTED",
          3: "SINKATTN_ERR_CUDA", 4: "SINKATTN_ERR_WORKSPACE", 5: "SINKATTN_ERR_TIMEOUT"}

_lib = None
_lock = threading.Lock()


class SinkAttnError(RuntimeError):
    def __init__(self, status: int, where: str, detail: str):
        self.status = status
        super().__init__(f"{where}: {STATUS.get(status, status)}: {detail}")


def lib():
    """Load libsinkattn.so (building it first if the toolkit is present)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            from . import build as _build
            try:
                _build.build()
            except Exception as e:  # no toolkit, compile error: fail loudly
                raise RuntimeError(f"libsinkattn.so is missing and could not be built: {e}") from e
        L = ctypes.CDLL(LIB_PATH)
        for name, res, args in SYMBOLS:
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        if L.sinkattn_params_size(0) != ctypes.sizeof(FwdParams) or \
                L.sinkattn_params_size(1) != ctypes.sizeof(BwdParams) or \
                L.sinkattn_params_size(2) != ctypes.sizeof(DecodeParams):
            raise RuntimeError("libsinkattn.so parameter structs do not match this binding")
        _lib = L
    return _lib


def check(status: int, where: str):
    if status != 0:
        detail = lib().sinkattn_last_error_message().decode()
        raise SinkAttnError(status, where, detail)


def device_error(reset: bool = True) -> int:
    """Synchronise and read (then clear) the library's device error word."""
    return int(lib().sinkattn_device_error(1 if reset else 0))


def launch_count() -> int:
    return int(lib().sinkattn_launch_count())
