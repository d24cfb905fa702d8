"""fp64 CPU oracle for attention with learnable per-head sinks.

TEST INFRASTRUCTURE ONLY: the test suite, the smoke check and the benchmark's
CPU-baseline leg are the only callers. The CUDA library never imports, links
or calls anything here, and nothing here imports the CUDA package.

What is computed, and from which passage (page "GPT-OSS Agentic RL Training: A
Practical Retrospective"):
  * "The Role of Attention Sinks": one learnable scalar S_h per head acts as a
    virtual token inside the softmax. Read plainly: exp(S_h) joins the softmax
    denominator, and the virtual token has no value vector.
  * "Implementation in FlashAttention v3", steps 1-2: the forward with sinks,
    and a backward that also returns dL/dS_h.
The formulas are written out in ``sinkattn_oracle.cpp``; that file is the
plain definition, row by row, in fp64.

Pins (all in ``tests/test_oracle.py``): torch's scaled-dot-product attention
with the sink appended as a real extra key of zero value (forward and autograd
backward), sinks at -inf against textbook attention, central finite
differences of the oracle's own forward, closed forms (one key, window of one),
probability mass summing to one, shift invariance, GQA repetition and varlen
concatenation.
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "sinkattn_oracle.cpp")
_LIB_PATH = os.path.join(_HERE, "_build", "liboracle_sinkattn.so")
_lib = None
_lock = threading.Lock()

_dp = ctypes.POINTER(ctypes.c_double)
_ip = ctypes.POINTER(ctypes.c_int32)


def build(force: bool = False) -> str:
    """Compile the C++ oracle into a shared object (plain g++, -O2, IEEE)."""
    os.makedirs(os.path.dirname(_LIB_PATH), exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    subprocess.check_call(["g++", "-O2", "-std=c++17", "-shared", "-fPIC", "-pthread",
                           _SRC, "-o", tmp])
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            fn = lib.oracle_sinkattn
            fn.restype = ctypes.c_int
            fn.argtypes = [_dp, _dp, _dp, _dp, _dp, _ip, ctypes.c_int32, ctypes.c_int32,
                           ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                           ctypes.c_double, ctypes.c_int32, _dp, _dp, _dp, _dp, _dp, _dp,
                           ctypes.c_int32]
            _lib = lib
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(_dp)


def default_threads() -> int:
    return os.cpu_count() or 1


def sinkattn(q, k, v, sinks, cu_seqlens, *, causal=True, window=0, scale=None,
             dout=None, want=("o", "lse"), nthreads=None, first_row=0):
    """Evaluate the definition on host arrays.

    q [total, Hq, d], k/v [total, Hkv, d], dout [total, Hq, d] (any float type,
    converted to fp64 exactly: bf16 and fp32 values are representable);
    sinks [Hq] or None (no sink); cu_seqlens int [nseq+1].
    ``want`` picks outputs among o, lse, dq, dk, dv, dsinks. Returns a dict of
    fp64 arrays: o [total,Hq,d], lse [Hq,total], dq, dk, dv, dsinks [Hq].
    ``first_row`` > 0 (causal only) computes only local rows and keys >=
    first_row of each sequence; entries elsewhere stay zero.
    """
    lib = _load()
    q = np.ascontiguousarray(q, dtype=np.float64)
    k = np.ascontiguousarray(k, dtype=np.float64)
    v = np.ascontiguousarray(v, dtype=np.float64)
    cu = np.ascontiguousarray(cu_seqlens, dtype=np.int32)
    total, Hq, d = q.shape
    Hkv = k.shape[1]
    nseq = cu.shape[0] - 1
    if int(cu[-1]) != total or k.shape != (total, Hkv, d) or v.shape != k.shape:
        raise ValueError("inconsistent shapes for the oracle")
    s = None if sinks is None else np.ascontiguousarray(sinks, dtype=np.float64)
    g = None if dout is None else np.ascontiguousarray(dout, dtype=np.float64)
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    out = {}
    shapes = {"o": (total, Hq, d), "lse": (Hq, total), "dq": (total, Hq, d),
              "dk": (total, Hkv, d), "dv": (total, Hkv, d), "dsinks": (Hq,)}
    for name in want:
        out[name] = np.zeros(shapes[name], dtype=np.float64)
    rc = lib.oracle_sinkattn(_ptr(q), _ptr(k), _ptr(v), _ptr(s), _ptr(g),
                             cu.ctypes.data_as(_ip), nseq, Hq, Hkv, d, int(bool(causal)),
                             int(window), float(scale), int(first_row),
                             _ptr(out.get("o")), _ptr(out.get("lse")), _ptr(out.get("dq")),
                             _ptr(out.get("dk")), _ptr(out.get("dv")), _ptr(out.get("dsinks")),
                             int(nthreads or default_threads()))
    if rc != 0:
        raise ValueError("oracle rejected its arguments")
    return out
