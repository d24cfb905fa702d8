"""The backward entry point that allocates nothing.

sinkattn_bwd_static_workspace serves callers that cannot allocate device
memory when they call the library: a host that has already handed the whole
device to its own memory pool, or code running where an allocation's implicit
synchronisation is not allowed. It uses a fixed array inside the library in
place of a caller-provided workspace. Here it is called through the C ABI and
must match the regular entry point, which takes a caller workspace, on two
calls in a row.
"""

import ctypes

import numpy as np
import pytest
import torch

from attention_learnable_sinks_gb300 import _binding, api
from attention_learnable_sinks_gb300._binding import BwdParams
from attention_learnable_sinks_gb300.workloads import make

from parity import assert_close, f64, rel_l2

pytestmark = pytest.mark.gpu

STATIC_BYTES = 64 << 20


def _params(w, dev, q, k, v, s, cu, o, lse, do, dq, dk, dv, ds):
    p = BwdParams()
    api._fill_fwd(p.fwd, q, k, v, s, cu, w.max_seqlen, w.causal, w.window, w.scale, o, lse)
    p.dout, p.dq, p.dk, p.dv, p.dsinks = (t.data_ptr() for t in (do, dq, dk, dv, ds))
    return p


def test_static_workspace_backward_matches_regular_entry_point(cuda_lib):
    w = make("noalloc", [700, 333, 1, 129], 8, 2, seed=21, window=0)
    dev = torch.device("cuda")
    q, k, v, do = (t.to(dev) for t in (w.q, w.k, w.v, w.dout))
    s, cu = w.sinks.to(dev), w.cu_seqlens.to(dev)
    assert api.workspace_bytes("bwd", w.nseq, w.total, w.Hq, w.Hkv) <= STATIC_BYTES
    o, lse = api.forward(q, k, v, s, cu, w.max_seqlen, scale=w.scale)
    ref = api.backward(q, k, v, s, cu, w.max_seqlen, o, lse, do, scale=w.scale)
    torch.cuda.synchronize()
    lib = _binding.lib()
    stream = torch.cuda.current_stream().cuda_stream
    for _ in range(2):
        dq, dk, dv = torch.full_like(q, 9.0), torch.full_like(k, 9.0), torch.full_like(v, 9.0)
        ds = torch.full_like(s, 9.0)
        p = _params(w, dev, q, k, v, s, cu, o, lse, do, dq, dk, dv, ds)
        _binding.check(lib.sinkattn_bwd_static_workspace(ctypes.byref(p), stream),
                       "sinkattn_bwd_static_workspace")
        torch.cuda.synchronize()
        assert _binding.device_error() == 0
        for name, got, want in (("dq", dq, ref[0]), ("dk", dk, ref[1]), ("dv", dv, ref[2])):
            assert_close(name, f64(got), f64(want))
        assert rel_l2(f64(ds), f64(ref[3])) <= 1e-2


def test_static_workspace_rejects_problems_above_its_size(cuda_lib):
    lib = _binding.lib()
    p = BwdParams()
    p.fwd.nseq, p.fwd.total, p.fwd.max_seqlen = 4, 8192, 2048
    p.fwd.Hq, p.fwd.Hkv, p.fwd.head_dim, p.fwd.causal = 64, 8, 64, 1
    n0 = lib.sinkattn_launch_count()
    assert lib.sinkattn_bwd_static_workspace(ctypes.byref(p), None) == 4
    assert b"static workspace" in lib.sinkattn_last_error_message()
    assert lib.sinkattn_launch_count() == n0
