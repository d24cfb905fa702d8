"""The backward entry point that allocates nothing.

sinkattn_bwd_static_workspace serves callers that cannot allocate device
memory when they call the library: a host that has already handed the whole
device to its own memory pool, or code running where an allocation's implicit
synchronisation is not allowed. It uses a fixed array inside the library in
place of a caller-provided workspace. Here it is called through the C ABI and
must match the regular entry point, which takes a caller workspace, in both
backward modes, on calls in a row. The first call is a different, larger
problem, so the array holds another packing's tile lists, D, sink partials
and dq accumulator when the compared calls start: nothing in it may need to
start at zero.
"""

import ctypes

import pytest
import torch

from attention_learnable_sinks_gb300 import _binding, api
from attention_learnable_sinks_gb300._binding import BwdParams
from attention_learnable_sinks_gb300.workloads import make

from parity import assert_close, f64, rel_l2

pytestmark = pytest.mark.gpu

STATIC_BYTES = 64 << 20


class _Problem:
    def __init__(self, w):
        dev = torch.device("cuda")
        self.w = w
        self.q, self.k, self.v, self.do = (t.to(dev) for t in (w.q, w.k, w.v, w.dout))
        self.s, self.cu = w.sinks.to(dev), w.cu_seqlens.to(dev)
        self.o, self.lse = api.forward(self.q, self.k, self.v, self.s, self.cu, w.max_seqlen,
                                       causal=w.causal, window=w.window, scale=w.scale)

    def regular(self, deterministic):
        w = self.w
        return api.backward(self.q, self.k, self.v, self.s, self.cu, w.max_seqlen, self.o, self.lse,
                            self.do, causal=w.causal, window=w.window, scale=w.scale,
                            deterministic=deterministic)

    def static(self, deterministic):
        w = self.w
        dq, dk, dv = (torch.full_like(t, 9.0) for t in (self.q, self.k, self.v))
        ds = torch.full_like(self.s, 9.0)
        p = BwdParams()
        api._fill_fwd(p.fwd, self.q, self.k, self.v, self.s, self.cu, w.max_seqlen, w.causal,
                      w.window, w.scale, self.o, self.lse)
        p.dout, p.dq, p.dk, p.dv, p.dsinks = (t.data_ptr() for t in (self.do, dq, dk, dv, ds))
        p.deterministic = 1 if deterministic else 0
        lib = _binding.lib()
        _binding.check(lib.sinkattn_bwd_static_workspace(ctypes.byref(p),
                                                         torch.cuda.current_stream().cuda_stream),
                       "sinkattn_bwd_static_workspace")
        torch.cuda.synchronize()
        assert _binding.device_error() == 0
        return dq, dk, dv, ds


def _check(got, ref):
    for name, g, r in zip(("dq", "dk", "dv"), got[:3], ref[:3]):
        assert_close(name, f64(g), f64(r))
    assert rel_l2(f64(got[3]), f64(ref[3])) <= 1e-2


def test_static_workspace_backward_matches_regular_entry_point(cuda_lib):
    # a larger packing first: its contents stay in the array
    big = _Problem(make("noalloc_big", [2000, 1500, 3, 900, 130], 8, 2, seed=22, window=0))
    assert api.workspace_bytes("bwd", big.w.nseq, big.w.total, 8, 2) <= STATIC_BYTES
    _check(big.static(False), big.regular(False))
    small = _Problem(make("noalloc", [700, 333, 1, 129], 8, 2, seed=21, window=0))
    for det in (False, True, False, True):
        _check(small.static(det), small.regular(det))


def test_static_workspace_deterministic_fits_larger_problems(cuda_lib):
    # four 2048-token sequences of 64 query heads: the atomic mode's fp32 dq
    # accumulator alone is 128 MiB, the deterministic mode needs a few MiB
    w = make("noalloc_dense", [2048] * 4, 64, 8, seed=23)
    need_det = api.workspace_bytes("bwd", w.nseq, w.total, w.Hq, w.Hkv, deterministic=True)
    need_atomic = api.workspace_bytes("bwd", w.nseq, w.total, w.Hq, w.Hkv)
    assert need_det <= STATIC_BYTES < need_atomic
    prob = _Problem(w)
    _check(prob.static(True), prob.regular(True))


def test_static_workspace_head_dim128_in_either_mode(cuda_lib):
    # head_dim 128 always takes the deterministic backward, so the dense
    # shape fits whichever mode is asked for, and both give the same bits
    w = make("noalloc_d128", [2048] * 4, 64, 8, seed=24, d=128)
    need = api.workspace_bytes("bwd", w.nseq, w.total, w.Hq, w.Hkv, head_dim=128)
    assert need == api.workspace_bytes("bwd", w.nseq, w.total, w.Hq, w.Hkv, deterministic=True,
                                       head_dim=128)
    assert need <= STATIC_BYTES
    prob = _Problem(w)
    ref = prob.regular(False)
    for det in (False, True):
        got = prob.static(det)
        for g, r in zip(got, ref):
            assert torch.equal(g, r)


def test_static_workspace_rejects_problems_above_its_size(cuda_lib):
    lib = _binding.lib()
    p = BwdParams()
    p.fwd.nseq, p.fwd.total, p.fwd.max_seqlen = 4, 8192, 2048
    p.fwd.Hq, p.fwd.Hkv, p.fwd.head_dim, p.fwd.causal = 64, 8, 64, 1
    n0 = lib.sinkattn_launch_count()
    assert lib.sinkattn_bwd_static_workspace(ctypes.byref(p), None) == 4
    assert b"static workspace" in lib.sinkattn_last_error_message()
    assert lib.sinkattn_launch_count() == n0
