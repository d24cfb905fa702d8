"""Deterministic backward (``deterministic=True``): dq comes from a
query-stationary pass that sums each query tile's key tiles in a fixed order.

Oracle parity of this mode runs beside the atomic mode in
``test_gpu_parity.py`` and ``test_gpu_configs.py``. Here:
  * every output is bit-identical over repeated calls, with the workspace and
    the outputs refilled with garbage in between, on two different streams;
  * dk, dv and dS_h are bit-identical to the atomic mode's (the main kernel
    computes them the same way in both), and dq agrees with the atomic dq to
    its bf16 rounding;
  * the autograd op passes the mode through.
"""

import numpy as np
import pytest
import torch

from attention_learnable_sinks_gb300 import _binding, api
from attention_learnable_sinks_gb300.workloads import config, make

from parity import assert_close, f64, run_oracle

pytestmark = pytest.mark.gpu


def _inputs(w):
    dev = "cuda"
    return dict(q=w.q.to(dev), k=w.k.to(dev), v=w.v.to(dev), s=w.sinks.to(dev),
                cu=w.cu_seqlens.to(dev), do=w.dout.to(dev))


def _bwd(w, t, o, lse, deterministic, workspace=None, outs=None):
    dq, dk, dv, ds = api.backward(t["q"], t["k"], t["v"], t["s"], t["cu"], max(w.max_seqlen, 1), o,
                                  lse, t["do"], causal=w.causal, window=w.window, scale=w.scale,
                                  deterministic=deterministic, workspace=workspace,
                                  **(outs or {}))
    return [x.clone() for x in (dq, dk, dv, ds)]


def _garbage(t):
    if t.dtype == torch.uint8:
        t.random_(0, 256)
    else:
        t.view(torch.int16 if t.element_size() == 2 else torch.int32).random_(-1000, 1000)


@pytest.mark.parametrize("name", ["ragged", "window", "dense"])
def test_repeated_calls_are_bit_identical(cuda_lib, name):
    if name == "dense":
        w = config("dense")
    elif name == "window":
        w = make("w", [1000, 129, 4000], 16, 2, seed=31, window=300)
    else:
        w = make("r", [300, 77, 0, 129, 1, 2048], 8, 1, seed=32)
    t = _inputs(w)
    o, lse = api.forward(t["q"], t["k"], t["v"], t["s"], t["cu"], max(w.max_seqlen, 1),
                         causal=w.causal, window=w.window, scale=w.scale)
    nbytes = api.workspace_bytes("bwd", w.cu_seqlens.numel() - 1, w.total, w.Hq, w.Hkv)
    ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    outs = dict(dq=torch.empty_like(t["q"]), dk=torch.empty_like(t["k"]),
                dv=torch.empty_like(t["v"]), dsinks=torch.empty(w.Hq, device="cuda"))
    runs = []
    streams = [torch.cuda.current_stream(), torch.cuda.Stream()]
    for i in range(4):
        torch.manual_seed(1000 + i)  # different, reproducible garbage per call
        for x in [ws, *outs.values()]:
            _garbage(x)
        torch.cuda.synchronize()
        with torch.cuda.stream(streams[i % 2]):
            runs.append(_bwd(w, t, o, lse, True, workspace=ws, outs=outs))
        torch.cuda.synchronize()
        assert _binding.device_error(reset=True) == 0
    for r in runs[1:]:
        for a, b, nm in zip(runs[0], r, ("dq", "dk", "dv", "dsinks")):
            assert torch.equal(a.view(torch.int16) if a.dtype == torch.bfloat16 else a.view(torch.int32),
                               b.view(torch.int16) if b.dtype == torch.bfloat16 else b.view(torch.int32)), \
                f"{name}: {nm} differs between calls"


@pytest.mark.parametrize("name", ["ragged", "dense"])
def test_modes_agree(cuda_lib, name):
    w = config("dense") if name == "dense" else make("m", [300, 77, 0, 129, 1, 2048], 8, 2, seed=33)
    t = _inputs(w)
    o, lse = api.forward(t["q"], t["k"], t["v"], t["s"], t["cu"], max(w.max_seqlen, 1),
                         causal=w.causal, window=w.window, scale=w.scale)
    at = _bwd(w, t, o, lse, False)
    de = _bwd(w, t, o, lse, True)
    torch.cuda.synchronize()
    assert _binding.device_error(reset=True) == 0
    for i, nm in ((1, "dk"), (2, "dv"), (3, "dsinks")):
        assert torch.equal(at[i], de[i]), f"{nm} differs between the two modes"
    # both dq are fp32 sums of the same terms, rounded once to bf16
    assert_close("dq modes", f64(de[0]), f64(at[0]), tol=4e-3)


def test_autograd_deterministic(cuda_lib):
    w = make("ag", [640, 200], 8, 2, seed=34, window=256)
    ref, *_ = run_oracle(w)
    grads = []
    for _ in range(2):
        t = _inputs(w)
        q, k, v, s = (t[n].clone().requires_grad_(True) for n in ("q", "k", "v", "s"))
        out = api.sink_attention(q, k, v, s, t["cu"], w.max_seqlen, causal=True, window=w.window,
                                 scale=w.scale, deterministic=True)
        out.backward(t["do"])
        grads.append([x.grad.clone() for x in (q, k, v, s)])
    for a, b in zip(*grads):
        assert torch.equal(a, b)
    assert_close("dq", f64(grads[0][0]), ref["dq"])
    assert_close("dk", f64(grads[0][1]), ref["dk"])
    assert_close("dv", f64(grads[0][2]), ref["dv"])
    assert np.all(np.isfinite(f64(grads[0][3])))
