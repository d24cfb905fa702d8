"""The host-streaming entry point and the sink-gradient accumulation flag.

``HostPipeline`` runs forward + backward over groups of whole sequences with
the copies of one group overlapped with the kernels of another; every token's
outputs come from the same kernels on the same data as one whole-batch call,
so o, dq, dk and dv must match a whole-batch call bit for bit, and dS_h (a sum
over the groups) to float rounding. Both are also checked against the oracle.
"""

import numpy as np
import pytest
import torch

from attention_learnable_sinks_gb300 import _binding, api
from attention_learnable_sinks_gb300.workloads import make

from parity import assert_close, assert_dsinks, dsink_condition, f64, run_oracle

pytestmark = pytest.mark.gpu


def _device_run(w, dev):
    q, k, v, do = (t.to(dev) for t in (w.q, w.k, w.v, w.dout))
    s, cu = w.sinks.to(dev), w.cu_seqlens.to(dev)
    o, lse = api.forward(q, k, v, s, cu, w.max_seqlen, causal=w.causal, window=w.window)
    dq, dk, dv, ds = api.backward(q, k, v, s, cu, w.max_seqlen, o, lse, do, causal=w.causal,
                                  window=w.window)
    return {n: t.cpu() for n, t in (("o", o), ("dq", dq), ("dk", dk), ("dv", dv), ("dsinks", ds))}


@pytest.mark.parametrize("groups", [1, 2, 3])
def test_host_pipeline_matches_whole_batch(cuda_lib, groups):
    w = make("pipeline", [300, 77, 0, 129, 1, 640, 256], 8, 2, seed=31)
    dev = torch.device("cuda")
    ref = _device_run(w, dev)
    pipe = api.HostPipeline(w.cu_seqlens, w.Hq, w.Hkv, causal=w.causal, window=w.window,
                            groups=groups)
    hin = [t.pin_memory() for t in (w.q, w.k, w.v, w.dout, w.sinks)]
    hout = [torch.empty_like(t).pin_memory() for t in (w.q, w.q, w.k, w.k, w.sinks)]
    for _ in range(2):  # the buffers are reused from one run to the next
        pipe.run(*hin, *hout)
        torch.cuda.synchronize()
    assert _binding.device_error() == 0
    for name, got in zip(("o", "dq", "dk", "dv"), hout[:4]):
        assert torch.equal(got, ref[name]), name
    np.testing.assert_allclose(hout[4].numpy(), ref["dsinks"].numpy(), rtol=1e-5, atol=1e-7)
    oracle, *_ = run_oracle(w)
    for name, got in zip(("o", "dq", "dk", "dv"), hout[:4]):
        assert_close(name, f64(got), oracle[name])
    cond = dsink_condition(w.sinks.numpy().astype(np.float64), oracle["lse"], oracle["o"],
                           oracle["_do"])
    assert_dsinks(hout[4].numpy().astype(np.float64), oracle["dsinks"], cond)


def test_accumulate_dsinks_adds(cuda_lib):
    w = make("accum", [200, 90], 8, 2, seed=32)
    dev = torch.device("cuda")
    q, k, v, do = (t.to(dev) for t in (w.q, w.k, w.v, w.dout))
    s, cu = w.sinks.to(dev), w.cu_seqlens.to(dev)
    o, lse = api.forward(q, k, v, s, cu, w.max_seqlen)
    _, _, _, ds1 = api.backward(q, k, v, s, cu, w.max_seqlen, o, lse, do)
    acc = torch.full_like(ds1, 0.5)
    api.backward(q, k, v, s, cu, w.max_seqlen, o, lse, do, dsinks=acc, accumulate_dsinks=True)
    api.backward(q, k, v, s, cu, w.max_seqlen, o, lse, do, dsinks=acc, accumulate_dsinks=True)
    torch.cuda.synchronize()
    assert torch.equal(acc, (0.5 + ds1) + ds1)
    with pytest.raises(ValueError):  # nothing to add to
        api.backward(q, k, v, None, cu, w.max_seqlen, o, lse, do, accumulate_dsinks=True)
