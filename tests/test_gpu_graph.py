"""The forward + backward captured into a CUDA graph and replayed.

The library never synchronises and allocates nothing, and the tensor maps
are encoded on the host before the launches, so a training step built from
its calls can be captured once and replayed (CUDA graphs instead of a
tracing compiler). The replay must give the eager step's results bit for
bit (deterministic backward), including after the inputs are rewritten in
place, and with the forward preparing the backward's workspace.
"""

import pytest
import torch

from attention_learnable_sinks_gb300 import _binding, api
from attention_learnable_sinks_gb300.workloads import make

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("d", [64, 128])
def test_graph_replay_equals_eager(cuda_lib, d):
    w = make(f"graph_d{d}", [700, 129, 1, 1500], 16, 2, seed=71, d=d)
    w2 = make(f"graph2_d{d}", [700, 129, 1, 1500], 16, 2, seed=72, d=d)
    dev = torch.device("cuda")
    q, k, v, do = (t.to(dev) for t in (w.q, w.k, w.v, w.dout))
    s, cu = w.sinks.to(dev), w.cu_seqlens.to(dev)
    o = torch.empty_like(q)
    lse = torch.empty(w.Hq, w.total, dtype=torch.float32, device=dev)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ds = torch.empty_like(s)
    ws_f = torch.empty(api.workspace_bytes("fwd", w.nseq, w.total, w.Hq, w.Hkv, head_dim=d),
                       dtype=torch.uint8, device=dev)
    ws_b = torch.empty(api.workspace_bytes("bwd", w.nseq, w.total, w.Hq, w.Hkv, head_dim=d),
                       dtype=torch.uint8, device=dev)

    def step():
        api.forward(q, k, v, s, cu, w.max_seqlen, out=o, lse=lse, workspace=ws_f, bwd_workspace=ws_b)
        api.backward(q, k, v, s, cu, w.max_seqlen, o, lse, do, dq=dq, dk=dk, dv=dv, dsinks=ds,
                     workspace=ws_b, deterministic=True)

    def outputs():
        return [t.clone() for t in (o, lse, dq, dk, dv, ds)]

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step()  # warm-up off the capture (first-call device setup)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    eager = outputs()

    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    for t in (o, lse, dq, dk, dv, ds):
        t.fill_(float("nan"))
    g.replay()
    torch.cuda.synchronize()
    assert _binding.device_error(reset=True) == 0
    for a, b in zip(outputs(), eager):
        assert torch.equal(a, b)

    # new inputs written into the captured buffers: the replay follows them
    for dst, src in ((q, w2.q), (k, w2.k), (v, w2.v), (do, w2.dout), (s, w2.sinks)):
        dst.copy_(src)
    step()
    torch.cuda.synchronize()
    eager2 = outputs()
    g.replay()
    torch.cuda.synchronize()
    assert _binding.device_error(reset=True) == 0
    for a, b in zip(outputs(), eager2):
        assert torch.equal(a, b)
    assert not torch.equal(eager2[0], eager[0])
