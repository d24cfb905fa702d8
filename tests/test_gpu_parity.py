"""CUDA path vs the fp64 oracle on small seeded problems, element by element
over whole tensors: ragged tails, empty and length-1 sequences, several
tiles, GQA group sizes 1/2/8, causal, non-causal and sliding windows, no
sink, strided (packed qkv) inputs, and the degenerate cases the method has.
"""

import numpy as np
import pytest
import torch

from attention_learnable_sinks_gb300 import _binding, api
from attention_learnable_sinks_gb300.workloads import config, make

from parity import (ALL, assert_dsinks, compare_full, dsink_condition, f64, run_cuda,
                    run_oracle)

pytestmark = pytest.mark.gpu

SMALL = [
    # name, lengths, Hq, Hkv, causal, window, extra
    ("one_token", [1], 8, 2, True, 0, {}),
    ("ragged_varlen", [300, 77, 0, 129, 1], 8, 1, True, 0, {}),
    ("noncausal", [513], 4, 4, False, 0, {}),
    ("window128_short_seq", [200, 100, 1000], 8, 2, True, 128, {}),
    ("window1", [700], 2, 1, True, 1, {}),
    ("window_wider_than_tile", [257, 640], 16, 2, True, 300, {}),
    ("group8", [384, 255], 16, 2, True, 0, {"sink_range": (-4.0, 4.0)}),
    ("peaked_logits", [600], 8, 1, True, 0, {"qk_std": 2.0, "sink_range": (-10.0, 10.0)}),
    ("sinks_minus30", [450], 4, 2, True, 0, {"odd_head_sink": -30.0}),
    ("group16", [300, 130], 16, 1, True, 0, {}),
    ("group3", [257, 100], 6, 2, True, 0, {}),
    ("mqa64", [200], 64, 1, True, 0, {}),
    ("mha_window", [390], 4, 4, True, 64, {}),
    ("window127", [520], 4, 1, True, 127, {}),
    ("window129", [520], 4, 1, True, 129, {}),
]


@pytest.mark.parametrize("case", SMALL, ids=[c[0] for c in SMALL])
def test_small_cases_match_oracle(cuda_lib, case):
    name, lengths, Hq, Hkv, causal, window, extra = case
    w = make(name, lengths, Hq, Hkv, seed=100 + len(name), causal=causal, window=window, **extra)
    ref, tok, qh, kvh = run_oracle(w)
    s = w.sinks.numpy().astype(np.float64)
    cond = dsink_condition(s, ref["lse"], ref["o"], ref["_do"])
    for det in (False, True):  # atomic dq, then the fixed-order dq pass
        got = run_cuda(w, deterministic=det)
        compare_full(w, got, ref)
        assert_dsinks(got["dsinks"], ref["dsinks"], cond)


def test_tiny_config_matches_oracle(cuda_lib):
    w = config("tiny")
    ref, *_ = run_oracle(w)
    cond = dsink_condition(w.sinks.numpy().astype(np.float64), ref["lse"], ref["o"], ref["_do"])
    for det in (False, True):
        got = run_cuda(w, deterministic=det)
        compare_full(w, got, ref)
        assert_dsinks(got["dsinks"], ref["dsinks"], cond)


def test_no_sink_matches_oracle(cuda_lib):
    w = make("nosink", [333, 90], 8, 2, seed=7)
    ref, *_ = run_oracle(w, sinks=False)
    for det in (False, True):
        got = run_cuda(w, sinks=False, deterministic=det)
        compare_full(w, got, ref)
        assert np.all(got["dsinks"] == 0)


def test_custom_scale(cuda_lib):
    w = make("scale", [260], 4, 1, seed=8)
    got = run_cuda(w, scale=0.3)
    ref, *_ = run_oracle(w, scale=0.3)
    compare_full(w, got, ref)


def test_strided_qkv_views(cuda_lib):
    # q, k, v as views into one packed [total, Hq + 2 Hkv, 64] buffer
    w = make("packed", [290, 130], 8, 2, seed=9)
    qkv = torch.cat([w.q, w.k, w.v], 1).cuda()
    q, k, v = qkv[:, :8], qkv[:, 8:10], qkv[:, 10:12]
    assert q.stride(0) == 12 * 64
    got = run_cuda(w, q_view=q, k_view=k, v_view=v)
    ref, *_ = run_oracle(w)
    compare_full(w, got, ref)


def test_autograd_op_matches_oracle(cuda_lib):
    w = make("autograd", [160, 96], 4, 2, seed=10)
    q = w.q.cuda().requires_grad_()
    k = w.k.cuda().requires_grad_()
    v = w.v.cuda().requires_grad_()
    s = w.sinks.cuda().requires_grad_()
    o = api.sink_attention(q, k, v, s, w.cu_seqlens.cuda(), w.max_seqlen)
    o.backward(w.dout.cuda())
    ref, *_ = run_oracle(w)
    got = {"o": o, "dq": q.grad, "dk": k.grad, "dv": v.grad}
    from parity import assert_close, f64
    for n in ("o", "dq", "dk", "dv"):
        assert_close(n, f64(got[n]), ref[n])
    cond = dsink_condition(w.sinks.numpy().astype(np.float64), ref["lse"], ref["o"], ref["_do"])
    assert_dsinks(f64(s.grad), ref["dsinks"], cond)


def test_module_with_sink_parameter_matches_oracle(cuda_lib):
    """SinkAttention holds the sinks as a parameter; its gradient after one
    backward is dL/dS_h, and an optimizer step moves it."""
    w = make("module", [300, 77], 8, 2, seed=12, window=100)
    layer = api.SinkAttention(8, window=100, device="cuda")
    with torch.no_grad():
        layer.sinks.copy_(w.sinks)
    q = w.q.cuda().requires_grad_()
    k = w.k.cuda().requires_grad_()
    v = w.v.cuda().requires_grad_()
    o = layer(q, k, v, w.cu_seqlens.cuda(), w.max_seqlen)
    o.backward(w.dout.cuda())
    ref, *_ = run_oracle(w)
    from parity import assert_close, f64
    for n, t in (("o", o), ("dq", q.grad), ("dk", k.grad), ("dv", v.grad)):
        assert_close(n, f64(t), ref[n])
    cond = dsink_condition(w.sinks.numpy().astype(np.float64), ref["lse"], ref["o"], ref["_do"])
    assert_dsinks(f64(layer.sinks.grad), ref["dsinks"], cond)
    before = layer.sinks.detach().clone()
    torch.optim.SGD(layer.parameters(), lr=0.1).step()
    assert torch.allclose(layer.sinks.detach(), before - 0.1 * layer.sinks.grad)


def test_batched_4d_layout(cuda_lib):
    w = make("batched", [200, 200], 4, 2, seed=11)
    q = w.q.cuda().view(2, 200, 4, 64)
    k = w.k.cuda().view(2, 200, 2, 64)
    v = w.v.cuda().view(2, 200, 2, 64)
    o = api.sink_attention(q, k, v, w.sinks.cuda())
    ref, *_ = run_oracle(w, want=("o",))
    from parity import assert_close, f64
    assert_close("o", f64(o.reshape(400, 4, 64)), ref["o"])


def test_empty_batch(cuda_lib):
    w = make("empty", [0, 0], 4, 2, seed=12)
    dev = "cuda"
    cu = w.cu_seqlens.to(dev)
    q = torch.zeros(0, 4, 64, dtype=torch.bfloat16, device=dev)
    k = torch.zeros(0, 2, 64, dtype=torch.bfloat16, device=dev)
    s = w.sinks.to(dev)
    o, lse = api.forward(q, k, k, s, cu, 0)
    ds = torch.full((4,), 7.0, device=dev)
    dq, dk, dv, ds = api.backward(q, k, k, s, cu, 0, o, lse, q, dsinks=ds)
    torch.cuda.synchronize()
    assert o.shape == (0, 4, 64) and torch.all(ds == 0)
    assert _binding.device_error() == 0


def test_malformed_cu_seqlens_sets_device_error(cuda_lib):
    # non-monotone offsets: the kernels skip all work and record the error
    w = make("bad", [64, 64], 4, 2, seed=13)
    dev = "cuda"
    bad = torch.tensor([0, 200, 128], dtype=torch.int32)  # lengths 200 and -72
    q, k, v = w.q.to(dev), w.k.to(dev), w.v.to(dev)
    o = torch.full_like(q, 3.0)
    api.forward(q, k, v, w.sinks.to(dev), bad.to(dev), 128, out=o)
    assert _binding.device_error(reset=True) == 1
    assert torch.all(o == 3.0)  # untouched
    # a length above max_seqlen is rejected the same way
    api.forward(q, k, v, w.sinks.to(dev), w.cu_seqlens.to(dev), 32, out=o)
    assert _binding.device_error(reset=True) == 1
    assert _binding.device_error() == 0


def test_rejects_bad_arguments_before_launch(cuda_lib):
    w = make("args", [64], 4, 2, seed=14)
    dev = "cuda"
    q, k, v, cu = w.q.to(dev), w.k.to(dev), w.v.to(dev), w.cu_seqlens.to(dev)
    n0 = _binding.launch_count()
    with pytest.raises(_binding.SinkAttnError) as e:
        api.forward(q, k, v, None, cu, 64, causal=False, window=8)
    assert e.value.status == 2
    assert _binding.launch_count() == n0


@pytest.mark.parametrize("case", [("dense_like", [1024, 1024], 16, 2, 0), ("ragged", [300, 77, 0, 129, 1], 8, 1, 0),
                                  ("window", [700, 129], 8, 2, 128)], ids=lambda c: c[0])
def test_forward_clears_backward_workspace(cuda_lib, case):
    """The forward, given the backward's workspace, clears the dq accumulator
    in it, and the backward told so skips its own clear. The workspace starts
    full of garbage, so a byte the forward missed would show in dq."""
    name, lengths, Hq, Hkv, window = case
    w = make(name, lengths, Hq, Hkv, seed=61, window=window)
    dev = "cuda"
    q, k, v, do = (t.to(dev) for t in (w.q, w.k, w.v, w.dout))
    s, cu = w.sinks.to(dev), w.cu_seqlens.to(dev)
    ws_b = torch.empty(api.workspace_bytes("bwd", w.nseq, w.total, Hq, Hkv), dtype=torch.uint8,
                       device=dev)
    ref, *_ = run_oracle(w)
    for fill in (0x7F, 0xA5):
        ws_b.fill_(fill)
        o, lse = api.forward(q, k, v, s, cu, w.max_seqlen, window=window, bwd_workspace=ws_b)
        dq, dk, dv, ds = api.backward(q, k, v, s, cu, w.max_seqlen, o, lse, do, window=window,
                                      workspace=ws_b, workspace_cleared=True)
        torch.cuda.synchronize()
        assert _binding.device_error(reset=True) == 0
        got = {"o": f64(o), "lse": f64(lse), "dq": f64(dq), "dk": f64(dk), "dv": f64(dv)}
        compare_full(w, got, ref)
        cond = dsink_condition(w.sinks.numpy().astype(np.float64), ref["lse"], ref["o"], ref["_do"])
        assert_dsinks(f64(ds), ref["dsinks"], cond)
