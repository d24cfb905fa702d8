"""head_dim 128 against the fp64 oracle, element by element over whole
tensors (page 4 of the sources, the xxqk.cn training log, runs its sink
attention at head_dim 128). The forward is the head_dim 64 kernel's
algorithm on 128-feature tiles; the backward takes dK / dV from a
key-stationary kernel over 64-row query blocks and dq from the fixed-order
query-stationary pass, so both backward modes give the same, run-to-run
identical result. Same tolerances and guard regions as the head_dim 64
parity tests."""

import numpy as np
import pytest
import torch

from attention_learnable_sinks_gb300 import _binding, api
from attention_learnable_sinks_gb300.workloads import make

from parity import assert_dsinks, compare_full, dsink_condition, run_cuda, run_oracle

pytestmark = pytest.mark.gpu

D = 128

CASES = [
    # name, lengths, Hq, Hkv, causal, window, extra
    ("one_token", [1], 8, 2, True, 0, {}),
    ("ragged_varlen", [300, 77, 0, 129, 1], 8, 1, True, 0, {}),
    ("noncausal", [513], 4, 4, False, 0, {}),
    ("noncausal_ragged", [200, 64, 131], 8, 2, False, 0, {}),
    ("window128_short_seq", [200, 100, 1000], 8, 2, True, 128, {}),
    ("window1", [700], 2, 1, True, 1, {}),
    ("window_wider_than_tile", [257, 640], 16, 2, True, 300, {}),
    ("group8", [384, 255], 16, 2, True, 0, {"sink_range": (-4.0, 4.0)}),
    ("peaked_logits", [600], 8, 1, True, 0, {"qk_std": 2.0, "sink_range": (-10.0, 10.0)}),
    ("sinks_minus30", [450], 4, 2, True, 0, {"odd_head_sink": -30.0}),
    ("several_units", [1024, 1024, 640, 1500], 16, 2, True, 0, {}),
    ("group16", [300, 130], 16, 1, True, 0, {}),
    ("group3", [257, 100], 6, 2, True, 0, {}),
    ("window129", [520], 4, 1, True, 129, {}),
]


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_head_dim128_matches_oracle(cuda_lib, case):
    name, lengths, Hq, Hkv, causal, window, extra = case
    w = make(name + "_d128", lengths, Hq, Hkv, seed=300 + len(name), causal=causal, window=window,
             d=D, **extra)
    assert w.q.shape[2] == D and abs(w.scale - D ** -0.5) < 1e-12
    ref, *_ = run_oracle(w)
    cond = dsink_condition(w.sinks.numpy().astype(np.float64), ref["lse"], ref["o"], ref["_do"])
    got = None
    for det in (False, True):  # both requests take the fixed-order dq pass at head_dim 128
        g = run_cuda(w, deterministic=det)
        compare_full(w, g, ref)
        assert_dsinks(g["dsinks"], ref["dsinks"], cond)
        if got is not None:
            for key in g:
                assert np.array_equal(g[key], got[key], equal_nan=True), key
        got = g


def test_head_dim128_no_sink_and_scale(cuda_lib):
    w = make("nosink_d128", [333, 90], 8, 2, seed=17, d=D)
    ref, *_ = run_oracle(w, sinks=False, scale=0.05)
    got = run_cuda(w, sinks=False, scale=0.05)
    compare_full(w, got, ref)
    assert np.all(got["dsinks"] == 0)


def test_head_dim128_strided_qkv_views(cuda_lib):
    # q, k, v as views into one packed [total, Hq + 2 Hkv, 128] buffer
    w = make("packed_d128", [290, 130], 8, 2, seed=19, d=D)
    qkv = torch.cat([w.q, w.k, w.v], 1).cuda()
    q, k, v = qkv[:, :8], qkv[:, 8:10], qkv[:, 10:12]
    assert q.stride(0) == 12 * D
    got = run_cuda(w, q_view=q, k_view=k, v_view=v)
    ref, *_ = run_oracle(w)
    compare_full(w, got, ref)


def test_head_dim128_dense_group(cuda_lib):
    """A dense batch at the training shape's heads (B=2, T=2048, Hq=64,
    Hkv=8): whole GQA group 3 and both sequences against the oracle."""
    w = make("dense_d128", [2048, 2048], 64, 8, seed=23, d=D)
    got = run_cuda(w)
    ref, tok, qh, kvh = run_oracle(w, kv_groups=[3])
    compare_full(w, got, ref, tok=tok, qh=qh, kvh=kvh)
    cond = dsink_condition(w.sinks.numpy().astype(np.float64)[qh], ref["lse"], ref["o"], ref["_do"])
    assert_dsinks(got["dsinks"][qh], ref["dsinks"], cond)


def test_head_dim128_autograd(cuda_lib):
    w = make("autograd_d128", [256, 100], 8, 2, seed=29, d=D)
    q, k, v = (t.cuda().requires_grad_(True) for t in (w.q, w.k, w.v))
    s = w.sinks.cuda().requires_grad_(True)
    o = api.sink_attention(q, k, v, s, w.cu_seqlens.cuda(), w.max_seqlen)
    o.backward(w.dout.cuda())
    got = run_cuda(w)
    assert torch.equal(o.detach().float().cpu(), torch.from_numpy(got["o"]).float())
    assert torch.equal(q.grad.float().cpu(), torch.from_numpy(got["dq"]).float())
    assert torch.equal(k.grad.float().cpu(), torch.from_numpy(got["dk"]).float())
    assert torch.equal(v.grad.float().cpu(), torch.from_numpy(got["dv"]).float())
    assert _binding.device_error(reset=True) == 0


@pytest.mark.slow
def test_head_dim128_long_sequence_group(cuda_lib):
    """One causal sequence of 8192 tokens with peaked logits (q, k ~ 2 N(0,1),
    sinks ~ U(-10, 10)): every output of GQA group 1 (query heads 8-15), so
    each key tile's dK / dV accumulate over up to 64 query tiles x 8 heads in
    the block kernel, and the dq pass walks up to 64 key tiles per unit."""
    w = make("long_d128", [8192], 16, 2, seed=31, d=D, qk_std=2.0, sink_range=(-10.0, 10.0))
    got = run_cuda(w)
    ref, tok, qh, kvh = run_oracle(w, kv_groups=[1])
    compare_full(w, got, ref, tok=tok, qh=qh, kvh=kvh)
    cond = dsink_condition(w.sinks.numpy().astype(np.float64)[qh], ref["lse"], ref["o"], ref["_do"])
    assert_dsinks(got["dsinks"][qh], ref["dsinks"], cond)
