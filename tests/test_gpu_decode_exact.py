"""Exact decode against the training forward, bit for bit.

The pages' central failure is that the inference engine and the training
stack give different token probabilities for the same tokens (page "GPT-OSS
Agentic RL Training: A Practical Retrospective", section "Correcting
Training-Inference Mismatch via Attention Sinks"). sinkattn_decode_exact
computes each new query row exactly as sinkattn_fwd computes the row at the
last position of the same sequence, so its o and lse must equal that row of
the training forward bit for bit: torch.equal, no tolerance. The keys come
from a paged cache whose never-written slots hold NaN, with the blocks
placed in a random order; the training forward reads the same keys and values
laid out contiguously.
"""

import numpy as np
import pytest
import torch

import oracle
from attention_learnable_sinks_gb300 import _binding, api
from attention_learnable_sinks_gb300.workloads import make_decode

pytestmark = pytest.mark.gpu

CASES = [
    # name, lengths, Hq, Hkv, block_size, window, sinks, head_dim
    ("dense_shape", [2048] * 4, 64, 8, 64, 0, True, 64),
    ("ragged_bs16", [1, 127, 128, 129, 1000, 2500, 4097, 300], 8, 2, 16, 0, True, 64),
    ("window128_bs32", [1, 127, 128, 129, 1000, 2500, 4097, 300], 8, 2, 32, 128, True, 64),
    ("window100_bs128", [99, 100, 101, 228, 1000, 3000], 16, 2, 128, 100, True, 64),
    ("window_longer_than_all", [50, 700], 4, 4, 64, 5000, True, 64),
    ("no_sink", [640, 77, 1500], 8, 1, 64, 0, False, 64),
    # head_dim 128: two 64-feature panels per cache block
    ("d128_dense_shape", [2048] * 4, 64, 8, 64, 0, True, 128),
    ("d128_ragged_bs16", [1, 127, 128, 129, 1000, 2500, 4097, 300], 8, 2, 16, 0, True, 128),
    ("d128_window128_bs32", [1, 127, 128, 129, 1000, 2500, 4097, 300], 8, 2, 32, 128, True, 128),
    ("d128_no_sink_bs128", [640, 77, 1500], 8, 1, 128, 0, False, 128),
]


def _training_last_rows(w, sinks):
    """sinkattn_fwd over the same keys laid out contiguously, the decode query
    at each sequence's last position: (o, lse) of those rows."""
    lens = w.meta["lengths"]
    cu = np.zeros(len(lens) + 1, dtype=np.int32)
    cu[1:] = np.cumsum(lens)
    gen = torch.Generator().manual_seed(11)
    q = torch.randn(int(cu[-1]), w.Hq, w.q.shape[2], generator=gen).to(torch.bfloat16)
    for b, L in enumerate(lens):
        if L:
            q[cu[b] + L - 1] = w.q[b]
    dev = "cuda"
    o, lse = api.forward(q.to(dev), w.meta["k_tokens"].to(dev), w.meta["v_tokens"].to(dev),
                         w.sinks.to(dev) if sinks else None, torch.from_numpy(cu).to(dev),
                         max(lens), causal=True, window=w.window, scale=w.scale)
    last = torch.from_numpy((cu[1:] - 1).astype(np.int64)).to(dev)
    return o[last], lse[:, last]


def _exact(w, sinks, table=None):
    dev = "cuda"
    return api.decode(w.q.to(dev), w.k_cache.to(dev), w.v_cache.to(dev),
                      (w.block_table if table is None else table).to(dev), w.seqlens.to(dev),
                      w.sinks.to(dev) if sinks else None, window=w.window, scale=w.scale,
                      exact=True)


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_exact_decode_equals_training_forward_bitwise(cuda_lib, case):
    name, lengths, Hq, Hkv, bs, window, sinks, d = case
    w = make_decode(name, lengths, Hq, Hkv, bs, seed=40 + len(name), window=window, d=d)
    o_train, lse_train = _training_last_rows(w, sinks)
    o_dec, lse_dec = _exact(w, sinks)
    torch.cuda.synchronize()
    assert _binding.device_error(reset=True) == 0
    assert torch.equal(o_dec, o_train), "o differs from the training forward's last rows"
    assert torch.equal(lse_dec, lse_train), "lse differs from the training forward's last rows"
    # ... and the same result as the split decode up to rounding
    o_split, lse_split = api.decode(w.q.cuda(), w.k_cache.cuda(), w.v_cache.cuda(),
                                    w.block_table.cuda(), w.seqlens.cuda(),
                                    w.sinks.cuda() if sinks else None, window=w.window,
                                    scale=w.scale)
    rel = (o_split.float() - o_dec.float()).norm() / o_dec.float().norm()
    assert rel <= 5e-3


def test_exact_decode_matches_oracle_with_empty_sequences(cuda_lib):
    """Against the fp64 decode oracle, with sequences of no keys (o = 0,
    lse = S_h) and table entries before the window holding garbage."""
    from oracle import decode as odec
    w = make_decode("exact_oracle", [0, 1, 300, 0, 2000], 8, 2, 32, seed=51, window=200)
    t = w.block_table.clone()
    t[4, : (2000 - 200) // 32] = -5  # wholly before the window: never read
    o, lse = _exact(w, True, table=t)
    torch.cuda.synchronize()
    assert _binding.device_error(reset=True) == 0

    def f64(x):
        return x.float().cpu().numpy().astype(np.float64)
    ro, rlse = odec.decode(f64(w.q), f64(w.k_cache), f64(w.v_cache), w.block_table.numpy(),
                           w.seqlens.numpy(), w.sinks.numpy(), window=w.window, scale=w.scale)
    got_o, got_lse = f64(o), f64(lse)
    for b, L in enumerate(w.meta["lengths"]):
        if L == 0:
            assert np.all(got_o[b] == 0)
            np.testing.assert_array_equal(got_lse[:, b], w.sinks.numpy().astype(np.float64))
            continue
        rel = np.linalg.norm(got_o[b] - ro[b]) / np.linalg.norm(ro[b])
        assert rel <= 1e-2, (b, rel)
        assert np.abs(got_lse[:, b] - rlse[:, b]).max() <= 1e-3


def test_exact_decode_head_dim128_matches_oracle(cuda_lib):
    from oracle import decode as odec
    w = make_decode("exact_oracle_d128", [0, 1, 300, 2000], 8, 2, 32, seed=53, window=200, d=128)
    o, lse = _exact(w, True)
    torch.cuda.synchronize()
    assert _binding.device_error(reset=True) == 0

    def f64(x):
        return x.float().cpu().numpy().astype(np.float64)
    ro, rlse = odec.decode(f64(w.q), f64(w.k_cache), f64(w.v_cache), w.block_table.numpy(),
                           w.seqlens.numpy(), w.sinks.numpy(), window=w.window, scale=w.scale)
    got_o, got_lse = f64(o), f64(lse)
    for b, L in enumerate(w.meta["lengths"]):
        if L == 0:
            assert np.all(got_o[b] == 0)
            continue
        rel = np.linalg.norm(got_o[b] - ro[b]) / np.linalg.norm(ro[b])
        assert rel <= 1e-2, (b, rel)
        assert np.abs(got_lse[:, b] - rlse[:, b]).max() <= 1e-3


def test_exact_decode_reports_bad_block_index(cuda_lib):
    w = make_decode("exact_bad", [300, 500], 8, 2, 16, seed=52)
    t = w.block_table.clone()
    t[1, 2] = w.k_cache.shape[0] + 3
    _exact(w, True, table=t)
    torch.cuda.synchronize()
    assert _binding.device_error(reset=True) == 1
