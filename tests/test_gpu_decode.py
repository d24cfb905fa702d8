"""Decode over a paged KV cache (``sinkattn_decode``) against the fp64 decode
oracle, element by element: every cache block size, GQA group sizes 1 to 16,
windows, forced and automatic split counts (empty splits included), empty
and one-key sequences, no sink, and the last row of the library's own
forward on the same keys. Unused cache slots hold NaN, so a read outside the
visible keys shows up as a NaN in the output."""

import numpy as np
import pytest
import torch

from oracle import decode as odec
from attention_learnable_sinks_gb300 import _binding, api
from attention_learnable_sinks_gb300.workloads import decode_config, make_decode

pytestmark = pytest.mark.gpu

TOL_REL = 1e-2   # relative L2 per (sequence, head) on O: bf16 in and out, fp32 sums
TOL_LSE = 1e-3   # max abs on LSE (natural log)


def f64(t):
    return t.detach().float().cpu().numpy().astype(np.float64)


def run_cuda(w, num_splits=0, sinks=True, table=None, seqlens=None):
    dev = "cuda"
    o, lse = api.decode(w.q.to(dev), w.k_cache.to(dev), w.v_cache.to(dev),
                        (w.block_table if table is None else table).to(dev),
                        (w.seqlens if seqlens is None else seqlens).to(dev),
                        w.sinks.to(dev) if sinks else None, window=w.window, scale=w.scale,
                        num_splits=num_splits)
    torch.cuda.synchronize()
    return f64(o), f64(lse)


def run_oracle(w, sinks=True):
    return odec.decode(f64(w.q), f64(w.k_cache), f64(w.v_cache), w.block_table.numpy(),
                       w.seqlens.numpy(), w.sinks.numpy() if sinks else None, window=w.window,
                       scale=w.scale)


def compare(w, got, ref, seqs=None):
    o, lse = got
    ro, rlse = ref
    seqs = range(w.nseq) if seqs is None else seqs
    for b in seqs:
        L = int(w.seqlens[b])
        if L == 0:
            assert np.all(o[b] == 0), f"sequence {b} without keys: o must be 0"
        for h in range(w.Hq):
            n = np.linalg.norm(ro[b, h])
            if n > 0:
                rel = np.linalg.norm(o[b, h] - ro[b, h]) / n
                assert rel <= TOL_REL, f"o seq {b} head {h}: rel L2 {rel:.3g}"
        same = lse[:, b] == rlse[:, b]  # equal infinities included
        diff = np.subtract(lse[:, b], rlse[:, b], out=np.zeros_like(rlse[:, b]), where=~same)
        err = np.abs(diff)
        assert np.all(err <= TOL_LSE), f"lse seq {b}: max err {err.max():.3g}"


CASES = [
    # name, lengths, Hq, Hkv, block_size, window, num_splits, extra
    ("basic_bs16", [1, 5, 127, 128, 129, 1000], 8, 2, 16, 0, 0, {}),
    ("empty_and_one_bs32", [0, 1, 0, 2, 33], 4, 4, 32, 0, 0, {}),
    ("g1_bs128_3splits", [300, 2000], 4, 4, 128, 0, 3, {}),
    ("g16_bs64", [700, 64, 4096], 16, 1, 64, 0, 0, {}),
    ("g8_window128", [50, 128, 129, 1000, 3000], 16, 2, 64, 128, 0, {}),
    ("window1", [1, 2, 500], 8, 2, 16, 1, 0, {}),
    ("window300_bs32_5splits", [299, 300, 301, 2000], 8, 1, 32, 300, 5, {}),
    ("64_splits_some_empty", [5000, 3], 8, 2, 16, 0, 64, {}),
    ("one_split", [5000, 17], 8, 2, 64, 0, 1, {}),
    ("peaked_logits", [900, 1500], 8, 1, 16, 0, 0, {"qk_std": 2.0, "sink_range": (-10.0, 10.0)}),
    ("sinks_minus30", [450, 33], 4, 2, 64, 0, 0, {"odd_head_sink": -30.0}),
    ("g2_window_long", [8192, 4000], 4, 2, 128, 1000, 0, {}),
    # head_dim 128: two 64-feature panels per cache block, M = 128 output dims
    ("d128_basic_bs16", [1, 5, 127, 128, 129, 1000], 8, 2, 16, 0, 0, {"d": 128}),
    ("d128_empty_and_one_bs32", [0, 1, 0, 2, 33], 4, 4, 32, 0, 0, {"d": 128}),
    ("d128_g16_bs64", [700, 64, 4096], 16, 1, 64, 0, 0, {"d": 128}),
    ("d128_window300_5splits", [299, 300, 301, 2000], 8, 1, 32, 300, 5, {"d": 128}),
    ("d128_one_split", [5000, 17], 8, 2, 64, 0, 1, {"d": 128}),
    ("d128_64_splits_some_empty", [5000, 3], 8, 2, 16, 0, 64, {"d": 128}),
    ("d128_peaked_bs128", [900, 1500], 8, 1, 128, 0, 0,
     {"d": 128, "qk_std": 2.0, "sink_range": (-10.0, 10.0)}),
]


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_decode_matches_oracle(cuda_lib, case):
    name, lengths, Hq, Hkv, bs, window, splits, extra = case
    w = make_decode(name, lengths, Hq, Hkv, bs, seed=200 + len(name), window=window, **extra)
    got = run_cuda(w, num_splits=splits)
    assert _binding.device_error(reset=True) == 0
    assert np.all(np.isfinite(got[0]))
    compare(w, got, run_oracle(w))


def test_decode_without_sink(cuda_lib):
    w = make_decode("nosink", [0, 1, 260, 1300], 8, 2, 16, seed=3, window=200)
    got = run_cuda(w, sinks=False)
    ref = run_oracle(w, sinks=False)
    compare(w, got, ref)
    assert np.all(got[1][:, 0] == -np.inf)


def test_split_count_does_not_change_the_result_much(cuda_lib):
    w = make_decode("splits", [3000, 77, 1025], 8, 2, 32, seed=4)
    ref = run_oracle(w)
    outs = [run_cuda(w, num_splits=s) for s in (1, 2, 7, 24, 0)]
    for got in outs:
        compare(w, got, ref)


def test_decode_equals_last_row_of_forward(cuda_lib):
    """The same keys laid out contiguously through sinkattn_fwd: its last row
    per sequence is the decode query's output."""
    w = make_decode("vsfwd", [1, 200, 1000, 2500], 8, 2, 64, seed=8, window=256)
    lens = w.meta["lengths"]
    cu = np.zeros(len(lens) + 1, dtype=np.int32)
    cu[1:] = np.cumsum(lens)
    g = torch.Generator().manual_seed(1)
    q = torch.randn(int(cu[-1]), w.Hq, 64, generator=g).to(torch.bfloat16)
    for b, L in enumerate(lens):
        q[cu[b] + L - 1] = w.q[b]
    dev = "cuda"
    o, lse = api.forward(q.to(dev), w.meta["k_tokens"].to(dev), w.meta["v_tokens"].to(dev),
                         w.sinks.to(dev), torch.from_numpy(cu).to(dev), max(lens), causal=True,
                         window=w.window, scale=w.scale)
    do, dlse = run_cuda(w)
    last = cu[1:] - 1
    fo, flse = f64(o)[last], f64(lse)[:, last]
    for b in range(len(lens)):
        for h in range(w.Hq):
            rel = np.linalg.norm(do[b, h] - fo[b, h]) / np.linalg.norm(fo[b, h])
            assert rel <= 5e-3, (b, h, rel)
    assert np.abs(dlse - flse).max() <= 1e-3


def test_table_entries_before_the_window_are_ignored(cuda_lib):
    w = make_decode("ignored", [1000, 130], 8, 2, 16, seed=12, window=100)
    base = run_cuda(w)
    t = w.block_table.clone()
    t[0, : (1000 - 100) // 16] = -7
    t[0, (1000 + 15) // 16:] = 10 ** 6  # past the last block
    got = run_cuda(w, table=t)
    assert _binding.device_error(reset=True) == 0
    np.testing.assert_array_equal(got[0], base[0])
    np.testing.assert_array_equal(got[1], base[1])


def test_bad_length_or_block_sets_the_device_error(cuda_lib):
    """Checked on the device before any copy: the bad sequence is reported
    through the error word; the others are still computed."""
    w = make_decode("bad", [300, 40, 500], 8, 2, 16, seed=13)
    ref = run_oracle(w)
    lens = w.seqlens.clone()
    lens[1] = w.block_table.shape[1] * 16 + 1
    got = run_cuda(w, seqlens=lens)
    assert _binding.device_error(reset=True) == 1
    compare(w, got, ref, seqs=[0, 2])
    t = w.block_table.clone()
    t[2, 3] = w.k_cache.shape[0] + 5
    got = run_cuda(w, table=t)
    assert _binding.device_error(reset=True) == 1
    compare(w, got, ref, seqs=[0, 1])


@pytest.mark.parametrize("name", ["decode", "decode_window"])
def test_decode_config_sampled(cuda_lib, name):
    """The benchmarked decode workloads at full size, in the launch the
    benchmark times (automatic split count), checked on a sample of sequences
    (the oracle is exact per sequence)."""
    w = decode_config(name)
    got = run_cuda(w)
    assert _binding.device_error(reset=True) == 0
    pick = [0, 7, 31, 63]
    sub = make_sub(w, pick)
    compare(sub, (got[0][pick], got[1][:, pick]), run_oracle(sub))


def make_sub(w, pick):
    """The same cache with only the picked sequences."""
    from dataclasses import replace
    return replace(w, q=w.q[pick], block_table=w.block_table[pick], seqlens=w.seqlens[pick])


def _random_decode(i):
    rng = np.random.default_rng(5000 + i)
    G = int(rng.choice([1, 2, 4, 8, 16]))
    Hkv = int(rng.integers(1, 3))
    edges = [0, 1, 2, 127, 128, 129, 255, 256, 257]
    lengths = [int(rng.choice(edges)) if rng.random() < 0.3 else int(rng.integers(0, 3001))
               for _ in range(int(rng.integers(1, 6)))]
    return dict(Hq=G * Hkv, Hkv=Hkv, lengths=lengths, bs=int(rng.choice([16, 32, 64, 128])),
                window=int(rng.choice([0, 0, 1, 100, 128, 1000])),
                splits=int(rng.choice([0, 0, 1, 3, 7])), d=64 if i % 2 == 0 else 128,
                seed=6000 + i)


@pytest.mark.parametrize("i", range(16))
def test_random_decode_matches_oracle(cuda_lib, i):
    """Seeded random draws: group size, kv heads, cache block size, lengths
    (tile edges and empty sequences on purpose), window, split count and
    head_dim; the split decode and the exact decode both against the oracle."""
    c = _random_decode(i)
    w = make_decode(f"random{i}", c["lengths"], c["Hq"], c["Hkv"], c["bs"], seed=c["seed"],
                    window=c["window"], d=c["d"])
    ref = run_oracle(w)
    got = run_cuda(w, num_splits=c["splits"])
    assert _binding.device_error(reset=True) == 0
    assert np.all(np.isfinite(got[0]))
    compare(w, got, ref)
    dev = "cuda"
    o, lse = api.decode(w.q.to(dev), w.k_cache.to(dev), w.v_cache.to(dev), w.block_table.to(dev),
                        w.seqlens.to(dev), w.sinks.to(dev), window=w.window, scale=w.scale,
                        exact=True)
    torch.cuda.synchronize()
    assert _binding.device_error(reset=True) == 0
    compare(w, (f64(o), f64(lse)), ref)
