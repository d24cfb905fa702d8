"""Pins for the decode oracle (``oracle.decode``), each against something other
than the function itself: the C oracle's full-sequence forward (a separate
implementation, row by row), a worked two-key example with exact numbers, the
one-key closed form, the sink alone, a constant-value invariant, relabelled
physical blocks, and keys outside the window or past the end never read."""

import math

import numpy as np
import pytest
import torch

import oracle
from oracle import decode as odec
from attention_learnable_sinks_gb300.workloads import make_decode


def _f64(t):
    return t.float().numpy().astype(np.float64)


def _full_sequence_last_rows(w):
    """Last row of each sequence from the C oracle's causal forward on the
    same keys laid out contiguously (earlier query rows are arbitrary)."""
    lens = w.meta["lengths"]
    cu = np.zeros(len(lens) + 1, dtype=np.int32)
    cu[1:] = np.cumsum(lens)
    total = int(cu[-1])
    rng = np.random.default_rng(0)
    q = rng.standard_normal((total, w.Hq, w.q.shape[2]))
    for b, L in enumerate(lens):
        if L:
            q[cu[b] + L - 1] = _f64(w.q[b])
    ref = oracle.sinkattn(q, _f64(w.meta["k_tokens"]), _f64(w.meta["v_tokens"]),
                          w.sinks.numpy().astype(np.float64), cu, causal=True, window=w.window,
                          scale=w.scale)
    return ref, cu


@pytest.mark.parametrize("lengths,Hq,Hkv,bs,window,d", [
    ([1, 5, 130, 300], 8, 2, 16, 0, 64),
    ([17, 129, 256], 4, 1, 128, 0, 64),
    ([200, 64, 9], 8, 4, 32, 7, 64),
    ([300, 129], 4, 2, 64, 128, 64),
    ([1, 5, 130, 300], 8, 2, 16, 0, 128),
    ([300, 129], 4, 2, 64, 128, 128),
])
def test_matches_last_row_of_c_oracle(lengths, Hq, Hkv, bs, window, d):
    w = make_decode("pin", lengths, Hq, Hkv, bs, seed=11, window=window, d=d)
    o, lse = odec.decode(_f64(w.q), _f64(w.k_cache), _f64(w.v_cache), w.block_table.numpy(),
                         w.seqlens.numpy(), w.sinks.numpy(), window=window, scale=w.scale)
    ref, cu = _full_sequence_last_rows(w)
    for b, L in enumerate(lengths):
        r = int(cu[b]) + L - 1
        np.testing.assert_allclose(o[b], ref["o"][r], rtol=0, atol=1e-12)
        np.testing.assert_allclose(lse[:, b], ref["lse"][:, r], rtol=0, atol=1e-12)


def test_worked_two_key_example():
    # scale 1, q = e_0; key 0 scores 0, key 1 scores ln 2, sink ln 3:
    # weights 1, 2, 3 -> Z = 6, o = (v0 + 2 v1) / 6, lse = ln 6
    q = np.zeros((1, 1, 64)); q[0, 0, 0] = 1.0
    k = np.zeros((1, 2, 1, 64)); k[0, 1, 0, 0] = math.log(2.0)
    v = np.zeros((1, 2, 1, 64)); v[0, 0, 0, :] = 6.0; v[0, 1, 0, :] = np.arange(64.0)
    o, lse = odec.decode(q, k, v, np.array([[0]]), np.array([2]), np.array([math.log(3.0)]),
                         scale=1.0)
    np.testing.assert_allclose(o[0, 0], (6.0 + 2.0 * np.arange(64.0)) / 6.0, rtol=1e-14)
    assert abs(lse[0, 0] - math.log(6.0)) < 1e-14


def test_one_key_closed_form():
    rng = np.random.default_rng(3)
    q = rng.standard_normal((1, 2, 64))
    k = rng.standard_normal((2, 16, 1, 64))
    v = rng.standard_normal((2, 16, 1, 64))
    S = np.array([0.3, -1.7])
    o, lse = odec.decode(q, k, v, np.array([[1]]), np.array([1]), S)
    for h in range(2):
        s0 = float(q[0, h] @ k[1, 0, 0]) / 8.0
        p0 = 1.0 / (1.0 + math.exp(S[h] - s0))
        np.testing.assert_allclose(o[0, h], p0 * v[1, 0, 0], rtol=1e-13)
        assert abs(lse[h, 0] - math.log(math.exp(s0) + math.exp(S[h]))) < 1e-13


def test_sink_alone_and_no_keys():
    q = np.ones((2, 2, 64))
    cache = np.full((1, 16, 1, 64), np.nan)
    table = np.array([[0], [0]])
    o, lse = odec.decode(q, cache, cache, table, np.array([0, 0]), np.array([1.5, -2.0]))
    assert np.all(o == 0) and np.allclose(lse[:, 0], [1.5, -2.0])
    o, lse = odec.decode(q, cache, cache, table, np.array([0, 0]), None)
    assert np.all(o == 0) and np.all(lse == -np.inf)


def test_constant_values_give_one_minus_sink_mass():
    # with every value row equal to c, o = c * (1 - exp(S_h - lse))
    w = make_decode("const", [40, 333], 8, 2, 16, seed=5, window=100)
    c = np.linspace(-1.0, 1.0, 64)
    v = np.broadcast_to(c, w.v_cache.shape).copy()
    o, lse = odec.decode(_f64(w.q), _f64(w.k_cache), v, w.block_table.numpy(), w.seqlens.numpy(),
                         w.sinks.numpy(), window=w.window)
    S = w.sinks.numpy().astype(np.float64)
    for b in range(2):
        mass = 1.0 - np.exp(S - lse[:, b])
        np.testing.assert_allclose(o[b], mass[:, None] * c[None, :], rtol=1e-12, atol=1e-14)


def test_relabelled_blocks_and_unread_slots():
    w = make_decode("perm", [77, 300, 1], 4, 2, 32, seed=9, window=64)
    args = dict(window=w.window, scale=w.scale)
    base = odec.decode(_f64(w.q), _f64(w.k_cache), _f64(w.v_cache), w.block_table.numpy(),
                       w.seqlens.numpy(), w.sinks.numpy(), **args)
    assert np.all(np.isfinite(base[0])) and np.all(np.isfinite(base[1]))
    # move every physical block to a new slot
    nb = w.k_cache.shape[0]
    perm = np.random.default_rng(1).permutation(nb)
    inv = np.empty_like(perm); inv[perm] = np.arange(nb)
    table = w.block_table.numpy().copy()
    table[table >= 0] = inv[table[table >= 0]]
    kc, vc = _f64(w.k_cache)[perm], _f64(w.v_cache)[perm]
    got = odec.decode(_f64(w.q), kc, vc, table, w.seqlens.numpy(), w.sinks.numpy(), **args)
    np.testing.assert_array_equal(got[0], base[0])
    np.testing.assert_array_equal(got[1], base[1])
    # entries of blocks wholly before the window are never looked up
    t2 = w.block_table.numpy().copy()
    t2[1, : (300 - 64) // 32] = 10 ** 6
    got = odec.decode(_f64(w.q), _f64(w.k_cache), _f64(w.v_cache), t2, w.seqlens.numpy(),
                      w.sinks.numpy(), **args)
    np.testing.assert_array_equal(got[0], base[0])


def test_window_longer_than_sequence_is_no_window():
    w = make_decode("wide", [50, 90], 4, 1, 16, seed=2)
    a = odec.decode(_f64(w.q), _f64(w.k_cache), _f64(w.v_cache), w.block_table.numpy(),
                    w.seqlens.numpy(), w.sinks.numpy())
    b = odec.decode(_f64(w.q), _f64(w.k_cache), _f64(w.v_cache), w.block_table.numpy(),
                    w.seqlens.numpy(), w.sinks.numpy(), window=90)
    np.testing.assert_array_equal(a[0], b[0])
    np.testing.assert_array_equal(a[1], b[1])
