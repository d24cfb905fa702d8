"""fp64 oracle for one decode step of attention with learnable sinks over a
paged KV cache.

TEST INFRASTRUCTURE ONLY, like the rest of this package: the test suite, the
smoke check and the benchmark's CPU-baseline leg are its only callers.

What is computed (page "GPT-OSS Agentic RL Training: A Practical
Retrospective"; "The Role of Attention Sinks" for the sink as a virtual token
that adds exp(S_h) to the softmax denominator and carries no value;
"Implementation in FlashAttention v3", step 1, for the forward with sinks,
which the pages took from an inference engine). For sequence b of length L
the query is the row at position L - 1; it sees keys j in [k0, L) with
k0 = max(0, L - W) under a window of W keys (k0 = 0 without one). Per query
head h, with kv head h // G:

    s_j = scale * <q_h, k_j>
    m   = max(S_h, max_j s_j)
    Z   = exp(S_h - m) + sum_j exp(s_j - m)
    o_h = sum_j exp(s_j - m) v_j / Z,      lse_h = m + log Z

A sequence with no keys gives o = 0 and lse = S_h (the sink alone), or
lse = -inf with no sink. Key j of sequence b lives in physical block
block_table[b, j // block_size], row j % block_size; only blocks holding a
visible key are read.

Pins (``tests/test_oracle_decode.py``): the last row of the C oracle's
full-sequence forward on the same keys (a separate implementation, row by
row), closed forms for one and two keys, the sink alone, probability mass
summing to one, invariance under relabelling physical blocks, and keys
outside the window or past the end (NaN in the cache) never reaching the
result.
"""

from __future__ import annotations

import numpy as np


def gather_keys(cache, block_table, b, lo, hi):
    """Rows [lo, hi) of sequence b from a paged cache [blocks, bs, H, d]."""
    bs = cache.shape[1]
    j = np.arange(lo, hi)
    blocks = np.asarray(block_table)[b, j // bs]
    return np.asarray(cache, dtype=np.float64)[blocks, j % bs]


def decode(q, k_cache, v_cache, block_table, seqlens, sinks, *, window=0, scale=None):
    """o [nseq, Hq, d] and lse [Hq, nseq], both fp64."""
    q = np.asarray(q, dtype=np.float64)
    nseq, Hq, d = q.shape
    Hkv = k_cache.shape[2]
    G = Hq // Hkv
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    s_h = None if sinks is None else np.asarray(sinks, dtype=np.float64)
    o = np.zeros((nseq, Hq, d))
    lse = np.zeros((Hq, nseq))
    for b in range(nseq):
        L = int(seqlens[b])
        k0 = max(0, L - window) if window > 0 else 0
        K = gather_keys(k_cache, block_table, b, k0, L)  # [n, Hkv, d]
        V = gather_keys(v_cache, block_table, b, k0, L)
        for h in range(Hq):
            g = h // G
            s = scale * (K[:, g, :] @ q[b, h])           # [n]
            m = max(s.max(initial=-np.inf), -np.inf if s_h is None else s_h[h])
            if m == -np.inf:                             # no keys and no sink
                lse[h, b] = -np.inf
                continue
            e = np.exp(s - m)
            Z = e.sum() + (0.0 if s_h is None else np.exp(s_h[h] - m))
            o[b, h] = (e @ V[:, g, :]) / Z
            lse[h, b] = m + np.log(Z)
    return o, lse
