"""Pins for the fp64 oracle, each against something other than the oracle.

The pages print no worked example for sink attention (page "GPT-OSS Agentic RL
Training: A Practical Retrospective" only says, in "The Role of Attention
Sinks", that each head's sink is a learnable scalar acting as a virtual token
in the softmax, and, in "Implementation in FlashAttention v3", that a backward
for dL/dS_h was written). So the oracle is pinned by:

* torch's scaled-dot-product attention (math backend, fp64) with the sink
  appended as a real extra key whose score is S_h and whose value is zero --
  the "virtual token" reading done with a library routine; its autograd gives
  the reference gradients, including dS_h through the additive mask;
* sinks absent -> textbook causal attention (SDPA with is_causal);
* central finite differences of the oracle's own forward;
* closed forms: a single key, a window of one key, a hand-worked two-key case;
* invariants: probability mass (sink included) sums to one, shift invariance,
  GQA = explicit repetition, varlen = concatenation, window >= length = causal,
  and results independent of the thread count.
"""

import math
import zlib

import numpy as np
import pytest
import torch
from torch.nn.attention import SDPBackend, sdpa_kernel

import oracle

ALL = ("o", "lse", "dq", "dk", "dv", "dsinks")


def rand_case(rng, lengths, Hq, Hkv, d, sink_lo=-2.0, sink_hi=2.0):
    total = sum(lengths)
    cu = np.zeros(len(lengths) + 1, dtype=np.int32)
    cu[1:] = np.cumsum(lengths)
    q = rng.standard_normal((total, Hq, d))
    k = rng.standard_normal((total, Hkv, d))
    v = rng.standard_normal((total, Hkv, d))
    do = rng.standard_normal((total, Hq, d))
    s = rng.uniform(sink_lo, sink_hi, Hq)
    return q, k, v, do, s, cu


def allowed_mask(L, causal, window):
    i = torch.arange(L)[:, None]
    j = torch.arange(L)[None, :]
    m = torch.ones(L, L, dtype=torch.bool)
    if causal:
        m &= j <= i
    if window > 0:
        m &= (i - j) < window
    return m


def sdpa_reference(q, k, v, do, sinks, cu, causal, window, scale):
    """Sink attention through torch SDPA: per sequence, append one key with
    zero key vector, zero value and additive mask S_h. Returns the same dict
    as the oracle (o, lse, dq, dk, dv, dsinks) from torch autograd."""
    total, Hq, d = q.shape
    Hkv = k.shape[1]
    G = Hq // Hkv
    tq = torch.tensor(q, requires_grad=True)
    tk = torch.tensor(k, requires_grad=True)
    tv = torch.tensor(v, requires_grad=True)
    ts = torch.tensor(sinks, requires_grad=True) if sinks is not None else None
    outs, lses = [], []
    for b in range(len(cu) - 1):
        a, e = int(cu[b]), int(cu[b + 1])
        L = e - a
        if L == 0:
            continue
        qb = tq[a:e].transpose(0, 1)                          # [Hq, L, d]
        kb = tk[a:e].transpose(0, 1).repeat_interleave(G, 0)  # [Hq, L, d]
        vb = tv[a:e].transpose(0, 1).repeat_interleave(G, 0)
        allow = allowed_mask(L, causal, window)
        bias = torch.zeros(L, L, dtype=torch.float64).masked_fill(~allow, float("-inf"))
        bias = bias.expand(Hq, L, L)
        if ts is not None:
            zk = torch.zeros(Hq, 1, d, dtype=torch.float64)
            kb = torch.cat([kb, zk], 1)
            # extra value column marks the virtual token: its output is p_sink
            vb = torch.cat([torch.cat([vb, torch.zeros(Hq, L, 1, dtype=torch.float64)], 2),
                            torch.cat([zk, torch.ones(Hq, 1, 1, dtype=torch.float64)], 2)], 1)
            bias = torch.cat([bias, ts[:, None, None].expand(Hq, L, 1)], 2)
        else:
            vb = torch.cat([vb, torch.zeros(Hq, L, 1, dtype=torch.float64)], 2)
        with sdpa_kernel(SDPBackend.MATH):
            ob = torch.nn.functional.scaled_dot_product_attention(
                qb, kb, vb, attn_mask=bias, scale=scale)
        outs.append(ob[..., :d].transpose(0, 1))
        # LSE from the sink share: p_sink = exp(S - LSE)  =>  LSE = S - log p_sink
        if ts is not None:
            lses.append((ts[:, None] - torch.log(ob[..., d])).detach())
        else:
            lses.append(None)
    o = torch.cat(outs, 0) if outs else torch.zeros(0, Hq, d, dtype=torch.float64)
    (o * torch.tensor(do)).sum().backward()
    res = {"o": o.detach().numpy(), "dq": tq.grad.numpy(), "dk": tk.grad.numpy(),
           "dv": tv.grad.numpy()}
    if ts is not None:
        res["dsinks"] = ts.grad.numpy()
        res["lse"] = torch.cat([x for x in lses], 1).numpy() if lses else np.zeros((Hq, 0))
    return res


def relerr(a, b):
    den = np.linalg.norm(b)
    return np.linalg.norm(a - b) / (den if den > 0 else 1.0)


CASES = [
    # lengths, Hq, Hkv, d, causal, window
    ([17], 2, 2, 8, True, 0),
    ([33], 4, 2, 16, True, 0),
    ([5, 0, 12, 1], 4, 1, 8, True, 0),
    ([19], 4, 4, 4, False, 0),
    ([23, 9], 2, 1, 8, True, 3),
    ([16], 8, 2, 64, True, 1),
    ([31], 4, 2, 8, True, 5),
    ([40, 7], 4, 2, 128, True, 0),    # head_dim 128
    ([12], 2, 1, 128, False, 0),
]


@pytest.mark.parametrize("case", CASES)
def test_oracle_matches_sdpa_with_virtual_sink_key(case):
    lengths, Hq, Hkv, d, causal, window = case
    rng = np.random.default_rng(zlib.crc32(str(case).encode()))  # stable across processes
    q, k, v, do, s, cu = rand_case(rng, lengths, Hq, Hkv, d)
    scale = 1.0 / math.sqrt(d)
    got = oracle.sinkattn(q, k, v, s, cu, causal=causal, window=window, scale=scale,
                          dout=do, want=ALL, nthreads=3)
    ref = sdpa_reference(q, k, v, do, s, cu, causal, window, scale)
    for name in ALL:
        np.testing.assert_allclose(got[name], ref[name], rtol=1e-10, atol=1e-11, err_msg=name)


@pytest.mark.parametrize("case", CASES[:4])
def test_no_sink_is_textbook_attention(case):
    lengths, Hq, Hkv, d, causal, window = case
    rng = np.random.default_rng(7)
    q, k, v, do, s, cu = rand_case(rng, lengths, Hq, Hkv, d)
    got = oracle.sinkattn(q, k, v, None, cu, causal=causal, window=window, dout=do,
                          want=("o", "dq", "dk", "dv", "dsinks"))
    assert np.all(got["dsinks"] == 0.0)
    # textbook attention: SDPA with the built-in causal flag, no extra key
    G = Hq // Hkv
    tq, tk, tv = (torch.tensor(x, requires_grad=True) for x in (q, k, v))
    outs = []
    for b in range(len(cu) - 1):
        a, e = int(cu[b]), int(cu[b + 1])
        if e == a:
            continue
        with sdpa_kernel(SDPBackend.MATH):
            outs.append(torch.nn.functional.scaled_dot_product_attention(
                tq[a:e].transpose(0, 1), tk[a:e].transpose(0, 1).repeat_interleave(G, 0),
                tv[a:e].transpose(0, 1).repeat_interleave(G, 0), is_causal=causal).transpose(0, 1))
    o = torch.cat(outs, 0)
    (o * torch.tensor(do)).sum().backward()
    np.testing.assert_allclose(got["o"], o.detach().numpy(), rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(got["dq"], tq.grad.numpy(), rtol=1e-9, atol=1e-11)
    np.testing.assert_allclose(got["dk"], tk.grad.numpy(), rtol=1e-9, atol=1e-11)
    np.testing.assert_allclose(got["dv"], tv.grad.numpy(), rtol=1e-9, atol=1e-11)


def test_very_negative_sink_equals_no_sink():
    rng = np.random.default_rng(3)
    q, k, v, do, s, cu = rand_case(rng, [13, 7], 4, 2, 8)
    a = oracle.sinkattn(q, k, v, np.full(4, -80.0), cu, dout=do, want=ALL)
    b = oracle.sinkattn(q, k, v, None, cu, dout=do, want=ALL)
    for name in ("o", "lse", "dq", "dk", "dv"):
        np.testing.assert_allclose(a[name], b[name], rtol=1e-12, atol=1e-14)
    assert np.max(np.abs(a["dsinks"])) < 1e-25


@pytest.mark.parametrize("causal,window", [(True, 0), (False, 0), (True, 4)])
def test_gradients_match_central_differences(causal, window):
    rng = np.random.default_rng(11)
    q, k, v, do, s, cu = rand_case(rng, [6, 9], 4, 2, 4)
    scale = 0.37
    got = oracle.sinkattn(q, k, v, s, cu, causal=causal, window=window, scale=scale,
                          dout=do, want=ALL)

    def loss(q_, k_, v_, s_):
        o = oracle.sinkattn(q_, k_, v_, s_, cu, causal=causal, window=window, scale=scale,
                            want=("o",), nthreads=1)["o"]
        return float(np.sum(o * do))

    h = 1e-6
    args = {"dq": q, "dk": k, "dv": v, "dsinks": s}
    for name, x in args.items():
        fd = np.zeros_like(x)
        flat = x.reshape(-1)
        for idx in range(flat.size):
            keep = flat[idx]
            flat[idx] = keep + h
            lp = loss(q, k, v, s)
            flat[idx] = keep - h
            lm = loss(q, k, v, s)
            flat[idx] = keep
            fd.reshape(-1)[idx] = (lp - lm) / (2 * h)
        np.testing.assert_allclose(got[name], fd, rtol=1e-6, atol=1e-8, err_msg=name)


def test_hand_worked_two_key_case():
    # d = 1, scale = 1, S = 0; q = (1, 1), k = (0, ln 3), v = (2, 5), dO = (1, 1).
    # Row 0 sees key 0: Z = e^0 + e^0 = 2, P00 = 1/2, O0 = 1, p_sink = 1/2.
    # Row 1 sees keys 0, 1: Z = 1 + 1 + 3 = 5, P = (1/5, 3/5), O1 = 17/5, p_sink = 1/5.
    # D = (1, 17/5); dS_sink = -(1/2 * 1 + 1/5 * 17/5) = -1.18.
    # dS00 = 1/2 (2 - 1) = 1/2, dS10 = 1/5 (2 - 17/5) = -0.28, dS11 = 3/5 (5 - 17/5) = 0.96.
    q = np.array([[[1.0]], [[1.0]]])
    k = np.array([[[0.0]], [[math.log(3.0)]]])
    v = np.array([[[2.0]], [[5.0]]])
    do = np.ones((2, 1, 1))
    r = oracle.sinkattn(q, k, v, np.array([0.0]), [0, 2], scale=1.0, dout=do, want=ALL)
    np.testing.assert_allclose(r["o"].ravel(), [1.0, 3.4], rtol=1e-14)
    np.testing.assert_allclose(r["lse"].ravel(), [math.log(2), math.log(5)], rtol=1e-14)
    np.testing.assert_allclose(r["dsinks"], [-1.18], rtol=1e-13)
    np.testing.assert_allclose(r["dv"].ravel(), [0.7, 0.6], rtol=1e-13)
    np.testing.assert_allclose(r["dq"].ravel(), [0.0, 0.96 * math.log(3)], rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(r["dk"].ravel(), [0.22, 0.96], rtol=1e-13)


def test_single_key_closed_form():
    rng = np.random.default_rng(5)
    d = 16
    q = rng.standard_normal((1, 3, d))
    k = rng.standard_normal((1, 3, d))
    v = rng.standard_normal((1, 3, d))
    S = np.array([-1.0, 0.5, 3.0])
    r = oracle.sinkattn(q, k, v, S, [0, 1], scale=0.25, want=("o", "lse"))
    for h in range(3):
        sc = 0.25 * float(q[0, h] @ k[0, h])
        w = math.exp(sc) / (math.exp(sc) + math.exp(S[h]))
        np.testing.assert_allclose(r["o"][0, h], w * v[0, h], rtol=1e-13)
        np.testing.assert_allclose(r["lse"][h, 0], math.log(math.exp(sc) + math.exp(S[h])), rtol=1e-13)


def test_window_of_one_closed_form():
    rng = np.random.default_rng(6)
    q, k, v, do, s, cu = rand_case(rng, [9], 2, 2, 8)
    r = oracle.sinkattn(q, k, v, s, cu, window=1, scale=0.5, want=("o",))
    for i in range(9):
        for h in range(2):
            sc = 0.5 * float(q[i, h] @ k[i, h])
            w = math.exp(sc) / (math.exp(sc) + math.exp(s[h]))
            np.testing.assert_allclose(r["o"][i, h], w * v[i, h], rtol=1e-12)


def test_probability_mass_with_sink_sums_to_one():
    rng = np.random.default_rng(8)
    q, k, v, do, s, cu = rand_case(rng, [21, 4], 4, 2, 8, -5, 5)
    ones = np.ones_like(v)
    for causal, window in [(True, 0), (True, 3), (False, 0)]:
        r = oracle.sinkattn(q, k, ones, s, cu, causal=causal, window=window, want=("o", "lse"))
        # with every value vector all-ones, each output component is sum_j P_ij
        p_sink = np.exp(s[:, None] - r["lse"]).T      # [total, Hq]
        np.testing.assert_allclose(r["o"][..., 0] + p_sink, 1.0, rtol=0, atol=1e-12)
        np.testing.assert_allclose(r["o"][..., 0], r["o"][..., -1], rtol=0, atol=1e-15)


def test_shift_invariance():
    # Append a coordinate so every score of a row moves by delta: q' = [q, delta/scale],
    # k' = [k, 1]; with S' = S + delta, O is unchanged and LSE moves by delta.
    rng = np.random.default_rng(9)
    q, k, v, do, s, cu = rand_case(rng, [11], 2, 1, 8)
    scale, delta = 0.3, 1.75
    a = oracle.sinkattn(q, k, v, s, cu, scale=scale, want=("o", "lse"))
    q2 = np.concatenate([q, np.full(q.shape[:2] + (1,), delta / scale)], 2)
    k2 = np.concatenate([k, np.ones(k.shape[:2] + (1,))], 2)
    v2 = np.concatenate([v, np.zeros(v.shape[:2] + (1,))], 2)
    b = oracle.sinkattn(q2, k2, v2, s + delta, cu, scale=scale, want=("o", "lse"))
    np.testing.assert_allclose(b["o"][..., :8], a["o"], rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(b["lse"], a["lse"] + delta, rtol=1e-13)


def test_gqa_equals_repeated_kv():
    rng = np.random.default_rng(10)
    q, k, v, do, s, cu = rand_case(rng, [10, 6], 8, 2, 8)
    g = oracle.sinkattn(q, k, v, s, cu, dout=do, want=ALL)
    kr, vr = np.repeat(k, 4, axis=1), np.repeat(v, 4, axis=1)
    r = oracle.sinkattn(q, kr, vr, s, cu, dout=do, want=ALL)
    for name in ("o", "lse", "dq", "dsinks"):
        np.testing.assert_allclose(g[name], r[name], rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(g["dk"], r["dk"].reshape(16, 2, 4, 8).sum(2), rtol=1e-11, atol=1e-13)
    np.testing.assert_allclose(g["dv"], r["dv"].reshape(16, 2, 4, 8).sum(2), rtol=1e-11, atol=1e-13)


def test_varlen_is_concatenation_of_sequences():
    rng = np.random.default_rng(12)
    lengths = [7, 0, 13, 3]
    q, k, v, do, s, cu = rand_case(rng, lengths, 4, 2, 8)
    whole = oracle.sinkattn(q, k, v, s, cu, window=4, dout=do, want=ALL)
    dsum = np.zeros(4)
    for b in range(len(lengths)):
        a, e = cu[b], cu[b + 1]
        part = oracle.sinkattn(q[a:e], k[a:e], v[a:e], s, [0, e - a], window=4,
                               dout=do[a:e], want=ALL)
        for name in ("o", "dq", "dk", "dv"):
            np.testing.assert_allclose(whole[name][a:e], part[name], rtol=1e-13, atol=1e-15)
        np.testing.assert_allclose(whole["lse"][:, a:e], part["lse"], rtol=1e-13)
        dsum += part["dsinks"]
    np.testing.assert_allclose(whole["dsinks"], dsum, rtol=1e-12)


def test_wide_window_equals_causal():
    rng = np.random.default_rng(13)
    q, k, v, do, s, cu = rand_case(rng, [12, 5], 2, 1, 8)
    a = oracle.sinkattn(q, k, v, s, cu, window=12, dout=do, want=ALL)
    b = oracle.sinkattn(q, k, v, s, cu, window=0, dout=do, want=ALL)
    for name in ALL:
        np.testing.assert_array_equal(a[name], b[name])


def test_thread_count_does_not_change_results():
    rng = np.random.default_rng(14)
    q, k, v, do, s, cu = rand_case(rng, [70, 45], 4, 2, 8)
    a = oracle.sinkattn(q, k, v, s, cu, dout=do, want=ALL, nthreads=1)
    b = oracle.sinkattn(q, k, v, s, cu, dout=do, want=ALL, nthreads=7)
    for name in ALL:
        np.testing.assert_array_equal(a[name], b[name])


def test_rejects_bad_arguments():
    rng = np.random.default_rng(15)
    q, k, v, do, s, cu = rand_case(rng, [4], 4, 2, 8)
    with pytest.raises(ValueError):
        oracle.sinkattn(q, k, v, s, cu, causal=False, window=2)
    with pytest.raises(ValueError):
        oracle.sinkattn(q, k[:, :1].repeat(3, 1), v[:, :1].repeat(3, 1), s, cu)


@pytest.mark.parametrize("window", [0, 5])
def test_first_row_restriction_matches_full_run(window):
    # Rows >= r and keys >= r of each sequence, computed alone, equal the same
    # entries of the unrestricted run (causal: only rows >= r see keys >= r).
    rng = np.random.default_rng(16)
    q, k, v, do, s, cu = rand_case(rng, [40, 9, 23], 4, 2, 8)
    full = oracle.sinkattn(q, k, v, s, cu, window=window, dout=do, want=ALL)
    r = 11
    part = oracle.sinkattn(q, k, v, s, cu, window=window, dout=do, want=ALL, first_row=r)
    dsum = np.zeros(4)
    for b in range(3):
        a, e = cu[b], cu[b + 1]
        sl = slice(a + r, e)
        for name in ("o", "dq", "dk", "dv"):
            np.testing.assert_array_equal(part[name][sl], full[name][sl])
            assert not np.any(part[name][a:a + r])
        np.testing.assert_array_equal(part["lse"][:, sl], full["lse"][:, sl])
        p_sink = np.exp(s[:, None] - full["lse"][:, sl])            # [Hq, rows]
        D = np.einsum("thd,thd->ht", do[sl], full["o"][sl])
        dsum += -(p_sink * D).sum(1)
    np.testing.assert_allclose(part["dsinks"], dsum, rtol=1e-12)
