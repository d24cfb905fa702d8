"""Multi-rank layouts on CPU ranks (gloo, world sizes 2 to 4), with the fp64
oracle standing in for the kernels on each rank.

* Data parallel: the batch's sequences are split by attention cost; each rank
  computes its sequences and the per-head sink gradients are summed with one
  all-reduce. Every output must equal the single-process oracle on the whole
  batch (rows and keys at the same global positions), dL/dS_h included.
* Head-split sequence parallelism (all-to-all to a head split before
  attention and back after it): each rank holds a contiguous token slice with
  all heads; after the exchange, attention runs on whole sequences for the
  rank's heads with their sinks, and the outputs come back to the token
  slices. Every output must equal the single-process oracle, and each rank's
  dL/dS_h for its heads is already complete.
"""

import os
import socket

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

import oracle
from attention_learnable_sinks_gb300 import sharding
from attention_learnable_sinks_gb300.workloads import make

ALL = ("o", "lse", "dq", "dk", "dv", "dsinks")


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _workload(d=64, hkv=2):
    # ragged lengths, an empty and a length-1 sequence, GQA 8:hkv
    return make("multirank", [150, 37, 0, 260, 1, 90], 8, hkv, seed=41, sink_range=(-3.0, 3.0), d=d)


def _f64(t):
    return t.float().numpy().astype(np.float64)


def _oracle_fwd(q, k, v, s, cu, max_seqlen, causal, window, scale):
    r = oracle.sinkattn(q.numpy(), k.numpy(), v.numpy(), None if s is None else s.numpy(),
                        cu.numpy(), causal=causal, window=window, scale=scale, want=("o", "lse"),
                        nthreads=2)
    return torch.from_numpy(r["o"]), torch.from_numpy(r["lse"])


def _oracle_bwd(q, k, v, s, cu, max_seqlen, o, lse, dout, causal, window, scale):
    r = oracle.sinkattn(q.numpy(), k.numpy(), v.numpy(), None if s is None else s.numpy(),
                        cu.numpy(), causal=causal, window=window, scale=scale,
                        dout=dout.numpy(), want=("dq", "dk", "dv", "dsinks"), nthreads=2)
    return (torch.from_numpy(r["dq"]), torch.from_numpy(r["dk"]), torch.from_numpy(r["dv"]),
            torch.from_numpy(r["dsinks"]))


def _reference(w):
    return oracle.sinkattn(_f64(w.q), _f64(w.k), _f64(w.v), _f64(w.sinks), w.cu_seqlens.numpy(),
                           causal=w.causal, window=w.window, scale=w.scale, dout=_f64(w.dout),
                           want=ALL, nthreads=2)


def _spawn(fn, world, *args):
    port = _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.SimpleQueue()
    procs = [ctx.Process(target=_entry, args=(fn, r, world, port, q, *args)) for r in range(world)]
    for p in procs:
        p.start()
    results = [q.get() for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0, f"rank process exited with {p.exitcode}"
    errs = [r for r in results if isinstance(r, str)]
    assert not errs, errs[0]
    return sorted(results, key=lambda r: r["rank"])


def _entry(fn, rank, world, port, q, *args):
    import traceback
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    try:
        dist.init_process_group("gloo", rank=rank, world_size=world)
        q.put(fn(rank, world, *args))
    except Exception:
        q.put(f"rank {rank}:\n{traceback.format_exc()}")
    finally:
        if dist.is_initialized():
            dist.destroy_process_group()


def _rank_data_parallel(rank, world, d=64):
    w = _workload(d)
    lens = (w.cu_seqlens[1:] - w.cu_seqlens[:-1]).tolist()
    parts = sharding.partition_sequences(lens, world, w.causal, w.window)
    tok, cu, maxlen = sharding.shard_tokens(w.cu_seqlens.tolist(), parts[rank])
    q, k, v, do = (_f64(t[tok]) for t in (w.q, w.k, w.v, w.dout))
    r = oracle.sinkattn(q, k, v, _f64(w.sinks), cu.numpy(), causal=w.causal, window=w.window,
                        scale=w.scale, dout=do, want=ALL, nthreads=2)
    ds = torch.from_numpy(r["dsinks"].copy())
    sharding.all_reduce_sink_grad(ds)
    r["dsinks_reduced"] = ds.numpy()
    return {"rank": rank, "tok": tok.numpy(), "seqs": parts[rank], **r}


@pytest.mark.parametrize("world, d", [(2, 64), (2, 128), (3, 64), (4, 64)])
def test_data_parallel_split_matches_whole_batch(world, d):
    w = _workload(d)
    ref = _reference(w)
    res = _spawn(_rank_data_parallel, world, d)
    seen = sorted(b for r in res for b in r["seqs"])
    assert seen == list(range(w.nseq)), "every sequence on exactly one rank"
    for r in res:
        tok = r["tok"]
        for name in ("o", "dq", "dk", "dv"):
            np.testing.assert_allclose(r[name], ref[name][tok], rtol=0, atol=1e-12)
        np.testing.assert_allclose(r["lse"], ref["lse"][:, tok], rtol=0, atol=1e-12)
        # after the all-reduce every rank holds the whole batch's dL/dS_h
        np.testing.assert_allclose(r["dsinks_reduced"], ref["dsinks"], rtol=1e-12, atol=1e-14)
    # and each rank alone held only part of it
    assert not np.allclose(res[0]["dsinks"], ref["dsinks"])


def _rank_head_split(rank, world, d=64, hkv=2):
    import torch.distributed as dist
    w = _workload(d, hkv)
    splits = sharding.token_split(w.total, world)
    t0 = sum(splits[:rank])
    sl = slice(t0, t0 + splits[rank])
    q, k, v, do = (torch.from_numpy(_f64(t[sl])) for t in (w.q, w.k, w.v, w.dout))
    sinks = torch.from_numpy(_f64(w.sinks))
    layer = sharding.HeadSplitAttention(w.cu_seqlens, w.max_seqlen, causal=w.causal,
                                        window=w.window, scale=w.scale, fwd_fn=_oracle_fwd,
                                        bwd_fn=_oracle_bwd)
    o = layer.forward(q, k, v, sinks)
    dq, dk, dv, ds = layer.backward(do)
    full = sharding.gather_sink_grad(ds)
    hs = sharding.head_slice(w.Hq)
    # the rank's own sink gradient needs no exchange: compare it before the sum
    own = ds[hs].numpy().copy()
    dist.barrier()
    return {"rank": rank, "slice": (sl.start, sl.stop), "heads": (hs.start, hs.stop),
            "o": o.numpy(), "dq": dq.numpy(), "dk": dk.numpy(), "dv": dv.numpy(),
            "dsinks_own": own, "dsinks": full.numpy(), "zero_elsewhere":
            bool((ds.numpy()[np.r_[0:hs.start, hs.stop:w.Hq]] == 0).all())}


@pytest.mark.parametrize("world, d, hkv", [(2, 64, 2), (2, 128, 2), (4, 64, 4)])
def test_head_split_all_to_all_matches_single_process(world, d, hkv):
    w = _workload(d, hkv)
    ref = _reference(w)
    res = _spawn(_rank_head_split, world, d, hkv)
    bounds = np.cumsum([0] + sharding.token_split(w.total, world))
    assert [r["slice"] for r in res] == [(int(a), int(b)) for a, b in zip(bounds[:-1], bounds[1:])]
    for r in res:
        a, b = r["slice"]
        for name in ("o", "dq", "dk", "dv"):
            np.testing.assert_allclose(r[name], ref[name][a:b], rtol=0, atol=1e-12)
        h0, h1 = r["heads"]
        np.testing.assert_allclose(r["dsinks_own"], ref["dsinks"][h0:h1], rtol=1e-12, atol=1e-14)
        assert r["zero_elsewhere"]
        np.testing.assert_allclose(r["dsinks"], ref["dsinks"], rtol=1e-12, atol=1e-14)


def test_partition_balances_cost():
    lens = [8192, 256, 4000, 4000, 3000, 100, 7000, 1, 0, 5000]
    for world in (1, 2, 3, 4, 8):
        parts = sharding.partition_sequences(lens, world)
        assert sorted(b for p in parts for b in p) == list(range(len(lens)))
        costs = [sum(sharding.attention_cost(lens[b]) for b in p) for p in parts]
        biggest = max(sharding.attention_cost(L) for L in lens)
        # greedy longest-first: no rank exceeds the mean by more than one sequence
        assert max(costs) <= sum(costs) / world + biggest
    assert sharding.partition_sequences([5, 5], 4)[2:] == [[], []]


def test_token_split_and_exchange_shapes():
    assert sharding.token_split(10, 4) == [3, 3, 2, 2]
    assert sharding.token_split(3, 4) == [1, 1, 1, 0]
    with pytest.raises(ValueError):
        sharding.partition_sequences([1], 0)
