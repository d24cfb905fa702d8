"""Multi-GPU layouts of sink attention: one process per GPU.

Two ways to split the work (page "GPT-OSS Agentic RL Training: A Practical
Retrospective"):

* Data parallel over whole sequences (``partition_sequences``,
  ``shard_tokens``, ``all_reduce_sink_grad``). Sequences never attend to each
  other, so each rank runs the forward and backward of its own sequences with
  no exchange at all. The one exchange of the path is the per-head sink
  gradient dL/dS_h: a sum over every row of every sequence, so the ranks'
  partial sums are added with one all-reduce of Hq floats, next to the
  trainer's other gradient reductions.

* Head-split sequence parallelism (section "Sequence Parallelism with
  FlashAttention v3": an all-to-all before attention gathers the sequence and
  splits it by attention head, another after attention restores the
  sequence-parallel layout). Every rank holds one contiguous slice of the
  packed tokens with all heads. ``tokens_to_heads`` regroups q, k, v (and dO)
  so that each rank holds every token of its share of the heads, attention
  runs there on whole sequences, and ``heads_to_tokens`` sends the outputs
  (and dq, dk, dv) back. The sinks belong to heads: each rank takes the sinks
  of its heads, and the dS_h it computes is the complete gradient of those
  heads, so the sink gradient needs no reduction inside the group.

Query head h reads kv head h // (Hq / Hkv), so giving rank r the query heads
[r Hq/W, (r+1) Hq/W) and the kv heads [r Hkv/W, (r+1) Hkv/W) keeps every
GQA group on one rank; Hkv must be a multiple of the group size W.

Collectives go through ``torch.distributed`` (NCCL between GPUs, gloo on
CPU); the attention itself is whatever backend is passed in, by default the
CUDA library through ``api.forward`` / ``api.backward``.
"""

from __future__ import annotations

from typing import Callable, List, Optional, Sequence, Tuple

import torch
import torch.distributed as dist


# ----------------------------------------------------------------- data parallel
def attention_cost(L: int, causal: bool = True, window: int = 0) -> int:
    """(row, key) pairs the mask allows in one sequence of length L."""
    L = int(L)
    if not causal:
        return L * L
    if 0 < window < L:
        return window * (window + 1) // 2 + (L - window) * window
    return L * (L + 1) // 2


def partition_sequences(lengths: Sequence[int], world: int, causal: bool = True,
                        window: int = 0) -> List[List[int]]:
    """Whole sequences per rank, balancing attention cost: longest first, each
    to the rank with the least cost so far (ties to the lower rank). Returns
    ``world`` sorted lists of sequence indices; every index appears once."""
    if world < 1:
        raise ValueError("world must be >= 1")
    order = sorted(range(len(lengths)),
                   key=lambda b: (-attention_cost(lengths[b], causal, window), b))
    load = [0] * world
    parts: List[List[int]] = [[] for _ in range(world)]
    for b in order:
        r = min(range(world), key=lambda i: (load[i], i))
        parts[r].append(b)
        load[r] += attention_cost(lengths[b], causal, window)
    return [sorted(p) for p in parts]


def shard_tokens(cu_seqlens: Sequence[int], seqs: Sequence[int]
                 ) -> Tuple[torch.Tensor, torch.Tensor, int]:
    """Token indices (into the global packing) of the given sequences, in
    order, and the local cu_seqlens and max_seqlen of their packing."""
    cu = [int(x) for x in cu_seqlens]
    idx, local = [], [0]
    for b in seqs:
        idx.append(torch.arange(cu[b], cu[b + 1], dtype=torch.int64))
        local.append(local[-1] + cu[b + 1] - cu[b])
    tok = torch.cat(idx) if idx else torch.zeros(0, dtype=torch.int64)
    lens = [cu[b + 1] - cu[b] for b in seqs]
    return tok, torch.tensor(local, dtype=torch.int32), max(lens) if lens else 0


def all_reduce_sink_grad(dsinks: torch.Tensor, group=None) -> torch.Tensor:
    """Sum each rank's partial dL/dS_h (its sequences' rows) in place."""
    if dist.is_initialized() and dist.get_world_size(group) > 1:
        dist.all_reduce(dsinks, op=dist.ReduceOp.SUM, group=group)
    return dsinks


# ----------------------------------------------------------------- head split
def token_split(total: int, world: int) -> List[int]:
    """Tokens per rank of a packed batch: contiguous, as equal as possible
    (the first total % world ranks take one more)."""
    base, extra = divmod(int(total), world)
    return [base + (1 if r < extra else 0) for r in range(world)]


def _group_info(group):
    return dist.get_world_size(group), dist.get_rank(group)


def tokens_to_heads(x: torch.Tensor, splits: Sequence[int], group=None) -> torch.Tensor:
    """[tokens of this rank, H, d] -> [all tokens, H / W heads of this rank, d].

    Rank s receives, from every rank r in rank order, r's tokens of the heads
    [s H/W, (s+1) H/W), so the result lists the tokens in global order."""
    W, rank = _group_info(group)
    T_r, H, d = x.shape
    if H % W:
        raise ValueError(f"{H} heads do not split over {W} ranks")
    if T_r != splits[rank]:
        raise ValueError("the local token count does not match the split")
    Hs = H // W
    send = x.reshape(T_r, W, Hs, d).permute(1, 0, 2, 3).contiguous().reshape(W * T_r, Hs, d)
    recv = torch.empty(sum(splits), Hs, d, dtype=x.dtype, device=x.device)
    dist.all_to_all_single(recv, send, output_split_sizes=list(splits),
                           input_split_sizes=[T_r] * W, group=group)
    return recv


def heads_to_tokens(y: torch.Tensor, splits: Sequence[int], group=None) -> torch.Tensor:
    """[all tokens, H / W heads of this rank, d] -> [tokens of this rank, H, d];
    the inverse of ``tokens_to_heads``."""
    W, rank = _group_info(group)
    T, Hs, d = y.shape
    T_r = splits[rank]
    recv = torch.empty(W * T_r, Hs, d, dtype=y.dtype, device=y.device)
    dist.all_to_all_single(recv, y.contiguous(), output_split_sizes=[T_r] * W,
                           input_split_sizes=list(splits), group=group)
    return recv.reshape(W, T_r, Hs, d).permute(1, 0, 2, 3).reshape(T_r, W * Hs, d)


def head_slice(H: int, group=None) -> slice:
    """This rank's heads among H."""
    W, rank = _group_info(group)
    return slice(rank * (H // W), (rank + 1) * (H // W))


def _cuda_forward(q, k, v, sinks, cu, max_seqlen, causal, window, scale):
    from . import api
    return api.forward(q, k, v, sinks, cu, max_seqlen, causal=causal, window=window, scale=scale)


def _cuda_backward(q, k, v, sinks, cu, max_seqlen, o, lse, dout, causal, window, scale):
    from . import api
    return api.backward(q, k, v, sinks, cu, max_seqlen, o, lse, dout, causal=causal,
                        window=window, scale=scale)


class HeadSplitAttention:
    """Sink attention over a token-sharded packed batch by regrouping it by
    head with all-to-all (section "Sequence Parallelism with FlashAttention
    v3"). Every rank of ``group`` passes its contiguous slice of the packed
    tokens (``token_split`` sizes) with all heads, and the global cu_seqlens.

    ``forward`` returns this rank's slice of O; ``backward`` takes its slice of
    dO and returns its slices of dq, dk, dv, plus dL/dS_h of all Hq heads with
    only this rank's heads filled in (zero elsewhere): adding the ranks'
    vectors, as a gradient reduction over the group does, gives the full
    gradient, and ``gather_sink_grad`` assembles it directly.

    ``fwd_fn`` / ``bwd_fn`` run attention on the regrouped data; they default
    to the CUDA library and take (q, k, v, sinks, cu_seqlens, max_seqlen, o,
    lse, dout, causal, window, scale) as ``api.forward`` / ``api.backward`` do.
    """

    def __init__(self, cu_seqlens: torch.Tensor, max_seqlen: int, *, causal=True, window=0,
                 scale=None, group=None, fwd_fn: Optional[Callable] = None,
                 bwd_fn: Optional[Callable] = None):
        self.group = group
        self.W, self.rank = _group_info(group)
        self.cu = cu_seqlens
        self.max_seqlen = int(max_seqlen)
        self.total = int(cu_seqlens[-1])
        self.splits = token_split(self.total, self.W)
        self.causal, self.window, self.scale = causal, window, scale
        self.fwd_fn = fwd_fn or _cuda_forward
        self.bwd_fn = bwd_fn or _cuda_backward
        self._saved = None

    def forward(self, q, k, v, sinks):
        Hq, Hkv = q.shape[1], k.shape[1]
        if Hkv % self.W or Hq % Hkv:
            raise ValueError("Hkv must be a multiple of the group size and divide Hq")
        qh = tokens_to_heads(q, self.splits, self.group)
        kh = tokens_to_heads(k, self.splits, self.group)
        vh = tokens_to_heads(v, self.splits, self.group)
        sh = sinks[head_slice(Hq, self.group)].contiguous() if sinks is not None else None
        o, lse = self.fwd_fn(qh, kh, vh, sh, self.cu, self.max_seqlen, self.causal,
                             self.window, self.scale)
        self._saved = (qh, kh, vh, sh, o, lse, Hq)
        return heads_to_tokens(o, self.splits, self.group)

    def backward(self, dout):
        qh, kh, vh, sh, o, lse, Hq = self._saved
        doh = tokens_to_heads(dout, self.splits, self.group)
        dq, dk, dv, ds = self.bwd_fn(qh, kh, vh, sh, self.cu, self.max_seqlen, o, lse, doh,
                                     self.causal, self.window, self.scale)
        full = None
        if ds is not None:
            full = torch.zeros(Hq, dtype=ds.dtype, device=ds.device)
            full[head_slice(Hq, self.group)] = ds
        return (heads_to_tokens(dq, self.splits, self.group),
                heads_to_tokens(dk, self.splits, self.group),
                heads_to_tokens(dv, self.splits, self.group), full)


def gather_sink_grad(dsinks_local: torch.Tensor, group=None) -> torch.Tensor:
    """The full dL/dS_h from ``HeadSplitAttention.backward``'s per-rank
    vectors (each holds only its heads; the sum over ranks is the gradient)."""
    out = dsinks_local.clone()
    if dist.get_world_size(group) > 1:
        dist.all_reduce(out, op=dist.ReduceOp.SUM, group=group)
    return out
