"""Seeded synthetic inputs for sink attention.

This module only draws random tensors and packs sequence offsets; it holds
none of the attention arithmetic, so both the CUDA path and the fp64 oracle
can take their inputs from it.

The pages benchmark nothing at the kernel level: the model they train is a
20B-class MoE LLM (page "GPT-OSS Agentic RL Training: A Practical
Retrospective", section "Agentic RL and GPT-OSS") on GSM8K, Retool and
VerifyIf. None of that is available, so these tensors stand in for one
attention layer of such a model: 64 query heads over 8 key/value heads of
width 64, bf16 activations, fp32 sinks, and for the RL rollout case a packed
batch of sequences of uneven length (section "Scaling Memory Efficiency for
Long Contexts": contexts grow as environment feedback is appended).

Recipe (all drawn on the CPU with ``torch.Generator().manual_seed(seed)``,
in the order lengths -> q -> k -> v -> dO -> sinks; values drawn in fp32 and
rounded to bf16 with round-to-nearest-even):

  tiny         seed 1  B=1  T=128   Hq=4  Hkv=1 causal            q,k,v,dO ~ N(0,1)   S ~ U(-2,2)
  dense        seed 2  B=4  T=2048  Hq=64 Hkv=8 causal            N(0,1)              S ~ U(-2,2)
  window       seed 3  as dense, causal window of 128 keys        N(0,1)              S ~ U(-4,4)
  varlen       seed 4  32 sequences, L ~ randint[256, 8192]       N(0,1)              even heads S ~ U(-2,2),
                       (inclusive), Hq=64 Hkv=8 causal                                odd heads S = -30
  long         seed 5  B=1  T=32768 Hq=64 Hkv=8 causal            q,k ~ 2 N(0,1)      S ~ U(-10,10)
                                                                  v,dO ~ N(0,1)
  long_window  seed 5  as long, causal window of 128 keys
  dense_d128   seed 12 as dense at head_dim 128 (the head width of the
                       training log on page 4, the xxqk.cn post)           N(0,1)     S ~ U(-2,2)
"""

from __future__ import annotations

from dataclasses import dataclass, field

import torch

HEAD_DIM = 64


@dataclass
class Workload:
    name: str
    q: torch.Tensor          # bf16 [total, Hq, d]
    k: torch.Tensor          # bf16 [total, Hkv, d]
    v: torch.Tensor          # bf16 [total, Hkv, d]
    dout: torch.Tensor       # bf16 [total, Hq, d]
    sinks: torch.Tensor      # fp32 [Hq]
    cu_seqlens: torch.Tensor  # int32 [nseq + 1]
    causal: bool = True
    window: int = 0
    scale: float = HEAD_DIM ** -0.5
    meta: dict = field(default_factory=dict)

    @property
    def total(self) -> int:
        return int(self.cu_seqlens[-1])

    @property
    def nseq(self) -> int:
        return int(self.cu_seqlens.numel() - 1)

    @property
    def max_seqlen(self) -> int:
        lens = self.cu_seqlens[1:] - self.cu_seqlens[:-1]
        return int(lens.max()) if lens.numel() else 0

    @property
    def Hq(self) -> int:
        return int(self.q.shape[1])

    @property
    def Hkv(self) -> int:
        return int(self.k.shape[1])


def _offsets(lengths) -> torch.Tensor:
    cu = torch.zeros(len(lengths) + 1, dtype=torch.int32)
    if len(lengths):
        cu[1:] = torch.cumsum(torch.as_tensor(lengths, dtype=torch.int64), 0).to(torch.int32)
    return cu


def make(name: str, lengths, Hq: int, Hkv: int, *, seed: int, causal: bool = True,
         window: int = 0, qk_std: float = 1.0, sink_range=(-2.0, 2.0),
         odd_head_sink=None, d: int = HEAD_DIM, no_sink: bool = False) -> Workload:
    """Draw one workload. ``lengths`` may be a list of ints or a callable
    taking the generator and returning one (so lengths are drawn first)."""
    g = torch.Generator().manual_seed(seed)
    if callable(lengths):
        lengths = lengths(g)
    lengths = [int(x) for x in lengths]
    total = sum(lengths)

    def draw(h, std):
        return (torch.randn(total, h, d, generator=g, dtype=torch.float32) * std).to(torch.bfloat16)

    q = draw(Hq, qk_std)
    k = draw(Hkv, qk_std)
    v = draw(Hkv, 1.0)
    dout = draw(Hq, 1.0)
    lo, hi = sink_range
    sinks = torch.rand(Hq, generator=g, dtype=torch.float32) * (hi - lo) + lo
    if odd_head_sink is not None:
        sinks[1::2] = odd_head_sink
    meta = {"lengths": lengths, "seed": seed, "no_sink": no_sink}
    return Workload(name, q, k, v, dout, sinks, _offsets(lengths), causal, window,
                    d ** -0.5, meta)


def _varlen_lengths(g):
    return torch.randint(256, 8192 + 1, (32,), generator=g).tolist()


CONFIGS = {
    "tiny": dict(lengths=[128], Hq=4, Hkv=1, seed=1),
    "dense": dict(lengths=[2048] * 4, Hq=64, Hkv=8, seed=2),
    "window": dict(lengths=[2048] * 4, Hq=64, Hkv=8, seed=3, window=128, sink_range=(-4.0, 4.0)),
    "varlen": dict(lengths=_varlen_lengths, Hq=64, Hkv=8, seed=4, odd_head_sink=-30.0),
    "long": dict(lengths=[32768], Hq=64, Hkv=8, seed=5, qk_std=2.0, sink_range=(-10.0, 10.0)),
    "long_window": dict(lengths=[32768], Hq=64, Hkv=8, seed=5, qk_std=2.0,
                        sink_range=(-10.0, 10.0), window=128),
    "dense_d128": dict(lengths=[2048] * 4, Hq=64, Hkv=8, seed=12, d=128),
}

# One-line descriptions, used in reports.
DESCRIPTIONS = {
    "tiny": "B=1 T=128 Hq=4 Hkv=1 d=64 causal",
    "dense": "B=4 T=2048 Hq=64 Hkv=8 d=64 causal",
    "window": "B=4 T=2048 Hq=64 Hkv=8 d=64 causal window=128",
    "varlen": "32 packed seqs L~U[256,8192] Hq=64 Hkv=8 d=64 causal, odd-head sinks -30",
    "long": "B=1 T=32768 Hq=64 Hkv=8 d=64 causal, q,k~2N(0,1), S~U(-10,10)",
    "long_window": "B=1 T=32768 Hq=64 Hkv=8 d=64 causal window=128, q,k~2N(0,1)",
    "dense_d128": "B=4 T=2048 Hq=64 Hkv=8 d=128 causal",
}


def config(name: str) -> Workload:
    return make(name, **CONFIGS[name])


@dataclass
class DecodeWorkload:
    """One decode step: a query row per sequence over a paged KV cache.

    Cache slots that hold no key of any sequence (the tail of each sequence's
    last block, spare blocks) are NaN, so a kernel that reads them where it
    should not shows it in its output."""
    name: str
    q: torch.Tensor            # bf16 [nseq, Hq, d]
    k_cache: torch.Tensor      # bf16 [num_blocks, block_size, Hkv, d]
    v_cache: torch.Tensor      # bf16 [num_blocks, block_size, Hkv, d]
    block_table: torch.Tensor  # int32 [nseq, max_blocks], -1 past a sequence's blocks
    seqlens: torch.Tensor      # int32 [nseq]
    sinks: torch.Tensor        # fp32 [Hq]
    window: int = 0
    scale: float = HEAD_DIM ** -0.5
    meta: dict = field(default_factory=dict)

    @property
    def nseq(self) -> int:
        return int(self.seqlens.numel())

    @property
    def Hq(self) -> int:
        return int(self.q.shape[1])

    @property
    def Hkv(self) -> int:
        return int(self.k_cache.shape[2])

    @property
    def block_size(self) -> int:
        return int(self.k_cache.shape[1])


def make_decode(name: str, lengths, Hq: int, Hkv: int, block_size: int, *, seed: int,
                window: int = 0, qk_std: float = 1.0, sink_range=(-2.0, 2.0),
                odd_head_sink=None, spare_blocks: int = 3, extra_columns: int = 1,
                d: int = HEAD_DIM) -> DecodeWorkload:
    """Draw one decode step. Order: lengths -> q -> keys -> values -> sinks ->
    the permutation that places logical blocks in physical ones."""
    g = torch.Generator().manual_seed(seed)
    if callable(lengths):
        lengths = lengths(g)
    lengths = [int(x) for x in lengths]
    nseq, total = len(lengths), sum(lengths)
    nblk = [(L + block_size - 1) // block_size for L in lengths]
    num_blocks = sum(nblk) + spare_blocks
    max_blocks = max(nblk + [0]) + extra_columns
    q = (torch.randn(nseq, Hq, d, generator=g) * qk_std).to(torch.bfloat16)
    k_tok = (torch.randn(total, Hkv, d, generator=g) * qk_std).to(torch.bfloat16)
    v_tok = torch.randn(total, Hkv, d, generator=g).to(torch.bfloat16)
    lo, hi = sink_range
    sinks = torch.rand(Hq, generator=g, dtype=torch.float32) * (hi - lo) + lo
    if odd_head_sink is not None:
        sinks[1::2] = odd_head_sink
    perm = torch.randperm(num_blocks, generator=g)
    nan = float("nan")
    k_cache = torch.full((num_blocks, block_size, Hkv, d), nan, dtype=torch.bfloat16)
    v_cache = torch.full((num_blocks, block_size, Hkv, d), nan, dtype=torch.bfloat16)
    table = torch.full((nseq, max_blocks), -1, dtype=torch.int32)
    nxt, off = 0, 0
    for b, L in enumerate(lengths):
        for i in range(nblk[b]):
            pb = int(perm[nxt])
            nxt += 1
            table[b, i] = pb
            n = min(block_size, L - i * block_size)
            k_cache[pb, :n] = k_tok[off + i * block_size: off + i * block_size + n]
            v_cache[pb, :n] = v_tok[off + i * block_size: off + i * block_size + n]
        off += L
    meta = {"lengths": lengths, "seed": seed, "k_tokens": k_tok, "v_tokens": v_tok}
    return DecodeWorkload(name, q, k_cache, v_cache, table,
                          torch.tensor(lengths, dtype=torch.int32), sinks, window, d ** -0.5, meta)


def _decode_lengths(g):
    return torch.randint(256, 8192 + 1, (64,), generator=g).tolist()


DECODE_CONFIGS = {
    "decode": dict(lengths=_decode_lengths, Hq=64, Hkv=8, block_size=64, seed=6),
    "decode_window": dict(lengths=_decode_lengths, Hq=64, Hkv=8, block_size=64, seed=6,
                          window=128, sink_range=(-4.0, 4.0)),
    "decode_d128": dict(lengths=_decode_lengths, Hq=64, Hkv=8, block_size=64, seed=6, d=128),
}

DECODE_DESCRIPTIONS = {
    "decode": "64 seqs L~U[256,8192] Hq=64 Hkv=8 d=64, paged cache of 64-token blocks",
    "decode_window": "as decode, window=128",
    "decode_d128": "as decode at head_dim 128",
}


def decode_config(name: str) -> DecodeWorkload:
    return make_decode(name, **DECODE_CONFIGS[name])
