"""Torch-facing entry points: ``forward``, ``backward`` and the autograd op
``sink_attention``. PyTorch supplies device memory and the stream; the work
is done by libsinkattn.so through its C ABI (argument marshalling only).
"""

from __future__ import annotations

import ctypes
from typing import Optional, Sequence

import torch

from . import _binding
from ._binding import BwdParams, DecodeParams, FwdParams, check

HEAD_DIM = 64               # the head dim of decode, and the default
HEAD_DIMS = (64, 128)       # head dims of forward and backward


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _stream_ptr(device) -> int:
    return torch.cuda.current_stream(device).cuda_stream


def _events(evs) -> Sequence[Optional[int]]:
    if evs is None:
        return (None, None)
    out = []
    for e in evs:
        h = e.cuda_event if e is not None else 0
        out.append(h or None)
    return out


def _check_tokens(name: str, t: torch.Tensor, head_dim: int):
    if t.dtype != torch.bfloat16 or not t.is_cuda or t.dim() != 3:
        raise ValueError(f"{name} must be a bf16 CUDA tensor [total, heads, head_dim]")
    if t.shape[2] != head_dim or t.stride(2) != 1 or t.stride(1) != head_dim:
        raise ValueError(f"{name}: must be [total, heads, {head_dim}] with heads and features "
                         f"contiguous (strides (*, {head_dim}, 1))")


def _fill_fwd(p: FwdParams, q, k, v, sinks, cu_seqlens, max_seqlen, causal, window, scale, o, lse):
    total, Hq, d = q.shape
    p.q, p.k, p.v = _ptr(q), _ptr(k), _ptr(v)
    p.sinks = _ptr(sinks)
    p.cu_seqlens = _ptr(cu_seqlens)
    p.o, p.lse = _ptr(o), _ptr(lse)
    p.q_row_stride, p.k_row_stride, p.v_row_stride = q.stride(0), k.stride(0), v.stride(0)
    p.nseq = cu_seqlens.numel() - 1
    p.total = total
    p.max_seqlen = int(max_seqlen)
    p.Hq, p.Hkv, p.head_dim = Hq, k.shape[1], d
    p.causal = 1 if causal else 0
    p.window = int(window)
    p.softmax_scale = float(scale) if scale is not None else 0.0


def _validate_inputs(q, k, v, sinks, cu_seqlens):
    if q.dim() != 3 or q.shape[2] not in HEAD_DIMS:
        raise ValueError("q must be [total, Hq, head_dim] with head_dim 64 or 128")
    d = q.shape[2]
    _check_tokens("q", q, d)
    _check_tokens("k", k, d)
    _check_tokens("v", v, d)
    if k.shape != v.shape or k.shape[0] != q.shape[0]:
        raise ValueError("k and v must be [total, Hkv, head_dim] with the same total and head_dim as q")
    if sinks is not None and (sinks.dtype != torch.float32 or not sinks.is_cuda or
                              sinks.shape != (q.shape[1],) or not sinks.is_contiguous()):
        raise ValueError("sinks must be a contiguous fp32 CUDA tensor [Hq]")
    if cu_seqlens.dtype != torch.int32 or not cu_seqlens.is_cuda or cu_seqlens.dim() != 1:
        raise ValueError("cu_seqlens must be an int32 CUDA tensor [nseq + 1]")


def forward(q, k, v, sinks, cu_seqlens, max_seqlen, *, causal=True, window=0, scale=None,
            out=None, lse=None, workspace=None, timing_events=None, bwd_workspace=None):
    """O [total, Hq, d] bf16 and LSE [Hq, total] fp32 (natural log), d = 64 or
    128. With ``bwd_workspace`` (the workspace the backward of this same
    problem will use; head_dim 64) the forward also prepares it: it clears the
    backward's dq accumulator and builds its key-tile list; pass
    ``workspace_cleared=True`` to that backward. At head_dim 128 it is not
    used."""
    _validate_inputs(q, k, v, sinks, cu_seqlens)
    L = _binding.lib()
    total, Hq, d = q.shape
    nseq = cu_seqlens.numel() - 1
    o = out if out is not None else torch.empty(total, Hq, d, dtype=torch.bfloat16, device=q.device)
    lse = lse if lse is not None else torch.empty(Hq, total, dtype=torch.float32, device=q.device)
    nbytes = L.sinkattn_fwd_workspace_size(nseq, total, Hq, k.shape[1], d)
    if workspace is None:
        workspace = torch.empty(max(nbytes, 1), dtype=torch.uint8, device=q.device)
    p = FwdParams()
    _fill_fwd(p, q, k, v, sinks, cu_seqlens, max_seqlen, causal, window, scale, o, lse)
    p.workspace, p.workspace_bytes = _ptr(workspace), workspace.numel()
    p.timing_events[0], p.timing_events[1] = _events(timing_events)
    if bwd_workspace is not None:
        p.bwd_workspace, p.bwd_workspace_bytes = _ptr(bwd_workspace), bwd_workspace.numel()
    check(L.sinkattn_fwd(ctypes.byref(p), _stream_ptr(q.device)), "sinkattn_fwd")
    return o, lse


def backward(q, k, v, sinks, cu_seqlens, max_seqlen, o, lse, dout, *, causal=True, window=0,
             scale=None, dq=None, dk=None, dv=None, dsinks=None, workspace=None,
             timing_events=None, accumulate_dsinks=False, deterministic=False,
             timing_events_dq=None, workspace_cleared=False):
    """dq, dk, dv (bf16, shaped like q, k, v but contiguous) and dsinks [Hq]
    fp32 (None when ``sinks`` is None). With ``accumulate_dsinks`` the sink
    gradient is added to the given ``dsinks`` instead of overwriting it. With
    ``deterministic`` dq is summed in a fixed order by a second,
    query-stationary pass, so every output is bit-identical from run to run;
    ``timing_events_dq`` (two CUDA events) are recorded around that pass.
    At head_dim 128 the backward always works this way.
    ``workspace_cleared``: the forward of this same problem was given this
    ``workspace`` as its ``bwd_workspace`` and cleared the dq accumulator in
    it (nothing may have written to it since), so the backward skips that."""
    _validate_inputs(q, k, v, sinks, cu_seqlens)
    for name, t in (("o", o), ("dout", dout)):
        _check_tokens(name, t, q.shape[2])
        if not t.is_contiguous() or t.shape != q.shape:
            raise ValueError(f"{name} must be contiguous and shaped like q")
    L = _binding.lib()
    total, Hq, d = q.shape
    Hkv = k.shape[1]
    nseq = cu_seqlens.numel() - 1
    dq = dq if dq is not None else torch.empty(total, Hq, d, dtype=torch.bfloat16, device=q.device)
    dk = dk if dk is not None else torch.empty(total, Hkv, d, dtype=torch.bfloat16, device=q.device)
    dv = dv if dv is not None else torch.empty(total, Hkv, d, dtype=torch.bfloat16, device=q.device)
    if sinks is not None and dsinks is None:
        dsinks = torch.empty(Hq, dtype=torch.float32, device=q.device)
    if workspace is None:  # sized for the mode: the deterministic backward has no dq accumulator
        nbytes = L.sinkattn_bwd_workspace_size_mode(nseq, total, Hq, Hkv, d, 1 if deterministic else 0)
        workspace = torch.empty(max(nbytes, 1), dtype=torch.uint8, device=q.device)
    p = BwdParams()
    _fill_fwd(p.fwd, q, k, v, sinks, cu_seqlens, max_seqlen, causal, window, scale, o, lse)
    p.dout, p.dq, p.dk, p.dv = _ptr(dout), _ptr(dq), _ptr(dk), _ptr(dv)
    p.dsinks = _ptr(dsinks)
    p.workspace, p.workspace_bytes = _ptr(workspace), workspace.numel()
    p.timing_events[0], p.timing_events[1] = _events(timing_events)
    if accumulate_dsinks and dsinks is None:
        raise ValueError("accumulate_dsinks needs a dsinks tensor to add to")
    p.accumulate_dsinks = 1 if accumulate_dsinks else 0
    p.deterministic = 1 if deterministic else 0
    p.timing_events_dq[0], p.timing_events_dq[1] = _events(timing_events_dq)
    p.workspace_cleared = 1 if workspace_cleared else 0
    check(L.sinkattn_bwd(ctypes.byref(p), _stream_ptr(q.device)), "sinkattn_bwd")
    return dq, dk, dv, dsinks


def decode(q, k_cache, v_cache, block_table, seqlens, sinks=None, *, window=0, scale=None,
           num_splits=0, out=None, lse=None, workspace=None, exact=False):
    """One query row per sequence against a paged KV cache.

    q [nseq, Hq, d] bf16; k_cache, v_cache [num_blocks, block_size, Hkv, d]
    bf16; block_table [nseq, max_blocks] int32; seqlens [nseq] int32 (keys per
    sequence, the new token's included). Returns o [nseq, Hq, d] bf16 and
    lse [Hq, nseq] fp32: the last row of ``forward`` over each sequence. With
    ``exact`` each row is computed exactly as ``forward`` computes that last
    row, so the two agree bit for bit (num_splits is then ignored). d is 64
    or 128."""
    for name, t in (("q", q), ("k_cache", k_cache), ("v_cache", v_cache)):
        if t.dtype != torch.bfloat16 or not t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous bf16 CUDA tensor")
    if q.dim() != 3 or q.shape[2] not in HEAD_DIMS:
        raise ValueError(f"q must be [nseq, Hq, d] with d in {HEAD_DIMS}")
    if k_cache.dim() != 4 or k_cache.shape != v_cache.shape or k_cache.shape[3] != q.shape[2]:
        raise ValueError("k_cache and v_cache must both be [num_blocks, block_size, Hkv, d]")
    for name, t in (("block_table", block_table), ("seqlens", seqlens)):
        if t.dtype != torch.int32 or not t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous int32 CUDA tensor")
    nseq, Hq, d = q.shape
    if block_table.dim() != 2 or block_table.shape[0] != nseq or seqlens.shape != (nseq,):
        raise ValueError("block_table must be [nseq, max_blocks] and seqlens [nseq]")
    if sinks is not None and (sinks.dtype != torch.float32 or not sinks.is_cuda or
                              sinks.shape != (Hq,) or not sinks.is_contiguous()):
        raise ValueError("sinks must be a contiguous fp32 CUDA tensor [Hq]")
    L = _binding.lib()
    o = out if out is not None else torch.empty(nseq, Hq, d, dtype=torch.bfloat16, device=q.device)
    lse = lse if lse is not None else torch.empty(Hq, nseq, dtype=torch.float32, device=q.device)
    if workspace is None:
        nbytes = 256 if exact else L.sinkattn_decode_workspace_size_d(
            nseq, Hq, num_splits if num_splits > 0 else 64, d)
        workspace = torch.empty(max(nbytes, 1), dtype=torch.uint8, device=q.device)
    p = DecodeParams()
    p.q, p.k_cache, p.v_cache = _ptr(q), _ptr(k_cache), _ptr(v_cache)
    p.block_table, p.seqlens, p.sinks = _ptr(block_table), _ptr(seqlens), _ptr(sinks)
    p.o, p.lse = _ptr(o), _ptr(lse)
    p.workspace, p.workspace_bytes = _ptr(workspace), workspace.numel()
    p.nseq, p.num_blocks, p.block_size = nseq, k_cache.shape[0], k_cache.shape[1]
    p.max_blocks_per_seq = block_table.shape[1]
    p.Hq, p.Hkv, p.head_dim = Hq, k_cache.shape[2], d
    p.window = int(window)
    p.num_splits = int(num_splits)
    p.softmax_scale = float(scale) if scale is not None else 0.0
    if exact:
        check(L.sinkattn_decode_exact(ctypes.byref(p), _stream_ptr(q.device)), "sinkattn_decode_exact")
    else:
        check(L.sinkattn_decode(ctypes.byref(p), _stream_ptr(q.device)), "sinkattn_decode")
    return o, lse


def workspace_bytes(kind: str, nseq: int, total: int, Hq: int, Hkv: int,
                    deterministic: bool = False, head_dim: int = HEAD_DIM) -> int:
    """Workspace bytes of the forward ("fwd") or of the backward ("bwd") in the
    given mode (the deterministic backward, which head_dim 128 always uses,
    needs no fp32 dq accumulator)."""
    L = _binding.lib()
    if kind == "fwd":
        return int(L.sinkattn_fwd_workspace_size(nseq, total, Hq, Hkv, head_dim))
    return int(L.sinkattn_bwd_workspace_size_mode(nseq, total, Hq, Hkv, head_dim,
                                                  1 if deterministic else 0))


class _SinkAttention(torch.autograd.Function):
    @staticmethod
    def forward(ctx, q, k, v, sinks, cu_seqlens, max_seqlen, causal, window, scale, deterministic):
        o, lse = forward(q, k, v, sinks, cu_seqlens, max_seqlen, causal=causal, window=window,
                         scale=scale)
        ctx.save_for_backward(q, k, v, sinks, cu_seqlens, o, lse)
        ctx.args = (max_seqlen, causal, window, scale, deterministic)
        return o

    @staticmethod
    def backward(ctx, do):
        q, k, v, sinks, cu_seqlens, o, lse = ctx.saved_tensors
        max_seqlen, causal, window, scale, deterministic = ctx.args
        dq, dk, dv, ds = backward(q, k, v, sinks, cu_seqlens, max_seqlen, o, lse,
                                  do.contiguous(), causal=causal, window=window, scale=scale,
                                  deterministic=deterministic)
        return dq, dk, dv, ds, None, None, None, None, None, None


def sink_attention(q, k, v, sinks=None, cu_seqlens=None, max_seqlen=None, *, causal=True,
                   window=0, scale=None, deterministic=False):
    """Attention with one learnable sink logit per query head.

    q [total, Hq, d], k/v [total, Hkv, d] bf16 (d = 64 or 128) with
    cu_seqlens (int32 [nseq+1]) for packed variable-length batches, or
    q [B, T, Hq, d], k/v [B, T, Hkv, d] for a dense batch. sinks: fp32 [Hq]
    or None.
    Returns O shaped like q. Differentiable in q, k, v and sinks; with
    ``deterministic`` the backward is bit-identical from run to run.
    """
    batched = q.dim() == 4
    if batched:
        B, T = q.shape[:2]
        q, k, v = (x.reshape(B * T, *x.shape[2:]) for x in (q, k, v))
        if cu_seqlens is None:
            cu_seqlens = torch.arange(0, (B + 1) * T, T, dtype=torch.int32, device=q.device)
            max_seqlen = T
    if cu_seqlens is None:
        cu_seqlens = torch.tensor([0, q.shape[0]], dtype=torch.int32, device=q.device)
        max_seqlen = q.shape[0]
    if max_seqlen is None:
        lens = cu_seqlens[1:] - cu_seqlens[:-1]
        max_seqlen = int(lens.max().item()) if lens.numel() else 0
    o = _SinkAttention.apply(q, k, v, sinks, cu_seqlens, max_seqlen, causal, window, scale,
                             deterministic)
    return o.reshape(B, T, *o.shape[1:]) if batched else o


class SinkAttention(torch.nn.Module):
    """The sink-attention layer with its sinks as a parameter: one fp32 logit
    per query head (``init`` everywhere at the start), trained like any
    other weight. ``forward(q, k, v, cu_seqlens=None, max_seqlen=None)``
    takes the shapes ``sink_attention`` takes and returns O."""

    def __init__(self, num_heads: int, *, causal: bool = True, window: int = 0, scale=None,
                 deterministic: bool = False, init: float = 0.0, device=None):
        super().__init__()
        self.sinks = torch.nn.Parameter(torch.full((num_heads,), float(init), dtype=torch.float32,
                                                   device=device))
        self.causal, self.window, self.scale = causal, window, scale
        self.deterministic = deterministic

    def forward(self, q, k, v, cu_seqlens=None, max_seqlen=None):
        return sink_attention(q, k, v, self.sinks, cu_seqlens, max_seqlen, causal=self.causal,
                              window=self.window, scale=self.scale, deterministic=self.deterministic)

    def extra_repr(self) -> str:
        return (f"num_heads={self.sinks.numel()}, causal={self.causal}, window={self.window}, "
                f"deterministic={self.deterministic}")


def _split_sequences(lens, causal: bool, window: int, groups: int):
    """Boundaries (sequence indices) of up to ``groups`` runs of consecutive
    sequences with about equal attention cost (allowed pairs)."""
    def cost(L):
        if not causal:
            return L * L
        if window > 0 and window < L:
            return window * (window + 1) // 2 + (L - window) * window
        return L * (L + 1) // 2
    costs = [cost(int(L)) for L in lens]
    total = sum(costs)
    groups = max(1, min(groups, len(costs)))
    bounds, acc, g = [0], 0, 1
    for i, c in enumerate(costs):
        acc += c
        if g < groups and acc >= total * g / groups and i + 1 < len(costs):
            bounds.append(i + 1)
            g += 1
    bounds.append(len(costs))
    return bounds


class HostPipeline:
    """Forward + backward of a packed batch held in pinned host memory.

    The batch is split into groups of whole sequences. The host-to-device
    copies of one group, the kernels of another and the device-to-host copies
    of a third run at the same time on three streams; the sink gradient is
    accumulated over the groups by the backward itself. Results equal one
    ``forward`` + ``backward`` over the whole batch (dS_h up to the order of
    its float additions). Device buffers, workspaces and streams are made
    once, for one batch shape (``cu_seqlens``, heads). ``deterministic``
    selects the backward whose dq is summed in a fixed order.
    """

    def __init__(self, cu_seqlens, Hq: int, Hkv: int, *, causal=True, window=0, scale=None,
                 groups: int = 2, device=None, deterministic=False, head_dim: int = HEAD_DIM):
        device = torch.device(device if device is not None else "cuda")
        cu = [int(x) for x in cu_seqlens.tolist()]
        lens = [b - a for a, b in zip(cu[:-1], cu[1:])]
        self.bounds = _split_sequences(lens, causal, window, groups)
        self.causal, self.window, self.scale = causal, window, scale
        self.deterministic = deterministic
        self.Hq, self.Hkv, self.total = Hq, Hkv, cu[-1]
        self.device = device
        self.head_dim = d = head_dim
        bf = dict(dtype=torch.bfloat16, device=device)
        self.q = torch.empty(self.total, Hq, d, **bf)
        self.k = torch.empty(self.total, Hkv, d, **bf)
        self.v = torch.empty(self.total, Hkv, d, **bf)
        self.dout = torch.empty(self.total, Hq, d, **bf)
        self.o = torch.empty_like(self.q)
        self.dq = torch.empty_like(self.q)
        self.dk = torch.empty_like(self.k)
        self.dv = torch.empty_like(self.v)
        self.sinks = torch.empty(Hq, dtype=torch.float32, device=device)
        self.dsinks = torch.empty(Hq, dtype=torch.float32, device=device)
        self.groups = []
        fw = bw = 1
        for a, b in zip(self.bounds[:-1], self.bounds[1:]):
            t0, t1 = cu[a], cu[b]
            local = torch.tensor([x - t0 for x in cu[a:b + 1]], dtype=torch.int32)
            self.groups.append({
                "t0": t0, "t1": t1, "nseq": b - a, "max_seqlen": max(lens[a:b]) if b > a else 0,
                "cu_host": local.pin_memory(),
                "cu": torch.empty(b - a + 1, dtype=torch.int32, device=device),
                "lse": torch.empty(Hq, t1 - t0, dtype=torch.float32, device=device),
                "qkv": torch.cuda.Event(), "do": torch.cuda.Event(),
                "fwd": torch.cuda.Event(), "bwd": torch.cuda.Event(),
            })
            fw = max(fw, workspace_bytes("fwd", b - a, t1 - t0, Hq, Hkv, head_dim=d))
            bw = max(bw, workspace_bytes("bwd", b - a, t1 - t0, Hq, Hkv, head_dim=d))
        self.ws_f = torch.empty(fw, dtype=torch.uint8, device=device)
        self.ws_b = torch.empty(bw, dtype=torch.uint8, device=device)
        self.s_in = torch.cuda.Stream(device)
        self.s_run = torch.cuda.Stream(device)
        self.s_out = torch.cuda.Stream(device)

    def h2d_bytes(self) -> int:
        per_tok = (2 * self.Hq + 2 * self.Hkv) * self.head_dim * 2
        return self.total * per_tok + 4 * self.Hq + sum(4 * g["cu"].numel() for g in self.groups)

    def d2h_bytes(self) -> int:
        return self.total * (2 * self.Hq + 2 * self.Hkv) * self.head_dim * 2 + 4 * self.Hq

    def run(self, hq, hk, hv, hdout, hsinks, ho, hdq, hdk, hdv, hdsinks):
        """Enqueue the whole batch: host inputs (pinned, shaped like the device
        buffers) in, host outputs out. Ordered after the current stream's work;
        the current stream waits for the last copy, so synchronising it (or an
        event recorded on it) covers everything."""
        cur = torch.cuda.current_stream(self.device)
        # inputs: a group's q / k / v first (the forward needs only them), then dO
        self.s_in.wait_stream(cur)
        with torch.cuda.stream(self.s_in):
            self.sinks.copy_(hsinks, non_blocking=True)
            for g in self.groups:
                sl = slice(g["t0"], g["t1"])
                g["cu"].copy_(g["cu_host"], non_blocking=True)
                for dst, src in ((self.q, hq), (self.k, hk), (self.v, hv)):
                    dst[sl].copy_(src[sl], non_blocking=True)
                g["qkv"].record(self.s_in)
                self.dout[sl].copy_(hdout[sl], non_blocking=True)
                g["do"].record(self.s_in)
        self.s_run.wait_stream(cur)
        with torch.cuda.stream(self.s_run):
            for i, g in enumerate(self.groups):
                sl = slice(g["t0"], g["t1"])
                q, k, v, do = self.q[sl], self.k[sl], self.v[sl], self.dout[sl]
                o = self.o[sl]
                self.s_run.wait_event(g["qkv"])
                forward(q, k, v, self.sinks, g["cu"], g["max_seqlen"], causal=self.causal,
                        window=self.window, scale=self.scale, out=o, lse=g["lse"],
                        workspace=self.ws_f)
                g["fwd"].record(self.s_run)
                self.s_run.wait_event(g["do"])
                backward(q, k, v, self.sinks, g["cu"], g["max_seqlen"], o, g["lse"], do,
                         causal=self.causal, window=self.window, scale=self.scale,
                         dq=self.dq[sl], dk=self.dk[sl], dv=self.dv[sl], dsinks=self.dsinks,
                         workspace=self.ws_b, accumulate_dsinks=i > 0,
                         deterministic=self.deterministic)
                g["bwd"].record(self.s_run)
        # outputs: a group's o as soon as its forward is done, then its gradients
        self.s_out.wait_stream(cur)
        with torch.cuda.stream(self.s_out):
            for g in self.groups:
                sl = slice(g["t0"], g["t1"])
                self.s_out.wait_event(g["fwd"])
                ho[sl].copy_(self.o[sl], non_blocking=True)
                self.s_out.wait_event(g["bwd"])
                for dst, src in ((hdq, self.dq), (hdk, self.dk), (hdv, self.dv)):
                    dst[sl].copy_(src[sl], non_blocking=True)
            hdsinks.copy_(self.dsinks, non_blocking=True)
        cur.wait_stream(self.s_out)
        return ho, hdq, hdk, hdv, hdsinks
