"""Helpers for comparing the CUDA path with the fp64 oracle.

Tolerances. O, dq, dk, dv: relative L2 error over the compared tensor
<= 1e-2 (bf16 inputs and outputs, fp32 accumulation). dS_h: relative L2 over
the compared heads <= 1e-2, and per head |err| <= 1e-2 * max(|ref|, C_h) with
C_h = sum_{b,i} |p_sink * D| (a sum with cancellation is ill-conditioned; C_h
is its condition scale). LSE: max |err| <= 1e-3 (fp32 statistics of bf16
scores; the bf16 rounding of O does not enter it).
"""

from __future__ import annotations

import numpy as np
import torch

import oracle
from attention_learnable_sinks_gb300 import _binding, api
from attention_learnable_sinks_gb300.workloads import Workload

TOL_REL = 1e-2
TOL_LSE = 1e-3
ALL = ("o", "lse", "dq", "dk", "dv", "dsinks")


def f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


# Guard regions around every output and workspace the library writes. A
# store outside its tensor (a ragged tail tile, a wrong stride) lands in a
# guard and changes it; the bodies start as the same pattern, so an element
# the library never writes stays NaN and fails the comparison.
GUARD_BYTES = 4096
_CANARY = {torch.bfloat16: (torch.int16, 0x7FA5),     # a bf16 NaN no kernel produces
           torch.float32: (torch.int32, 0x7FC0A5A5),  # an fp32 NaN payload
           torch.uint8: (torch.uint8, 0xA5)}


class Guarded:
    """A device tensor of ``shape`` inside a larger buffer whose head and tail
    (GUARD_BYTES each) hold a canary bit pattern, as does the body at first."""

    def __init__(self, shape, dtype, device):
        ity, pat = _CANARY[dtype]
        esz = torch.empty(0, dtype=dtype).element_size()
        self.n = int(np.prod(shape)) if len(shape) else 1
        self.pad = GUARD_BYTES // esz
        self.buf = torch.empty(self.n + 2 * self.pad, dtype=dtype, device=device)
        self.bits = self.buf.view(ity)
        self.bits.fill_(pat)
        self.pattern = pat
        self.t = self.buf[self.pad:self.pad + self.n].view(shape)

    def check(self, name):
        head = self.bits[:self.pad]
        tail = self.bits[self.pad + self.n:]
        pat = self.pattern
        assert bool((head == pat).all()), f"{name}: guard region before the tensor was overwritten"
        assert bool((tail == pat).all()), f"{name}: guard region after the tensor was overwritten"


def run_cuda(w: Workload, device="cuda", q_view=None, k_view=None, v_view=None, scale=None,
             sinks=True, deterministic=False):
    """One forward + backward through the C ABI; returns fp64 host arrays.
    ``deterministic`` selects the backward whose dq is summed in a fixed order.
    Every output and both workspaces sit between guard regions that must come
    back unchanged."""
    q = q_view if q_view is not None else w.q.to(device)
    k = k_view if k_view is not None else w.k.to(device)
    v = v_view if v_view is not None else w.v.to(device)
    s = w.sinks.to(device) if sinks else None
    cu = w.cu_seqlens.to(device)
    do = w.dout.to(device)
    sc = w.scale if scale is None else scale
    total, Hq, Hkv, d = w.total, w.Hq, w.Hkv, w.q.shape[2]
    nseq = w.nseq
    bf, f32 = torch.bfloat16, torch.float32
    g = {"o": Guarded((total, Hq, d), bf, device), "lse": Guarded((Hq, total), f32, device),
         "dq": Guarded((total, Hq, d), bf, device), "dk": Guarded((total, Hkv, d), bf, device),
         "dv": Guarded((total, Hkv, d), bf, device), "dsinks": Guarded((Hq,), f32, device),
         "ws_fwd": Guarded((max(api.workspace_bytes("fwd", nseq, total, Hq, Hkv, head_dim=d), 1),),
                           torch.uint8, device),
         "ws_bwd": Guarded((max(api.workspace_bytes("bwd", nseq, total, Hq, Hkv, head_dim=d), 1),),
                           torch.uint8, device)}
    o, lse = api.forward(q, k, v, s, cu, max(w.max_seqlen, 1), causal=w.causal, window=w.window,
                         scale=sc, out=g["o"].t, lse=g["lse"].t, workspace=g["ws_fwd"].t)
    dq, dk, dv, ds = api.backward(q, k, v, s, cu, max(w.max_seqlen, 1), o, lse, do,
                                  causal=w.causal, window=w.window, scale=sc,
                                  dq=g["dq"].t, dk=g["dk"].t, dv=g["dv"].t,
                                  dsinks=g["dsinks"].t if sinks else None,
                                  workspace=g["ws_bwd"].t, deterministic=deterministic)
    torch.cuda.synchronize()
    err = _binding.device_error(reset=True)
    assert err == 0, f"device error word {err}"
    for name, gt in g.items():
        if name == "dsinks" and not sinks:
            continue
        gt.check(name)
    out = {"o": f64(o), "lse": f64(lse), "dq": f64(dq), "dk": f64(dk), "dv": f64(dv)}
    out["dsinks"] = f64(ds) if ds is not None else np.zeros(w.Hq)
    return out


def token_index(cu: np.ndarray, seqs, first_row=0, last_rows=None):
    idx = []
    for b in seqs:
        a, e = int(cu[b]), int(cu[b + 1])
        lo = a + first_row
        hi = e if last_rows is None else min(e, a + last_rows)
        idx.append(np.arange(lo, hi))
    return np.concatenate(idx) if idx else np.zeros(0, dtype=np.int64)


def run_oracle(w: Workload, kv_groups=None, seqs=None, want=ALL, first_row=0, prefix=None,
               sinks=True, scale=None):
    """The oracle on a selection of complete GQA groups and whole sequences
    (optionally only their first ``prefix`` tokens, which a causal mask makes
    self-contained). Returns (results, tokens, q_heads, kv_heads)."""
    cu = w.cu_seqlens.numpy().astype(np.int64)
    nseq = len(cu) - 1
    G = w.Hq // w.Hkv
    kv_heads = np.arange(w.Hkv) if kv_groups is None else np.asarray(kv_groups)
    q_heads = np.concatenate([np.arange(g * G, (g + 1) * G) for g in kv_heads])
    seqs = list(range(nseq)) if seqs is None else list(seqs)
    if prefix is not None:
        assert w.causal
    tok = token_index(cu, seqs, 0, prefix)
    lens = [min(int(cu[b + 1] - cu[b]), prefix) if prefix is not None else int(cu[b + 1] - cu[b])
            for b in seqs]
    sub_cu = np.zeros(len(seqs) + 1, dtype=np.int32)
    sub_cu[1:] = np.cumsum(lens)
    q = f64(w.q[tok][:, q_heads])
    k = f64(w.k[tok][:, kv_heads])
    v = f64(w.v[tok][:, kv_heads])
    do = f64(w.dout[tok][:, q_heads])
    s = w.sinks.numpy().astype(np.float64)[q_heads] if sinks else None
    res = oracle.sinkattn(q, k, v, s, sub_cu, causal=w.causal, window=w.window,
                          scale=w.scale if scale is None else scale, dout=do, want=want,
                          first_row=first_row)
    res["_cu"] = sub_cu
    res["_do"] = do
    return res, tok, q_heads, kv_heads


def rel_l2(got, ref):
    den = float(np.linalg.norm(ref))
    num = float(np.linalg.norm(got - ref))
    return num / den if den > 0 else num


def assert_close(name, got, ref, tol=TOL_REL):
    e = rel_l2(got, ref)
    assert e <= tol, f"{name}: relative L2 error {e:.3e} > {tol}"
    return e


def assert_lse(got, ref):
    e = float(np.max(np.abs(got - ref))) if ref.size else 0.0
    assert e <= TOL_LSE, f"lse: max abs error {e:.3e} > {TOL_LSE}"
    return e


def dsink_condition(sinks, lse, o, do):
    """C_h = sum_{b,i} |exp(S_h - LSE_i) * (dO_i . O_i)| from oracle O/LSE."""
    p_sink = np.exp(sinks[:, None] - lse)                   # [H, tokens]
    D = np.einsum("thd,thd->ht", do, o)
    return np.abs(p_sink * D).sum(1)


def assert_dsinks(got, ref, cond):
    e = rel_l2(got, ref)
    assert e <= TOL_REL, f"dsinks: relative L2 error {e:.3e} > {TOL_REL}"
    bound = TOL_REL * np.maximum(np.abs(ref), cond)
    bad = np.abs(got - ref) > bound
    assert not bad.any(), f"dsinks per-head error above bound at heads {np.nonzero(bad)[0]}"
    return e


def compare_full(w: Workload, got, ref, tok=None, qh=None, kvh=None, rows=None, keys=None):
    """Compare every output on the selected tokens / heads. ``rows`` / ``keys``
    restrict row outputs (o, lse, dq) and key outputs (dk, dv) to positions
    within the selection."""
    tok = np.arange(w.total) if tok is None else tok
    qh = np.arange(w.Hq) if qh is None else qh
    kvh = np.arange(w.Hkv) if kvh is None else kvh
    rsel = slice(None) if rows is None else rows
    ksel = slice(None) if keys is None else keys
    errs = {}
    errs["o"] = assert_close("o", got["o"][tok][:, qh][rsel], ref["o"][rsel])
    errs["lse"] = assert_lse(got["lse"][qh][:, tok][:, rsel], ref["lse"][:, rsel])
    errs["dq"] = assert_close("dq", got["dq"][tok][:, qh][rsel], ref["dq"][rsel])
    if "dk" in ref:
        errs["dk"] = assert_close("dk", got["dk"][tok][:, kvh][ksel], ref["dk"][ksel])
        errs["dv"] = assert_close("dv", got["dv"][tok][:, kvh][ksel], ref["dv"][ksel])
    return errs
