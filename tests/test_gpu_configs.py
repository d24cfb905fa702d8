"""CUDA path vs the fp64 oracle at the five workload configurations, at full
size, in the same launch configuration the benchmark times.

tiny, dense, window and long_window are compared element by element over
whole tensors, once with the atomic dq and once with the deterministic
backward (dq summed in a fixed order). varlen and long are too large for the oracle in full, so:
  * varlen: all outputs of one complete GQA group (8 query heads, kv head 0)
    on four whole sequences (shortest, longest and two others); dS_h of two
    heads (one U(-2,2), one -30) over all 32 sequences; |dS_h| tiny for
    every -30 head.
  * long (T = 32768, causal): a prefix of 1024 tokens is a self-contained
    problem under the causal mask (rows and keys there); the last 256 rows and
    keys are exact with the oracle restricted to them; dS_h of two heads over
    all rows.
"""

import numpy as np
import pytest

from attention_learnable_sinks_gb300.workloads import config

from parity import (assert_dsinks, compare_full, dsink_condition, run_cuda, run_oracle)

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("name", ["tiny", "dense", "window", "long_window"])
def test_config_full_tensor(cuda_lib, name):
    w = config(name)
    ref, *_ = run_oracle(w)
    cond = dsink_condition(w.sinks.numpy().astype(np.float64), ref["lse"], ref["o"], ref["_do"])
    for det in (False, True):  # atomic dq, then the fixed-order dq pass
        got = run_cuda(w, deterministic=det)
        errs = compare_full(w, got, ref)
        errs["dsinks"] = assert_dsinks(got["dsinks"], ref["dsinks"], cond)
        print(name, "deterministic" if det else "atomic", {k: f"{v:.2e}" for k, v in errs.items()})


def _dsinks_refs(w, heads):
    """dS_h over every sequence, for the given query heads (each as its own
    one-head problem with its kv head): (reference values, condition scales)."""
    import oracle
    from parity import f64
    G = w.Hq // w.Hkv
    refs, conds = [], []
    cu = w.cu_seqlens.numpy()
    for h in heads:
        r = oracle.sinkattn(f64(w.q[:, h:h + 1]), f64(w.k[:, h // G:h // G + 1]),
                            f64(w.v[:, h // G:h // G + 1]),
                            w.sinks.numpy().astype(np.float64)[h:h + 1], cu, causal=w.causal,
                            window=w.window, scale=w.scale, dout=f64(w.dout[:, h:h + 1]),
                            want=("o", "lse", "dsinks"))
        refs.append(r["dsinks"][0])
        conds.append(dsink_condition(w.sinks.numpy().astype(np.float64)[h:h + 1], r["lse"],
                                     r["o"], f64(w.dout[:, h:h + 1]))[0])
    return list(heads), np.array(refs), np.array(conds)


def _dsinks_check(got, refs):
    heads, ref, cond = refs
    return assert_dsinks(got["dsinks"][heads], ref, cond)


def test_varlen_sampled(cuda_lib):
    w = config("varlen")
    lens = np.diff(w.cu_seqlens.numpy())
    order = np.argsort(lens)
    seqs = sorted({int(order[0]), int(order[-1]), int(order[len(order) // 2]), 5})
    ref, tok, qh, kvh = run_oracle(w, kv_groups=[0], seqs=seqs)
    srefs = _dsinks_refs(w, [0, 1])
    for det in (False, True):  # atomic dq, then the fixed-order dq pass
        got = run_cuda(w, deterministic=det)
        errs = compare_full(w, got, ref, tok, qh, kvh)
        errs["dsinks"] = _dsinks_check(got, srefs)
        odd = got["dsinks"][1::2]
        assert np.max(np.abs(odd)) <= 1e-6, "sink gradient of the -30 heads should vanish"
        print("varlen", "deterministic" if det else "atomic",
              {k: f"{v:.2e}" for k, v in errs.items()}, "seqs", seqs, "lens", lens[seqs])


def test_long_sampled(cuda_lib):
    w = config("long")
    T = w.total
    # prefix: rows and keys [0, 1024) form a causal problem of their own ... but only
    # the rows' outputs (o, lse, dq) are complete there; keys also feed later rows.
    pre = run_oracle(w, kv_groups=[3], seqs=[0], prefix=1024, want=("o", "lse", "dq"))
    # suffix: rows and keys [T-256, T) with the oracle restricted to them
    first = T - 256
    suf = run_oracle(w, kv_groups=[5], seqs=[0], first_row=first)
    srefs = _dsinks_refs(w, [0, 41])
    for det in (False, True):
        got = run_cuda(w, deterministic=det)
        ref, tok, qh, kvh = pre
        errs = compare_full(w, got, ref, tok, qh, kvh)
        ref, tok, qh, kvh = suf
        errs.update({k + "_suffix": v for k, v in
                     compare_full(w, got, ref, tok, qh, kvh, rows=slice(first, T),
                                  keys=slice(first, T)).items()})
        errs["dsinks"] = _dsinks_check(got, srefs)
        print("long", "deterministic" if det else "atomic", {k: f"{v:.2e}" for k, v in errs.items()})
