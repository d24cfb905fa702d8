"""The parity comparison sees a plausible mistake. The CUDA path's outputs on
one seeded case are compared, with the tolerances of every parity test,
against copies of the fp64 oracles into which one mistake has been planted
on the CPU (the lists in test_oracle_mutations.py: for training a dropped or
scaled sink, the sign of dS_h, a wrong GQA map, a window one key too wide,
dS without D, dk without the scale, dv from q, LSE without the maximum; for
decode also a window one key too narrow, no scale, the last key dropped, the
wrong slot in a cache block, K read as V). Every such copy must fail the
comparison, and the unchanged copy must pass it, so the parity tests are not
satisfied by outputs that are merely close to the method."""

import importlib.util
import os
import shutil
import sys

import numpy as np
import pytest

from attention_learnable_sinks_gb300.workloads import make

from parity import assert_dsinks, compare_full, dsink_condition, f64, run_cuda
from test_gpu_decode import compare as compare_decode
from test_gpu_decode import run_cuda as run_decode
from test_oracle_mutations import CPP, CPP_MUTANTS, DEC, DEC_MUTANTS, ROOT

pytestmark = pytest.mark.gpu


def _oracle_copy(tmp, tag, sites, fname=CPP):
    dst = os.path.join(tmp, tag, "oracle")
    shutil.copytree(os.path.join(ROOT, "oracle"), dst, ignore=shutil.ignore_patterns("_build", "__pycache__"))
    path = os.path.join(dst, fname)
    text = open(path).read()
    for a, b in sites:
        assert text.count(a) == 1, a
        text = text.replace(a, b)
    open(path, "w").write(text)
    name = f"oracle_{os.path.basename(tmp)}_{tag}"
    spec = importlib.util.spec_from_file_location(name, os.path.join(dst, "__init__.py"),
                                                  submodule_search_locations=[dst])
    mod = importlib.util.module_from_spec(spec)
    sys.modules[name] = mod  # so that its submodules (the decode oracle) import from the copy
    spec.loader.exec_module(mod)
    return mod


def _passes(w, got, mod):
    ref = mod.sinkattn(f64(w.q), f64(w.k), f64(w.v), w.sinks.numpy().astype(np.float64),
                       w.cu_seqlens.numpy(), causal=w.causal, window=w.window, scale=w.scale,
                       dout=f64(w.dout), want=("o", "lse", "dq", "dk", "dv", "dsinks"))
    try:
        compare_full(w, got, ref)
        cond = dsink_condition(w.sinks.numpy().astype(np.float64), ref["lse"], ref["o"], f64(w.dout))
        assert_dsinks(got["dsinks"], ref["dsinks"], cond)
    except AssertionError:
        return False
    return True


def test_parity_fails_against_every_planted_mistake(cuda_lib, tmp_path):
    w = make("discriminate", [300, 129, 64], 8, 2, seed=41, window=16)
    got = run_cuda(w)
    assert _passes(w, got, _oracle_copy(str(tmp_path), "unchanged", [])), \
        "the CUDA path must match an unchanged copy of the oracle"
    passed = []
    for i, (name, a, b) in enumerate(CPP_MUTANTS):
        sites = a if isinstance(a, list) else [(a, b)]
        if _passes(w, got, _oracle_copy(str(tmp_path), f"m{i}", sites)):
            passed.append(name)
    assert not passed, "parity passed against planted mistakes: " + ", ".join(passed)


def _decode_passes(w, got, mod):
    dec = importlib.import_module(mod.__name__ + ".decode")
    try:  # a mistake may break the oracle outright (mismatched shapes): that fails too
        ref = dec.decode(f64(w.q), f64(w.k_cache), f64(w.v_cache), w.block_table.numpy(),
                         w.seqlens.numpy(), w.sinks.numpy(), window=w.window, scale=w.scale)
    except ValueError:
        return False
    try:
        compare_decode(w, got, ref)
    except AssertionError:
        return False
    return True


def test_decode_parity_fails_against_every_planted_mistake(cuda_lib, tmp_path):
    from attention_learnable_sinks_gb300.workloads import make_decode
    w = make_decode("discriminate_decode", [1, 9, 130, 700, 2000], 8, 2, 16, seed=42, window=8)
    got = run_decode(w)
    assert _decode_passes(w, got, _oracle_copy(str(tmp_path), "unchanged", [], DEC)), \
        "the decode must match an unchanged copy of the decode oracle"
    passed = []
    for i, (name, a, b) in enumerate(DEC_MUTANTS):
        if _decode_passes(w, got, _oracle_copy(str(tmp_path), f"d{i}", [(a, b)], DEC)):
            passed.append(name)
    assert not passed, "decode parity passed against planted mistakes: " + ", ".join(passed)
