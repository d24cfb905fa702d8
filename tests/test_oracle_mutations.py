"""Mistakes planted in copies of the oracle must fail its pins (CPU only).

Each case copies the ``oracle`` package into a temporary directory, plants
one plausible mistake in the copy (a dropped or scaled sink term, a sign, a
wrong GQA map, a missing factor, an off-by-one window, a wrong operand), and
runs the pin tests against the copy in a separate process whose import path
puts the copy first. The unchanged copy must pass the same pins, so a failure
comes from the planted mistake and from nothing else. The mistakes live only
in the temporary copies; the oracle itself is never modified.
"""

import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CPP = "sinkattn_oracle.cpp"
CPP_MUTANTS = [
    ("sink dropped from Z", "double Z = std::isinf(S) ? 0.0 : std::exp(S - M);", "double Z = 0.0;"),
    ("sink multiplied by the scale", "return p.sinks ? p.sinks[h] :", "return p.sinks ? p.scale * p.sinks[h] :"),
    ("sign of dS_h", "part += -p_sink * Di;", "part += p_sink * Di;"),
    ("GQA map h mod Hkv", "const int h = un.head, kvh = h / G;", "const int h = un.head, kvh = h % p.Hkv;"),
    ("window one key too wide", [  # the mask and both row / key ranges it implies
        ("if (p.window > 0 && i - j >= p.window) return false;", "if (p.window > 0 && i - j > p.window) return false;"),
        ("*lo = p.window > 0 ? std::max<int64_t>(0, i - p.window + 1) : 0;",
         "*lo = p.window > 0 ? std::max<int64_t>(0, i - p.window) : 0;"),
        ("*hi = p.window > 0 ? std::min<int64_t>(L, j + p.window) : L;",
         "*hi = p.window > 0 ? std::min<int64_t>(L, j + p.window + 1) : L;")], None),
    ("dS without D", "const double dS = P[j] * (dot(doi, vj, d) - Di);", "const double dS = P[j] * dot(doi, vj, d);"),
    ("dk without the scale", "dk_row[t] += scale * dS * qi[t];", "dk_row[t] += dS * qi[t];"),
    ("dv from q", "dv_row[t] += Pij * doi[t];", "dv_row[t] += Pij * qi[t];"),
    ("LSE without the maximum", "const double LSE = M + std::log(Z);", "const double LSE = std::log(Z);"),
]
DEC = "decode.py"
DEC_MUTANTS = [
    ("window one key too wide", "k0 = max(0, L - window) if window > 0 else 0",
     "k0 = max(0, L - window - 1) if window > 0 else 0"),
    ("window one key too narrow", "k0 = max(0, L - window) if window > 0 else 0",
     "k0 = max(0, L - window + 1) if window > 0 else 0"),
    ("sink dropped from Z", "Z = e.sum() + (0.0 if s_h is None else np.exp(s_h[h] - m))", "Z = e.sum()"),
    ("sink multiplied by the scale", "Z = e.sum() + (0.0 if s_h is None else np.exp(s_h[h] - m))",
     "Z = e.sum() + (0.0 if s_h is None else np.exp(scale * s_h[h] - m))"),
    ("GQA map h mod Hkv", "g = h // G", "g = h % Hkv"),
    ("no scale", "s = scale * (K[:, g, :] @ q[b, h])", "s = (K[:, g, :] @ q[b, h])"),
    ("last key dropped", "K = gather_keys(k_cache, block_table, b, k0, L)",
     "K = gather_keys(k_cache, block_table, b, k0, max(k0, L - 1))"),
    ("wrong slot in a cache block", "return np.asarray(cache, dtype=np.float64)[blocks, j % bs]",
     "return np.asarray(cache, dtype=np.float64)[blocks, (j + 1) % bs]"),
    ("LSE without the maximum", "lse[h, b] = m + np.log(Z)", "lse[h, b] = np.log(Z)"),
    ("K read as V", "V = gather_keys(v_cache, block_table, b, k0, L)",
     "V = gather_keys(k_cache, block_table, b, k0, L)"),
]
PINS = {CPP: "tests/test_oracle.py", DEC: "tests/test_oracle_decode.py"}


def _run_pins(tmp, fname, old, new):
    """0: the pins pass on the copy; 1: a pin fails; anything else: an error."""
    dst = os.path.join(tmp, "oracle")
    shutil.copytree(os.path.join(ROOT, "oracle"), dst,
                    ignore=shutil.ignore_patterns("_build", "__pycache__"))
    if old is not None:
        path = os.path.join(dst, fname)
        text = open(path).read()
        for a, b in (old if isinstance(old, list) else [(old, new)]):
            assert text.count(a) == 1, f"mutation site not found once in {fname}: {a}"
            text = text.replace(a, b)
        open(path, "w").write(text)
    # PYTHONSAFEPATH keeps "python -m" from putting the working directory
    # (the repository, with the real oracle) ahead of the copy
    env = dict(os.environ, PYTHONPATH=os.pathsep.join([tmp, ROOT]), PYTHONSAFEPATH="1")
    r = subprocess.run([sys.executable, "-m", "pytest", PINS[fname], "-q", "-x", "-p", "no:cacheprovider",
                        "-m", "not gpu"], cwd=ROOT, env=env, capture_output=True, text=True, timeout=900)
    return r.returncode, r.stdout[-2000:] + r.stderr[-2000:]


def _check(tmp_path, fname, mutants):
    jobs = [(None, None, "unchanged copy")] + [(a, b, n) for n, a, b in mutants]
    dirs = [str(tmp_path / f"m{i}") for i in range(len(jobs))]
    for d in dirs:
        os.makedirs(d)
    with ThreadPoolExecutor(max_workers=min(len(jobs), os.cpu_count() or 1)) as ex:
        res = list(ex.map(lambda i: _run_pins(dirs[i], fname, jobs[i][0], jobs[i][1]), range(len(jobs))))
    code, out = res[0]
    assert code == 0, f"the pins fail on an unchanged copy of the oracle:\n{out}"
    missed = [jobs[i][2] for i in range(1, len(jobs)) if res[i][0] != 1]
    assert not missed, "planted mistakes the pins did not catch (or that broke the run): " + ", ".join(missed)


def test_pins_catch_mistakes_planted_in_the_training_oracle(tmp_path):
    _check(tmp_path, CPP, CPP_MUTANTS)


def test_pins_catch_mistakes_planted_in_the_decode_oracle(tmp_path):
    _check(tmp_path, DEC, DEC_MUTANTS)
