"""The C ABI without a GPU: the library loads, exports every function that
include/sinkattn.h declares, its parameter structs match the binding, and
bad arguments are rejected on the host before anything is launched."""

import ctypes
import os
import re

import pytest

from attention_learnable_sinks_gb300 import _binding
from attention_learnable_sinks_gb300._binding import BwdParams, DecodeParams, FwdParams

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    src = open(os.path.join(ROOT, "include", "sinkattn.h")).read()
    return re.findall(r"SINKATTN_API\s+[\w\s\*]+?\b(sinkattn_\w+)\s*\(", src)


def test_library_exports_every_declared_symbol():
    lib = _binding.lib()
    names = declared_functions()
    assert len(names) >= 11
    bound = {n for n, _, _ in _binding.SYMBOLS}
    for n in names:
        assert hasattr(lib, n), f"{n} not exported"
        assert n in bound, f"{n} not bound in _binding.SYMBOLS"


def test_param_struct_sizes_match():
    lib = _binding.lib()
    assert lib.sinkattn_params_size(0) == ctypes.sizeof(FwdParams)
    assert lib.sinkattn_params_size(1) == ctypes.sizeof(BwdParams)
    assert lib.sinkattn_params_size(2) == ctypes.sizeof(DecodeParams)
    assert lib.sinkattn_params_size(3) == 0


def test_param_struct_field_offsets_match(tmp_path):
    """Every field of the binding's structs sits where the C header puts it
    (sizes alone miss two same-sized fields in swapped order). A small C
    program compiled against include/sinkattn.h prints the offsets."""
    import shutil
    import subprocess
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    structs = (("sinkattn_fwd_params", FwdParams), ("sinkattn_bwd_params", BwdParams),
               ("sinkattn_decode_params", DecodeParams))
    lines = ["#include <stddef.h>", "#include <stdio.h>", '#include "sinkattn.h"',
             "int main(void) {"]
    for cname, cls in structs:
        for name, _ in cls._fields_:
            lines.append(f'  printf("{cname}.{name} %zu\\n", offsetof({cname}, {name}));')
        lines.append(f'  printf("{cname} %zu\\n", sizeof({cname}));')
    lines += ["  return 0;", "}"]
    src = tmp_path / "offsets.c"
    src.write_text("\n".join(lines) + "\n")
    exe = tmp_path / "offsets"
    subprocess.run([cc, "-std=c11", "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)],
                   check=True, capture_output=True)
    got = dict(l.rsplit(" ", 1) for l in subprocess.run([str(exe)], check=True, capture_output=True,
                                                        text=True).stdout.splitlines())
    for cname, cls in structs:
        for name, _ in cls._fields_:
            assert int(got[f"{cname}.{name}"]) == getattr(cls, name).offset, f"{cname}.{name}"
        assert int(got[cname]) == ctypes.sizeof(cls), cname


def test_decode_workspace_sizes():
    lib = _binding.lib()
    w64 = lib.sinkattn_decode_workspace_size(5, 64, 8)
    assert w64 == lib.sinkattn_decode_workspace_size_d(5, 64, 8, 64)
    # (max, sum) pairs, then one output row per (sequence, head, split)
    n = 5 * 64 * 8
    assert w64 == ((n * 8 + 255) // 256) * 256 + n * 64 * 4
    assert lib.sinkattn_decode_workspace_size_d(5, 64, 8, 128) == ((n * 8 + 255) // 256) * 256 + n * 128 * 4
    assert lib.sinkattn_decode_workspace_size_d(5, 64, 8, 96) == 0
    assert lib.sinkattn_decode_workspace_size_d(5, 64, 65, 64) == 0


def test_workspace_sizes():
    lib = _binding.lib()
    f = lib.sinkattn_fwd_workspace_size(4, 8192, 64, 8, 64)
    b = lib.sinkattn_bwd_workspace_size(4, 8192, 64, 8, 64)
    assert 0 < f < b
    assert b >= 8192 * 64 * 64 * 4  # fp32 dq accumulator
    assert lib.sinkattn_fwd_workspace_size(4, 8192, 64, 8, 96) == 0
    assert lib.sinkattn_bwd_workspace_size(4, 8192, 64, 8, 256) == 0
    # head_dim 128: same lists; the backward is always the deterministic one
    # (no fp32 dq accumulator), whatever mode is asked for
    assert lib.sinkattn_fwd_workspace_size(4, 8192, 64, 8, 128) == f
    det = lib.sinkattn_bwd_workspace_size_mode(4, 8192, 64, 8, 64, 1)
    assert det < b
    assert lib.sinkattn_bwd_workspace_size(4, 8192, 64, 8, 128) == det
    assert lib.sinkattn_bwd_workspace_size_mode(4, 8192, 64, 8, 128, 0) == det
    assert lib.sinkattn_bwd_workspace_size(4, 8192, 63, 8, 64) == 0
    assert lib.sinkattn_bwd_workspace_size(-1, 8192, 64, 8, 64) == 0


def test_status_strings():
    lib = _binding.lib()
    for code in range(6):
        assert lib.sinkattn_status_string(code)
    assert lib.sinkattn_status_string(99) == b"unknown status"


def _params(**kw):
    p = FwdParams()
    fake = 0x10000  # never dereferenced: every case below fails or returns before a launch
    p.q = p.k = p.v = p.o = p.lse = p.cu_seqlens = fake
    p.nseq, p.total, p.max_seqlen = 1, 128, 128
    p.Hq, p.Hkv, p.head_dim, p.causal, p.window = 4, 2, 64, 1, 0
    buf = (ctypes.c_uint8 * 4096)()
    p.workspace, p.workspace_bytes = ctypes.addressof(buf), 4096
    for k, v in kw.items():
        setattr(p, k, v)
    return p, buf


@pytest.mark.parametrize("change,status", [
    ({"head_dim": 96}, 2),
    ({"head_dim": 256}, 2),
    ({"head_dim": 128, "q_row_stride": 4 * 64}, 1),  # covers the heads at 64, not at 128
    ({"Hq": 5}, 1),
    ({"Hkv": 0}, 1),
    ({"causal": 0, "window": 16}, 2),
    ({"causal": 2}, 1),
    ({"cu_seqlens": None}, 1),
    ({"q": None}, 1),
    ({"q": 0x10008}, 1),          # not 16-byte aligned
    ({"q_row_stride": 4 * 64 + 4}, 1),
    ({"k_row_stride": 64}, 1),     # does not cover both kv heads
    ({"max_seqlen": 0}, 1),
    ({"softmax_scale": float("nan")}, 1),
    ({"workspace_bytes": 8}, 4),
    ({"workspace": None}, 4),
])
def test_forward_rejects_bad_arguments(change, status):
    lib = _binding.lib()
    n0 = lib.sinkattn_launch_count()
    p, buf = _params(**change)
    assert lib.sinkattn_fwd(ctypes.byref(p), None) == status
    assert lib.sinkattn_last_error_message()
    assert lib.sinkattn_launch_count() == n0


def test_empty_forward_needs_no_device():
    lib = _binding.lib()
    p, buf = _params(total=0, max_seqlen=0)
    assert lib.sinkattn_fwd(ctypes.byref(p), None) == 0
    assert lib.sinkattn_last_error_message() == b""


def test_backward_rejects_missing_outputs():
    lib = _binding.lib()
    b = BwdParams()
    p, buf = _params()
    b.fwd = p
    big = (ctypes.c_uint8 * (1 << 22))()
    b.workspace, b.workspace_bytes = ctypes.addressof(big), len(big)
    b.dout = b.dq = b.dk = 0x10000
    b.dv = None
    assert lib.sinkattn_bwd(ctypes.byref(b), None) == 1
    b.dv = 0x10000
    b.fwd.lse = None
    assert lib.sinkattn_bwd(ctypes.byref(b), None) == 1
    assert lib.sinkattn_bwd(None, None) == 1


def test_sequence_groups_for_the_host_pipeline():
    from attention_learnable_sinks_gb300.api import _split_sequences
    # bounds are sequence indices, cover everything, and cut only between sequences
    assert _split_sequences([2048] * 4, True, 0, 2) == [0, 2, 4]
    assert _split_sequences([2048] * 4, True, 0, 1) == [0, 4]
    assert _split_sequences([5], True, 0, 3) == [0, 1]
    assert _split_sequences([], True, 0, 2) == [0, 0]
    b = _split_sequences([100, 4000, 50, 50, 3000], True, 0, 3)
    assert b[0] == 0 and b[-1] == 5 and all(x < y for x, y in zip(b, b[1:]))
    # a windowed cost grows linearly, so equal lengths still split evenly
    assert _split_sequences([1000] * 6, True, 128, 3) == [0, 2, 4, 6]


def _decode_params(**kw):
    p = DecodeParams()
    fake = 0x10000  # never dereferenced: every case below fails or returns before a launch
    p.q = p.k_cache = p.v_cache = p.block_table = p.seqlens = p.o = p.lse = fake
    p.nseq, p.num_blocks, p.block_size, p.max_blocks_per_seq = 2, 8, 16, 4
    p.Hq, p.Hkv, p.head_dim, p.window, p.num_splits = 8, 2, 64, 0, 0
    buf = (ctypes.c_uint8 * 4096)()
    p.workspace, p.workspace_bytes = ctypes.addressof(buf), 4096
    for k, v in kw.items():
        setattr(p, k, v)
    return p, buf


@pytest.mark.parametrize("change,status", [
    ({"head_dim": 96}, 2),
    ({"head_dim": 128, "block_size": 8}, 2),   # head_dim 128 passes; the block size does not
    ({"Hq": 6, "Hkv": 2}, 2),      # group of 3
    ({"Hq": 64, "Hkv": 2}, 2),     # group of 32
    ({"Hkv": 3}, 1),
    ({"nseq": 65536}, 1),
    ({"block_size": 8}, 2),
    ({"block_size": 256}, 2),
    ({"num_blocks": 0}, 1),
    ({"max_blocks_per_seq": 0}, 1),
    ({"num_blocks": 1 << 27, "block_size": 16}, 1),  # 2^31 cache rows
    ({"num_splits": 65}, 1),
    ({"num_splits": -1}, 1),
    ({"softmax_scale": float("inf")}, 1),
    ({"q": None}, 1),
    ({"block_table": None}, 1),
    ({"k_cache": 0x10004}, 1),     # not 16-byte aligned
    ({"workspace": None}, 4),
    ({"num_splits": 64, "workspace_bytes": 64}, 4),
])
def test_decode_rejects_bad_arguments(change, status):
    lib = _binding.lib()
    n0 = lib.sinkattn_launch_count()
    p, buf = _decode_params(**change)
    assert lib.sinkattn_decode(ctypes.byref(p), None) == status
    assert lib.sinkattn_last_error_message()
    assert lib.sinkattn_launch_count() == n0


@pytest.mark.parametrize("change,status", [
    ({"head_dim": 96}, 2),
    ({"head_dim": 256}, 2),
    ({"head_dim": 128, "block_size": 8}, 2),   # head_dim 128 passes; the block size does not
    ({"head_dim": 128, "q": None}, 1),
    ({"workspace_bytes": 8}, 4),
])
def test_exact_decode_rejects_bad_arguments(change, status):
    # the exact decode takes head_dim 64 or 128; every case fails before a launch
    lib = _binding.lib()
    n0 = lib.sinkattn_launch_count()
    p, buf = _decode_params(**change)
    assert lib.sinkattn_decode_exact(ctypes.byref(p), None) == status
    assert lib.sinkattn_last_error_message()
    assert lib.sinkattn_launch_count() == n0


def test_decode_without_sequences_needs_no_device():
    lib = _binding.lib()
    p, buf = _decode_params(nseq=0, q=None, workspace=None)
    assert lib.sinkattn_decode(ctypes.byref(p), None) == 0
    assert lib.sinkattn_decode(None, None) == 1


def test_decode_workspace_size():
    lib = _binding.lib()
    one = lib.sinkattn_decode_workspace_size(64, 64, 1)
    assert one >= 64 * 64 * (2 + 64) * 4
    assert lib.sinkattn_decode_workspace_size(64, 64, 8) >= 8 * 64 * 64 * 66 * 4
    assert lib.sinkattn_decode_workspace_size(64, 64, 0) == 0
    assert lib.sinkattn_decode_workspace_size(64, 64, 65) == 0
    assert lib.sinkattn_decode_workspace_size(-1, 64, 1) == 0


def test_module_holds_one_fp32_sink_per_head():
    import torch
    from attention_learnable_sinks_gb300 import SinkAttention
    layer = SinkAttention(12, window=64, init=-1.5)
    assert [n for n, _ in layer.named_parameters()] == ["sinks"]
    assert layer.sinks.shape == (12,) and layer.sinks.dtype == torch.float32
    assert bool((layer.sinks == -1.5).all()) and layer.sinks.requires_grad
    assert "num_heads=12" in repr(layer) and "window=64" in repr(layer)
