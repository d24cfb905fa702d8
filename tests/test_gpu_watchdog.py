"""The kernels' bounded waits, run out on purpose without any fault.

With the copy-withholding test hook on, the copy-issuing warp of each
pipelined kernel hands out its first work item and then issues nothing, so
the warps that wait for those copies reach the wait limit (set to 20 ms
here). Each kernel must then record SINKATTN_ERR_TIMEOUT in the device error
word, let what it issued finish, free its tensor memory and return: the call
completes, the CUDA context stays usable, and the next normal call on the
same context matches the oracle again.
"""

import numpy as np
import pytest
import torch

from attention_learnable_sinks_gb300 import _binding, api
from attention_learnable_sinks_gb300.workloads import make, make_decode

from parity import compare_full, run_cuda, run_oracle

pytestmark = pytest.mark.gpu

TIMEOUT = 5  # SINKATTN_ERR_TIMEOUT
LIMIT_NS = 20_000_000


def _expect_timeout(fn):
    lib = _binding.lib()
    assert _binding.device_error(reset=True) == 0
    lib.sinkattn_set_wait_limit_ns(LIMIT_NS)
    lib.sinkattn_test_withhold_copies(1)
    try:
        fn()
        torch.cuda.synchronize()  # the kernels returned: no hang, no fault
    finally:
        lib.sinkattn_test_withhold_copies(0)
        lib.sinkattn_set_wait_limit_ns(0)
    assert _binding.device_error(reset=True) == TIMEOUT


@pytest.mark.parametrize("d", [64, 128])
def test_forward_and_backward_waits_run_out_then_recover(cuda_lib, d):
    # head_dim 128: the 128-feature forward, the dK / dV block kernel and the
    # 128-feature dq pass
    w = make(f"watchdog_d{d}", [300, 129, 640], 8, 2, seed=31, d=d)
    dev = "cuda"
    q, k, v, do = (t.to(dev) for t in (w.q, w.k, w.v, w.dout))
    s, cu = w.sinks.to(dev), w.cu_seqlens.to(dev)
    o, lse = api.forward(q, k, v, s, cu, w.max_seqlen)
    torch.cuda.synchronize()
    assert _binding.device_error(reset=True) == 0

    _expect_timeout(lambda: api.forward(q, k, v, s, cu, w.max_seqlen))
    for det in (False, True):
        _expect_timeout(lambda: api.backward(q, k, v, s, cu, w.max_seqlen, o, lse, do,
                                             deterministic=det))
    # the context is intact: a normal call afterwards matches the oracle
    ref, *_ = run_oracle(w)
    for det in (False, True):
        compare_full(w, run_cuda(w, deterministic=det), ref)


@pytest.mark.parametrize("d", [64, 128])
def test_decode_waits_run_out_then_recover(cuda_lib, d):
    w = make_decode(f"watchdog_decode_d{d}", [200, 1000, 3000], 8, 2, block_size=64, seed=32, d=d)
    dev = "cuda"
    args = [t.to(dev) for t in (w.q, w.k_cache, w.v_cache, w.block_table, w.seqlens)]
    s = w.sinks.to(dev)
    o_ref, lse_ref = api.decode(*args, s, num_splits=1)
    torch.cuda.synchronize()
    assert _binding.device_error(reset=True) == 0
    for splits in (1, 4):
        _expect_timeout(lambda: api.decode(*args, s, num_splits=splits))
    _expect_timeout(lambda: api.decode(*args, s, exact=True))
    o, lse = api.decode(*args, s, num_splits=1)
    torch.cuda.synchronize()
    assert _binding.device_error(reset=True) == 0
    assert torch.equal(o, o_ref) and torch.equal(lse, lse_ref)
    assert np.isfinite(lse.cpu().numpy()).all()
