"""The library's runtime calls around the GEMMs.

* qk_release gives the cached workspace memory back to the device: after an
  INT8 call (whose f16 copies of A and B, 2 (M + N) K bytes, come from the
  library's pool) the device's free memory grows by at least that much, and
  the next call still runs and gives the same bits.
* qk_set_wait_timeout_ns bounds every kernel wait: with a 20 ms bound a
  normal call neither times out nor changes its result, and 0 restores the
  default.
"""
import numpy as np
import pytest
import torch

import block_scaled_precision_tcgen05_gb300 as qk
import qk_inputs as qi
from gpu_util import host_bits, run_fp8, run_int8

pytestmark = pytest.mark.gpu


def test_release_returns_workspace_memory():
    M, N, K = 4096, 4096, 4096
    p = qi.int8_problem(M, N, K, seed=3)
    first = host_bits(run_int8(p))
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    free_before, _ = torch.cuda.mem_get_info()
    assert qk.load_library().qk_release() == qk.QK_OK
    free_after, _ = torch.cuda.mem_get_info()
    assert free_after - free_before >= 2 * (M + N) * K, (free_before, free_after)
    assert np.array_equal(host_bits(run_int8(p)), first), "a call after qk_release must give the same bits"
    assert qk.device_status() == 0


def test_wait_bound_setter():
    p = qi.fp8_problem(1024, 2048, 4096, seed=4)
    ref = host_bits(run_fp8(p))
    try:
        qk.set_wait_timeout_ns(20_000_000)
        for _ in range(3):
            assert np.array_equal(host_bits(run_fp8(p)), ref)
        assert qk.device_status() == 0
    finally:
        qk.set_wait_timeout_ns(0)
    assert np.array_equal(host_bits(run_fp8(p)), ref)
    assert qk.device_status() == 0
