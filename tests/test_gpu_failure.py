"""Failure detection without a GPU fault: a kernel whose barrier wait can
never complete gives up after its bound, records the give-up in the device
status word, and the context stays usable for the next GEMM."""
import ctypes

import numpy as np
import pytest
import torch

import block_scaled_precision_tcgen05_gb300 as qk
import oracle
import qk_inputs as qi
from gpu_util import assert_bit_exact, host_bits, run_int8

pytestmark = pytest.mark.gpu


def test_bounded_wait_reports_timeout_and_context_survives():
    lib = qk.load_library()
    assert qk.device_status(clear=True) == 0
    rc = lib.qk_wait_timeout_probe(ctypes.c_uint64(20_000_000), None)
    assert rc == qk.QK_ERR_TIMEOUT, qk.status_string(rc)
    assert qk.device_status(clear=True) == 0  # the probe cleared the word it set
    p = qi.int8_problem(128, 128, 256, seed=2, bias=True)
    got = host_bits(run_int8(p))
    assert_bit_exact(got, oracle.gemm_int8_rowwise(p.A, p.B, p.sa, p.sb, bias=p.bias), "after timeout")


def test_gemms_leave_the_status_word_clear():
    p = qi.int8_problem(300, 264, 1040, seed=4, bias=False)
    run_int8(p)
    assert qk.device_status(clear=False) == 0


def test_launch_counter_counts_kernels():
    before = qk.launch_count()
    p = qi.int8_problem(64, 64, 64, seed=1, bias=False)
    run_int8(p)
    assert qk.launch_count() - before == 2  # the f16 widening pass and the GEMM


def test_python_binding_rejects_bad_tensors():
    A = torch.zeros((128, 64), dtype=torch.int8, device="cuda")
    B = torch.zeros((64, 64), dtype=torch.int8, device="cuda")
    sa = torch.ones(128, device="cuda")
    sb = torch.ones(64, device="cuda")
    with pytest.raises(ValueError):
        qk.gemm_int8_rowwise(A, B.float(), sa, sb)
    with pytest.raises(ValueError):
        qk.gemm_int8_rowwise(A, B, sa[:100], sb)
    with pytest.raises(ValueError):
        qk.gemm_int8_rowwise(A.t(), B, sa, sb)
    with pytest.raises(qk.QkError) as e:
        qk.gemm_int8_rowwise(A[:, :40].contiguous(), B[:, :40].contiguous(), sa, sb)
    assert e.value.status == qk.QK_ERR_ALIGN
    with pytest.raises(ValueError):             # no float64 output type
        qk.gemm_int8_rowwise(A, B, sa, sb, out=torch.empty((128, 64), dtype=torch.float64, device="cuda"))
    with pytest.raises(ValueError):             # out's dtype contradicts out_dtype
        qk.gemm_int8_rowwise(A, B, sa, sb, out=torch.empty((128, 64), dtype=torch.float16, device="cuda"),
                             out_dtype=torch.float32)
    np.testing.assert_array_equal(qk.gemm_int8_rowwise(A, B, sa, sb).float().cpu().numpy(), 0)
