"""qk_gemm_int8_rowwise_noalloc: the INT8 GEMM for callers that cannot let a
library allocate device memory (a process whose HBM already belongs to its
own allocator, a hot loop that must not block on allocator calls, a policy
against hidden allocations).  It must give exactly what the allocating entry
point gives, call after call, while its fixed scratch array is reused.

This file sorts last so that a run stopping at the first failure has already
run every other test; it also passes on its own in a fresh process."""
import ctypes

import numpy as np
import pytest
import torch

import block_scaled_precision_tcgen05_gb300 as qk
import qk_inputs as qi

SCRATCH_BYTES = 32 << 20


def _abi_call(lib, name, A, B, sa, sb, bias, out):
    M, K = A.shape
    N = B.shape[0]
    p = lambda t: None if t is None else ctypes.c_void_p(t.data_ptr())
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return getattr(lib, name)(p(A), p(B), p(sa), p(sb), p(bias), p(out), M, N, K, stream)


def _device_problem(M, N, K, seed, bias):
    pr = qi.int8_problem(M, N, K, seed=seed, bias=bias)
    dev = lambda x: torch.from_numpy(np.ascontiguousarray(x)).cuda()
    b = None if pr.bias is None else dev(pr.bias.view(np.int16)).view(torch.bfloat16)
    return dev(pr.A), dev(pr.B), dev(pr.sa), dev(pr.sb), b


def _bits(t):
    return t.view(torch.int16).cpu().numpy()


@pytest.mark.gpu
def test_noalloc_matches_the_allocating_entry_point_on_calls_in_a_row():
    lib = qk.load_library()
    # (M + N) * K * 2 bytes: 8.3 MB and 18.9 MB, both inside the 32 MiB scratch
    for (M, N, K, seed, bias) in [(1000, 1024, 2048, 1, True), (777, 1536, 4096, 2, False)]:
        A, B, sa, sb, b = _device_problem(M, N, K, seed, bias)
        ref = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
        assert _abi_call(lib, "qk_gemm_int8_rowwise", A, B, sa, sb, b, ref) == qk.QK_OK
        torch.cuda.synchronize()
        free_before = None
        for call in range(2):
            out = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
            torch.cuda.synchronize()
            if call == 1:
                free_before = torch.cuda.mem_get_info()[0]
            assert _abi_call(lib, "qk_gemm_int8_rowwise_noalloc", A, B, sa, sb, b, out) == qk.QK_OK
            torch.cuda.synchronize()
            if call == 1:
                assert torch.cuda.mem_get_info()[0] == free_before, "device memory changed during the call"
            # INT8 parity is bit-exact: the same bf16 patterns as the allocating entry point
            assert np.array_equal(_bits(out), _bits(ref)), f"call {call} of {M}x{N}x{K} differs"
    assert qk.device_status(clear=False) == 0


def test_noalloc_rejects_problems_beyond_its_scratch():
    # validation happens on the host before any CUDA call, so this runs anywhere
    lib = qk.load_library()
    fake = ctypes.c_void_p(0x100000)
    M, N, K = 4096, 4096, 4096                  # (M + N) * K * 2 = 128 MiB > 32 MiB
    assert (M + N) * K * 2 > SCRATCH_BYTES
    rc = lib.qk_gemm_int8_rowwise_noalloc(fake, fake, fake, fake, None, fake, M, N, K, None)
    assert rc == qk.QK_ERR_SCRATCH
    assert "32 MiB" in qk.status_string(rc)
    assert lib.qk_gemm_int8_rowwise_noalloc(fake, fake, fake, fake, None, fake, 0, N, K, None) == qk.QK_OK


_FRESH_PROCESS = r"""
import ctypes, sys
import numpy as np
import torch
sys.path.insert(0, ROOT)
import block_scaled_precision_tcgen05_gb300 as qk
import oracle
import qk_inputs as qi

lib = qk.load_library()
M, N, K = 512, 768, 1024                    # (M + N) * K * 2 = 2.6 MB of scratch
pr = qi.int8_problem(M, N, K, seed=5, bias=True)
dev = lambda x: torch.from_numpy(np.ascontiguousarray(x)).cuda()
A, B, sa, sb = dev(pr.A), dev(pr.B), dev(pr.sa), dev(pr.sb)
bias = dev(pr.bias.view(np.int16)).view(torch.bfloat16)
outs = [torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda") for _ in range(2)]
p = lambda t: ctypes.c_void_p(t.data_ptr())
stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
torch.cuda.synchronize()
torch.cuda.mem_get_info()
free = []
for out in outs:
    free.append(torch.cuda.mem_get_info()[0])
    rc = lib.qk_gemm_int8_rowwise_noalloc(p(A), p(B), p(sa), p(sb), p(bias), p(out), M, N, K, stream)
    assert rc == qk.QK_OK, rc
    torch.cuda.synchronize()
free.append(torch.cuda.mem_get_info()[0])
# the first call on the device looks up the scratch array (and loads the
# kernels' module); the second one must not change the device's free memory
assert free[2] == free[1], free
ref = oracle.gemm_int8_rowwise(pr.A, pr.B, pr.sa, pr.sb, bias=pr.bias)
for i, out in enumerate(outs):
    got = out.view(torch.int16).cpu().numpy().view(np.uint16)
    assert np.array_equal(got, ref), f"call {i} differs from the oracle"
assert qk.device_status(clear=False) == 0
print("FRESH_PROCESS_OK")
"""


@pytest.mark.gpu
def test_noalloc_first_calls_in_a_fresh_process():
    # Only the no-allocation entry point runs in this process, so nothing else
    # has created the library's memory pool or touched the scratch array before
    # it: two calls, bit-exact against the CPU oracle, free device memory
    # unchanged across the second.
    import os
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    code = f"ROOT = {root!r}\n" + _FRESH_PROCESS
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=600)
    assert r.returncode == 0 and "FRESH_PROCESS_OK" in r.stdout, r.stdout + r.stderr
