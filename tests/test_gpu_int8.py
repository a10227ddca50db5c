"""INT8 row/column-scaled GEMM on the GPU against the oracle: bit-exact.

comfy-kitchen PR #174, Validation (bit-for-bit agreement, zero error) and
the updates "Keep the cached INT8 epilogue scale order exact" and "Preserve
signed zero without INT8 bias".  Outputs are NaN-filled before each call so an
element the kernel never writes cannot pass.
"""
import numpy as np
import pytest
import torch

import oracle
import qk_inputs as qi
from gpu_util import assert_bit_exact, host_bits, run_int8, to_dev

pytestmark = pytest.mark.gpu

SHAPES = [
    (256, 256, 512),      # the small configuration
    (1, 8, 16),           # smallest legal problem
    (100, 136, 64),       # ragged M and N inside one tile
    (128, 128, 1024),     # exactly one accumulation chunk
    (129, 264, 1040),     # one row and a 16-K chunk past the edges
    (300, 520, 2048),     # several tiles, two chunks
    (77, 2112, 5376),     # skinny M, deep K with a partial last chunk
    (640, 1024, 3072),    # many tiles per CTA
]


@pytest.mark.parametrize("bias", [False, True], ids=["nobias", "bias"])
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_int8_matches_oracle(shape, bias):
    M, N, K = shape
    p = qi.int8_problem(M, N, K, seed=M + N + K, bias=bias)
    got = host_bits(run_int8(p))
    ref = oracle.gemm_int8_rowwise(p.A, p.B, p.sa, p.sb, bias=p.bias)
    assert_bit_exact(got, ref, f"int8 {shape} bias={bias}")


@pytest.mark.parametrize("K", [1024, 2048, 1040, 131056])
def test_int8_extreme_sums_are_exact(K):
    # all -128 (and a +127 column) drive every chunk sum to +-2^24 and the
    # total near the int32 limit (131056 * 16384 = 2147221504)
    M, N = 8, 16
    A = np.full((M, K), -128, np.int8)
    B = np.full((N, K), -128, np.int8)
    B[1] = 127
    A[2, ::3] = 1
    B[3, 5::7] = -1
    sa = np.full(M, 1.0, np.float32)
    sb = np.full(N, 1.0, np.float32)
    p = qi.Int8Problem(A, B, sa, sb, None, M, N, K)
    got = host_bits(run_int8(p))
    ref, acc = oracle.gemm_int8_rowwise(A, B, sa, sb, return_acc=True)
    assert acc[0, 0] == K * 16384
    assert_bit_exact(got, ref, f"extreme K={K}")


def test_int8_small_terms_next_to_large_partial_sums():
    # a partial sum just below 2^24 followed by +-1 products: any loss of the
    # low bits in the fp32 tensor-core accumulation would show up here
    K = 1024
    A = np.zeros((4, K), np.int8)
    B = np.zeros((8, K), np.int8)
    A[:, :1023] = -128
    B[:, :1023] = -128
    A[:, 1023] = 1
    B[:, 1023] = np.array([1, -1, 1, -1, 1, -1, 1, -1])
    A[1, 0] = 1  # 2^24 - 16384 + 128... asymmetric
    p = qi.Int8Problem(A, B, np.ones(4, np.float32), np.ones(8, np.float32), None, 4, 8, K)
    got = host_bits(run_int8(p))
    ref, acc = oracle.gemm_int8_rowwise(A, B, p.sa, p.sb, return_acc=True)
    assert acc[0, 0] == 1023 * 16384 + 1
    assert_bit_exact(got, ref, "near-2^24 partial sums")


def test_int8_signed_zero_without_bias():
    M, N, K = 128, 64, 64
    A = np.zeros((M, K), np.int8)
    A[64:, 0] = -3
    B = np.ones((N, K), np.int8)
    sa = np.full(M, -0.5, np.float32)
    sa[64:] = 1.0
    sb = np.full(N, 0.25, np.float32)
    sb[32:] = 0.0
    p = qi.Int8Problem(A, B, sa, sb, None, M, N, K)
    got = host_bits(run_int8(p))
    ref = oracle.gemm_int8_rowwise(A, B, sa, sb)
    assert np.all(ref[:64] == 0x8000)          # 0 * (-0.5) = -0
    assert np.all(ref[64:, 32:] == 0x8000)     # (-3) * 1 * (+0) = -0
    assert_bit_exact(got, ref, "signed zero, no bias")
    p.bias = np.zeros(N, np.uint16)
    got = host_bits(run_int8(p))
    ref = oracle.gemm_int8_rowwise(A, B, sa, sb, bias=p.bias)
    assert np.all(ref[:64] == 0x0000)          # -0 + +0 = +0
    assert_bit_exact(got, ref, "signed zero, zero bias")


def test_int8_epilogue_association_witnesses():
    # (acc*sa)*sb and acc*(sa*sb) round to different bf16 values here
    from oracle_pins import _find_association_witness, _int8_rows_for_acc
    for acc, sa, sb, left, right in _find_association_witness():
        a, b = _int8_rows_for_acc(acc)
        K = a.shape[1]
        A = np.repeat(a, 3, axis=0)
        B = np.repeat(b, 8, axis=0)
        p = qi.Int8Problem(A, B, np.full(3, sa, np.float32), np.full(8, sb, np.float32), None, 3, 8, K)
        got = host_bits(run_int8(p))
        assert np.all(got == left) and left != right


def test_int8_output_written_in_place_and_reused():
    p = qi.int8_problem(200, 264, 512, seed=5, bias=True)
    out = torch.full((200, 264), float("nan"), dtype=torch.bfloat16, device="cuda")
    run_int8(p, out)
    first = host_bits(out)
    run_int8(p, out)
    assert np.array_equal(first, host_bits(out))
    assert_bit_exact(first, oracle.gemm_int8_rowwise(p.A, p.B, p.sa, p.sb, bias=p.bias), "reuse")


def test_int8_on_a_side_stream():
    p = qi.int8_problem(256, 256, 512, seed=3, bias=False)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        A, B, sa, sb = to_dev(p.A), to_dev(p.B), to_dev(p.sa), to_dev(p.sb)
        import block_scaled_precision_tcgen05_gb300 as qk
        out = qk.gemm_int8_rowwise(A, B, sa, sb)
    s.synchronize()
    assert_bit_exact(host_bits(out), oracle.gemm_int8_rowwise(p.A, p.B, p.sa, p.sb), "side stream")
