"""Scale codes at the ends of their ranges, and NaN codes, on the GPU.

* UE8M0 codes 0, 1, 253 and 254 (2^-127, 2^-126, 2^126, 2^127) on A's blocks,
  each against a compensating code on B's, so that every block's product of
  scales stays inside fp32's normal range (OCP MX v1.0's E8M0 scale, as read
  for ROCm/mori PR #806's raw [rows, K/32] scales); MXFP8 and MXFP4.
* UE4M3 block scales with a zero exponent field (subnormal: m/8 * 2^-6) and
  the zero code on NVFP4 (ROCm/aiter PR #6262's NVFP4 operands).

Both are compared with the oracle element by element, within the tolerance of
the other MX tests.

NaN codes -- UE8M0 0xFF, E4M3 0x7F / 0xFF (elements of MXFP8, FP8 per-token
and FP8 blockscale operands), UE4M3 0x7F -- must turn exactly the outputs they
reach into NaN and leave every other output as the oracle computes it.  Only
NaN-ness is compared, not the bit pattern of a NaN.  UE4M3 codes with bit 7
set lie outside the format: the kernel reads their low seven bits.
"""
import numpy as np
import pytest

import oracle
import qk_inputs as qi
from gpu_util import assert_close, host_bits, run_blockscale, run_fp8, run_mx, run_nvfp4

pytestmark = pytest.mark.gpu

FMTS = [qi.FMT_MXFP8_E4M3, qi.FMT_MXFP4_E2M1]
FMT_IDS = ["mxfp8", "mxfp4"]


def _nan_pattern_matches(got_bits, ref, rows, cols, what):
    """The oracle's NaN mask is exactly the given rows and columns, the GPU's
    NaN mask equals it, and the finite outputs agree within the tolerance."""
    M, N = ref.shape
    expect = np.zeros((M, N), bool)
    expect[list(rows), :] = True
    expect[:, list(cols)] = True
    assert np.array_equal(np.isnan(ref), expect), f"{what}: oracle NaN mask"
    g = qi.from_bf16_bits(got_bits)
    assert np.array_equal(np.isnan(g), expect), f"{what}: GPU NaN mask differs in {int((np.isnan(g) != expect).sum())} outputs"
    keep_r = [m for m in range(M) if m not in rows]
    keep_c = [n for n in range(N) if n not in cols]
    assert_close(got_bits[np.ix_(keep_r, keep_c)], ref[np.ix_(keep_r, keep_c)], f"{what}: finite outputs")


@pytest.mark.parametrize("fmt", FMTS, ids=FMT_IDS)
def test_mx_extreme_ue8m0_codes(fmt):
    M, N, K = 200, 264, 1024
    p = qi.mx_problem(fmt, M, N, K, seed=41)
    nb = K // 32
    base = np.array([0, 1, 252, 253, 127, 2, 126, 251])[np.arange(nb) % 8]
    da = (np.arange(M)[:, None] + np.arange(nb)[None, :]) % 2
    db = (3 * np.arange(N)[:, None] + np.arange(nb)[None, :]) % 2
    sA = (base[None, :] + da).astype(np.uint8)
    sB = (254 - base[None, :] - db).astype(np.uint8)
    for code in (0, 1, 253, 254):
        assert (sA == code).any() and (sB == code).any()
    # every block's product of scales is 2^(da - db), da - db in {-1, 0, 1}
    assert set(np.unique(sA[:, None, :].astype(int) + sB[None, :, :].astype(int) - 254)) <= {-1, 0, 1}
    q = qi.MxProblem(fmt, p.A, sA, p.B, sB, None, M, N, K)
    got = host_bits(run_mx(q))
    ref = oracle.gemm_mx(fmt, p.A, sA, p.B, sB)
    assert np.isfinite(ref).all()
    assert_close(got, ref, f"fmt {fmt} extreme UE8M0 codes")


@pytest.mark.parametrize("fmt", FMTS, ids=FMT_IDS)
def test_mx_nan_scale_code(fmt):
    M, N, K = 130, 264, 512
    p = qi.mx_problem(fmt, M, N, K, seed=43)
    sA, sB = p.sA.copy(), p.sB.copy()
    sA[5, 3] = 0xFF
    sB[7, 0] = 0xFF
    sB[200, 15] = 0xFF
    q = qi.MxProblem(fmt, p.A, sA, p.B, sB, None, M, N, K)
    got = host_bits(run_mx(q))
    ref = oracle.gemm_mx(fmt, p.A, sA, p.B, sB)
    _nan_pattern_matches(got, ref, {5}, {7, 200}, f"fmt {fmt} UE8M0 0xFF")


def test_mxfp8_nan_elements():
    M, N, K = 130, 264, 512
    p = qi.mx_problem(qi.FMT_MXFP8_E4M3, M, N, K, seed=47)
    A, B = p.A.copy(), p.B.copy()
    A[9, 40] = 0x7F
    A[100, 511] = 0xFF
    B[11, 100] = 0xFF
    q = qi.MxProblem(qi.FMT_MXFP8_E4M3, A, p.sA, B, p.sB, None, M, N, K)
    got = host_bits(run_mx(q))
    ref = oracle.gemm_mx(qi.FMT_MXFP8_E4M3, A, p.sA, B, p.sB)
    _nan_pattern_matches(got, ref, {9, 100}, {11}, "MXFP8 E4M3 NaN elements")


def test_fp8_rowwise_nan_elements():
    M, N, K = 130, 264, 512
    p = qi.fp8_problem(M, N, K, seed=53)
    A, B = p.A.copy(), p.B.copy()
    A[3, 10] = 0x7F
    B[5, 20] = 0xFF
    B[263, 0] = 0x7F
    q = qi.Fp8Problem(A, B, p.sa, p.sb, None, M, N, K)
    got = host_bits(run_fp8(q))
    ref = oracle.gemm_fp8_rowwise(A, B, p.sa, p.sb)
    _nan_pattern_matches(got, ref, {3}, {5, 263}, "FP8 per-token NaN elements")


def test_fp8_blockscale_nan_elements():
    M, N, K = 130, 264, 640
    p = qi.blockscale_problem(M, N, K, seed=59)
    A, B = p.A.copy(), p.B.copy()
    A[64, 300] = 0xFF
    B[130, 639] = 0x7F
    q = qi.BlockscaleProblem(A, B, p.sa, p.sb, None, M, N, K)
    got = host_bits(run_blockscale(q))
    ref = oracle.gemm_fp8_blockscale(A, B, p.sa, p.sb)
    _nan_pattern_matches(got, ref, {64}, {130}, "FP8 blockscale NaN elements")


def test_nvfp4_subnormal_block_scales():
    # A's block scales all have a zero exponent field (codes 0..7: 0 and
    # m/8 * 2^-6); B's keep the recipe's normal codes
    M, N, K = 200, 264, 512
    p = qi.nvfp4_problem(M, N, K, seed=61)
    nb = K // 16
    sA = ((3 * np.arange(M)[:, None] + np.arange(nb)[None, :]) % 8).astype(np.uint8)
    assert (sA == 0).any() and (sA == 7).any()
    assert np.all(oracle.decode_ue4m3(sA) < 2.0 ** -6)
    q = qi.Nvfp4Problem(p.A, sA, p.B, p.sB, p.global_a, p.global_b, None, M, N, K)
    got = host_bits(run_nvfp4(q))
    ref = oracle.gemm_nvfp4(p.A, sA, p.B, p.sB, p.global_a, p.global_b)
    assert np.isfinite(ref).all() and np.abs(ref).max() > 0
    assert_close(got, ref, "NVFP4 subnormal UE4M3 block scales")


def test_nvfp4_nan_scale_code():
    M, N, K = 130, 264, 512
    p = qi.nvfp4_problem(M, N, K, seed=67)
    sA, sB = p.sA.copy(), p.sB.copy()
    sA[5, 2] = 0x7F
    sB[7, 31] = 0x7F
    q = qi.Nvfp4Problem(p.A, sA, p.B, sB, p.global_a, p.global_b, None, M, N, K)
    got = host_bits(run_nvfp4(q))
    ref = oracle.gemm_nvfp4(p.A, sA, p.B, sB, p.global_a, p.global_b)
    _nan_pattern_matches(got, ref, {5}, {7}, "NVFP4 UE4M3 0x7F")


def test_nvfp4_scale_bit7_is_ignored():
    # UE4M3 codes with bit 7 set are outside the format (the quantizers never
    # write them; the oracle decodes them as NaN to make any use visible).
    # The kernel reads the low seven bits: the result equals the oracle's on
    # the codes with bit 7 cleared.
    M, N, K = 128, 256, 512
    p = qi.nvfp4_problem(M, N, K, seed=71)
    sA = p.sA.copy()
    sA[5, 2] |= 0x80
    sA[9, :] |= 0x80
    sB = p.sB.copy()
    sB[17, 0] |= 0x80
    q = qi.Nvfp4Problem(p.A, sA, p.B, sB, p.global_a, p.global_b, None, M, N, K)
    got = host_bits(run_nvfp4(q))
    ref = oracle.gemm_nvfp4(p.A, sA & 0x7F, p.B, sB & 0x7F, p.global_a, p.global_b)
    assert_close(got, ref, "NVFP4 UE4M3 codes with bit 7 set")
