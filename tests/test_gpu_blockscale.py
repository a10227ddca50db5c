"""FP8 blockscale GEMM (fp32 scales per 1x128 of A and 128x128 of B) on the
GPU against the oracle, within |gpu - ref| <= 1e-2*|ref| + 1e-2*rms(ref)
element-wise and cosine >= 0.99999.

Shapes cover any M unpadded, N and K not multiples of 128 (a ragged last
scale block on both), one K-block and many, and a closed-form case in which
every K-block and N-block carries a distinct power-of-two scale, so a scale
applied to the wrong block cannot hide."""
import numpy as np
import pytest
import torch

import block_scaled_precision_tcgen05_gb300 as qk
import oracle
import qk_inputs as qi
from gpu_util import assert_close, host_bits, run_blockscale

pytestmark = pytest.mark.gpu

SHAPES = [
    (1, 8, 16),
    (100, 136, 128),
    (128, 256, 272),      # ragged last K-block
    (256, 264, 1024),
    (300, 520, 2048),
    (1000, 392, 1296),
    (384, 1024, 4096),
]


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_blockscale_matches_oracle(shape):
    M, N, K = shape
    p = qi.blockscale_problem(M, N, K, seed=M + K)
    got = host_bits(run_blockscale(p))
    ref = oracle.gemm_fp8_blockscale(p.A, p.B, p.sa, p.sb)
    assert_close(got, ref, f"blockscale {shape}")


def test_blockscale_with_bias():
    p = qi.blockscale_problem(200, 264, 640, seed=11, bias=True)
    got = host_bits(run_blockscale(p))
    assert_close(got, oracle.gemm_fp8_blockscale(p.A, p.B, p.sa, p.sb, bias=p.bias), "bias")


def test_blockscale_closed_form():
    # A, B all 1.0 (E4M3 0x38): out[m,n] = sum_g len_g * sa[m,g] * sb[n//128,g]
    M, N, K = 256, 392, 592          # K-blocks 128 x 4 + 80; N-blocks 128 x 3 + 8
    KB, NB = 5, 4
    A = np.full((M, K), 0x38, np.uint8)
    B = np.full((N, K), 0x38, np.uint8)
    m = np.arange(M)[:, None]
    g = np.arange(KB)[None, :]
    nb = np.arange(NB)[:, None]
    sa = np.exp2(((m + 2 * g) % 5) - 2).astype(np.float32)
    sb = np.exp2(((3 * nb + g) % 4) - 1).astype(np.float32)
    p = qi.BlockscaleProblem(A, B, sa, sb, None, M, N, K)
    got = host_bits(run_blockscale(p))
    ref = oracle.gemm_fp8_blockscale(A, B, sa, sb)
    lens = np.array([128, 128, 128, 128, 80], np.float64)
    sbn = sb[np.arange(N) // 128]                       # [N, KB]
    expect = (sa.astype(np.float64)[:, None, :] * sbn.astype(np.float64)[None, :, :] * lens).sum(axis=2)
    assert np.array_equal(ref, expect)
    assert np.array_equal(got, qi.to_bf16_bits(expect.astype(np.float32))), "exact sums must round exactly"


def test_blockscale_argument_errors():
    lib = qk.load_library()
    x = torch.zeros(64, dtype=torch.uint8, device="cuda")
    p = x.data_ptr()
    assert lib.qk_gemm_fp8_blockscale(p, p, p, p, None, p, 1, 8, 24, None) == qk.QK_ERR_ALIGN
    assert lib.qk_gemm_fp8_blockscale(p, p, p, p, None, p, 1, 12, 32, None) == qk.QK_ERR_ALIGN
    assert lib.qk_gemm_fp8_blockscale(p, None, p, p, None, p, 1, 8, 32, None) == qk.QK_ERR_ARG
    assert lib.qk_gemm_fp8_blockscale(p, p, p, p, None, p, 1, 0, 32, None) == qk.QK_OK
