"""MXFP8 GEMM with few rows (M <= 128) on the block-scaled modes of the two
few-row kernels, stream-K (QK_MX_SKINNY=2) and cluster split-K
(QK_MX_SKINNY=3), against the oracle within |gpu - ref| <= 1e-2*|ref| +
1e-2*rms(ref) and cosine >= 0.99999.

The shapes cover one tile split over many CTAs (or over a cluster of 8),
tiles shared by two or three CTAs, whole tiles per CTA, a ragged last
K-block (K % 128 == 32 or 96), where the scale rows' length K/32 is not a
multiple of 4 and the scale warps load bytes into registers (with K % 128 ==
0 they copy 4-byte words by cp.async), a ragged last weight tile and both
activation tile heights (64 and 128 rows)."""
import numpy as np
import pytest

import oracle
import qk_inputs as qi
from gpu_util import assert_close, host_bits, run_mx

pytestmark = pytest.mark.gpu

SHAPES = [
    (1, 8, 16384),       # one tile over 128 CTAs
    (17, 136, 4064),     # two tiles, ragged last K-block, K/32 = 127
    (64, 2112, 7168),    # 17 tiles x 56 K-blocks
    (33, 7168, 1568),    # K/32 = 49: byte-wise scale loads
    (7, 4096, 4096),     # K % 128 == 0: cp.async scale copies
    (65, 1000, 640),     # 128-row activation tile, ragged last weight tile
    (128, 19456, 256),   # whole tiles per CTA
    (48, 5120, 2048),    # 40 tiles: clusters of 3 (uneven rows per CTA)
]


@pytest.fixture(params=["2", "3"], ids=["streamk", "cluster"])
def fewrow(request, monkeypatch):
    monkeypatch.setenv("QK_MX_SKINNY", request.param)
    return request.param


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_mxfp8_fewrow_matches_oracle(fewrow, shape):
    M, N, K = shape
    p = qi.mx_problem(qi.FMT_MXFP8_E4M3, M, N, K, seed=M + N)
    got = host_bits(run_mx(p))
    ref = oracle.gemm_mx(p.fmt, p.A, p.sA, p.B, p.sB)
    assert_close(got, ref, f"mxfp8 few-row mode {fewrow} {shape}")


def test_mxfp8_fewrow_bias_and_reproducible(fewrow):
    p = qi.mx_problem(qi.FMT_MXFP8_E4M3, 40, 3000, 3072, seed=5, bias=True)
    first = host_bits(run_mx(p))
    assert_close(first, oracle.gemm_mx(p.fmt, p.A, p.sA, p.B, p.sB, bias=p.bias), "bias")
    for _ in range(3):
        assert np.array_equal(host_bits(run_mx(p)), first), "fixed-order reduction must be reproducible"


def test_mxfp8_fewrow_exact_powers_of_two(fewrow):
    # elements in {0, +-1, +-2} and scales 2^e with |e| <= 3: every scaled
    # product is a multiple of 2^-6, and the partial sums of these random
    # signs stay far below 2^18, where such multiples are exact in fp32, so
    # the split of K changes no bit
    M, N, K = 48, 520, 8192
    rng = np.random.default_rng(3)
    vals = np.array([0.0, 1.0, -1.0, 2.0, -2.0], np.float32)
    A = qi.encode_e4m3(vals[rng.integers(0, 5, (M, K))])
    B = qi.encode_e4m3(vals[rng.integers(0, 5, (N, K))])
    sA = (127 + rng.integers(-3, 4, (M, K // 32))).astype(np.uint8)
    sB = (127 + rng.integers(-3, 4, (N, K // 32))).astype(np.uint8)
    p = qi.MxProblem(qi.FMT_MXFP8_E4M3, A, sA, B, sB, None, M, N, K)
    got = host_bits(run_mx(p))
    ref = oracle.gemm_mx(p.fmt, A, sA, B, sB)
    assert np.array_equal(got, qi.to_bf16_bits(ref.astype(np.float32)))


@pytest.mark.parametrize("shape", [(32, 21504, 2048), (64, 2112, 7168), (48, 12288, 2048), (100, 2112, 4096)],
                         ids=["streamk", "cluster", "cluster-s1", "cluster-128"])
def test_mxfp8_default_dispatch_few_rows(shape):
    # without the switch: 168 tiles (no cluster wave fits) x 16 K-blocks ->
    # stream-K; 17 tiles with a long K -> cluster split-K; 96 tiles -> one
    # CTA per tile; and the cluster kernel for 128 activation rows
    M, N, K = shape
    p = qi.mx_problem(qi.FMT_MXFP8_E4M3, M, N, K, seed=9, bias=True)
    got = host_bits(run_mx(p))
    assert_close(got, oracle.gemm_mx(p.fmt, p.A, p.sA, p.B, p.sB, bias=p.bias), f"default dispatch {shape}")
