"""FP8 per-token x per-channel GEMM with few rows (M <= 128) on the two
few-row kernels, stream-K (QK_FP8_SKINNY=2) and cluster split-K
(QK_FP8_SKINNY=3), and through the default dispatch, against the oracle
within |gpu - ref| <= 1e-2*|ref| + 1e-2*rms(ref) and cosine >= 0.99999.

The shapes make CTAs share tiles in every way the stream-K schedule allows:
one tile split over 128 CTAs (its owner adds 127 partials), tiles split over
two or three CTAs, CTAs that finish several whole tiles, a ragged last
K-block and a ragged last tile; the cluster kernel sees splits of 8 down to 1
(several waves when forced).  Partials are added in a fixed order, so
repeated calls are bit-identical."""
import numpy as np
import pytest
import torch

import oracle
import qk_inputs as qi
from gpu_util import assert_close, host_bits, run_fp8

pytestmark = pytest.mark.gpu

SHAPES = [
    (1, 8, 16384),       # one tile over 128 CTAs
    (17, 136, 4096),     # two tiles over 64 CTAs
    (64, 2112, 7168),    # 17 tiles x 56 K-blocks over all SMs
    (63, 7168, 1792),    # 56 tiles x 14 K-blocks
    (64, 21504, 1552),   # 168 tiles, ragged last K-block
    (65, 1000, 640),     # 128-row activation tile, ragged last weight tile
    (100, 264, 2048),
    (128, 19456, 256),   # 152 tiles x 2 K-blocks: whole tiles per CTA
    (48, 5120, 2048),    # 40 tiles: clusters of 3 (22 rows per CTA, the last 4)
    (64, 3072, 3072),    # 24 tiles: clusters of 6 (11 rows per CTA, the last 9)
]


@pytest.fixture(params=["0", "2", "3"], ids=["default", "streamk", "cluster"])
def fewrow(request, monkeypatch):
    monkeypatch.setenv("QK_FP8_SKINNY", request.param)
    return request.param


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_fewrow_matches_oracle(fewrow, shape):
    M, N, K = shape
    p = qi.fp8_problem(M, N, K, seed=M + N)
    got = host_bits(run_fp8(p))
    ref = oracle.gemm_fp8_rowwise(p.A, p.B, p.sa, p.sb)
    assert_close(got, ref, f"fp8 {shape}")


def test_fewrow_bias_and_reproducible(fewrow):
    p = qi.fp8_problem(40, 3000, 3072, seed=5, bias=True)
    first = host_bits(run_fp8(p))
    assert_close(first, oracle.gemm_fp8_rowwise(p.A, p.B, p.sa, p.sb, bias=p.bias), "bias")
    for _ in range(3):
        assert np.array_equal(host_bits(run_fp8(p)), first), "fixed-order reduction must be reproducible"


def test_fewrow_exact_small_integers(fewrow):
    # E4M3 integers with unit scales: every partial and total is an exact
    # integer in fp32, so the split across CTAs cannot change any bit
    M, N, K = 48, 520, 8192
    rng = np.random.default_rng(2)
    vals = np.array([0.0, 1.0, -1.0, 2.0, -2.0], np.float32)
    A = qi.encode_e4m3(vals[rng.integers(0, 5, (M, K))])
    B = qi.encode_e4m3(vals[rng.integers(0, 5, (N, K))])
    p = qi.Fp8Problem(A, B, np.ones(M, np.float32), np.ones(N, np.float32), None, M, N, K)
    got = host_bits(run_fp8(p))
    ref = oracle.gemm_fp8_rowwise(A, B, p.sa, p.sb)
    assert np.array_equal(got, qi.to_bf16_bits(ref.astype(np.float32)))
