"""MXFP4 and NVFP4 GEMMs with few rows (M <= 128) on the FP4 modes of the two
few-row kernels, stream-K (QK_MX_SKINNY=2) and cluster split-K
(QK_MX_SKINNY=3), against the oracle within the MX tolerance
(|gpu - ref| <= 1e-2*|ref| + 1e-2*rms(ref), cosine >= 0.99999).

A ring stage holds 128 bytes of K per row, 256 packed E2M1 elements, with two
UE8M0 (MXFP4, ROCm/FlyDSL PR #990) or four UE4M3 (NVFP4, ROCm/aiter PR #6262)
scale words per row.  The shapes cover one tile split over many CTAs (or a
cluster of 8), tiles shared by two or three CTAs, clusters of 3 and 6
(uneven output rows per CTA), whole tiles per CTA, a
ragged last K-block (K % 256 == 224 or 32: the last MMAs of K = 64 run on
zero-filled elements, and the scale rows end inside a stage, so the scale
warp loads bytes into registers; with K % 256 == 0 it copies words by
cp.async), a ragged last weight tile and both activation tile heights (64
and 128 rows)."""
import numpy as np
import pytest

import oracle
import qk_inputs as qi
from gpu_util import assert_close, host_bits, run_mx, run_nvfp4

pytestmark = pytest.mark.gpu

SHAPES = [
    (1, 8, 16384),       # one tile, 64 K-blocks of 128 bytes
    (17, 136, 4064),     # two tiles, ragged last K-block
    (64, 2112, 7168),    # 17 tiles x 28 K-blocks
    (33, 7168, 1568),    # K % 256 == 32: one MMA in the last stage
    (7, 4096, 4096),     # K % 256 == 0: cp.async scale copies
    (65, 1000, 640),     # 128-row activation tile, ragged last weight tile
    (128, 19456, 256),   # whole tiles per CTA
    (48, 5120, 2048),    # 40 tiles: clusters of 3 (uneven rows per CTA)
    (64, 3072, 3072),    # 24 tiles: clusters of 6
]
IDS = ["x".join(map(str, s)) for s in SHAPES]


@pytest.fixture(params=["2", "3"], ids=["streamk", "cluster"])
def fewrow(request, monkeypatch):
    monkeypatch.setenv("QK_MX_SKINNY", request.param)
    return request.param


@pytest.mark.parametrize("shape", SHAPES, ids=IDS)
def test_mxfp4_fewrow_matches_oracle(fewrow, shape):
    M, N, K = shape
    p = qi.mx_problem(qi.FMT_MXFP4_E2M1, M, N, K, seed=M + N + 1)
    got = host_bits(run_mx(p))
    ref = oracle.gemm_mx(p.fmt, p.A, p.sA, p.B, p.sB)
    assert_close(got, ref, f"mxfp4 few-row mode {fewrow} {shape}")


@pytest.mark.parametrize("shape", SHAPES, ids=IDS)
def test_nvfp4_fewrow_matches_oracle(fewrow, shape):
    M, N, K = shape
    p = qi.nvfp4_problem(M, N, K, seed=M + N + 2)
    got = host_bits(run_nvfp4(p))
    ref = oracle.gemm_nvfp4(p.A, p.sA, p.B, p.sB, p.global_a, p.global_b)
    assert_close(got, ref, f"nvfp4 few-row mode {fewrow} {shape}")


def test_fp4_fewrow_bias_and_reproducible(fewrow):
    p = qi.mx_problem(qi.FMT_MXFP4_E2M1, 40, 3000, 3072, seed=5, bias=True)
    first = host_bits(run_mx(p))
    assert_close(first, oracle.gemm_mx(p.fmt, p.A, p.sA, p.B, p.sB, bias=p.bias), "mxfp4 bias")
    for _ in range(2):
        assert np.array_equal(host_bits(run_mx(p)), first), "fixed-order reduction must be reproducible"
    q = qi.nvfp4_problem(40, 3000, 3072, seed=6, bias=True)
    got = host_bits(run_nvfp4(q))
    assert_close(got, oracle.gemm_nvfp4(q.A, q.sA, q.B, q.sB, q.global_a, q.global_b, bias=q.bias), "nvfp4 bias")
    # without per-tensor scales the epilogue multiplies by 1
    got1 = host_bits(run_nvfp4(q, global_scales=False))
    assert_close(got1, oracle.gemm_nvfp4(q.A, q.sA, q.B, q.sB, 1.0, 1.0, bias=q.bias), "nvfp4 no global scales")


def test_mxfp4_fewrow_exact_powers_of_two(fewrow):
    # E2M1 elements in {0, +-1, +-2} and scales 2^e with |e| <= 3: every
    # scaled product is a multiple of 2^-6 and the partial sums of these
    # random signs stay far below 2^18, so no split of K changes a bit
    M, N, K = 48, 520, 8192
    rng = np.random.default_rng(3)
    codes = np.array([0x0, 0x2, 0xA, 0x4, 0xC], np.uint8)  # 0, 1, -1, 2, -2
    a = codes[rng.integers(0, 5, (M, K))]
    b = codes[rng.integers(0, 5, (N, K))]
    A = (a[:, 0::2] | (a[:, 1::2] << 4)).astype(np.uint8)
    B = (b[:, 0::2] | (b[:, 1::2] << 4)).astype(np.uint8)
    sA = (127 + rng.integers(-3, 4, (M, K // 32))).astype(np.uint8)
    sB = (127 + rng.integers(-3, 4, (N, K // 32))).astype(np.uint8)
    p = qi.MxProblem(qi.FMT_MXFP4_E2M1, A, sA, B, sB, None, M, N, K)
    got = host_bits(run_mx(p))
    ref = oracle.gemm_mx(p.fmt, A, sA, B, sB)
    assert np.array_equal(got, qi.to_bf16_bits(ref.astype(np.float32)))


@pytest.mark.parametrize("shape", [(32, 21504, 4096), (64, 2112, 7168), (64, 7168, 2048), (100, 2112, 8192)],
                         ids=["streamk", "cluster", "cluster-s1", "cluster-128"])
def test_fp4_default_dispatch_few_rows(shape):
    # without the switch, the dispatch rule on 128-byte K-blocks picks the
    # few-row kernels or the tile kernel; every choice matches the oracle
    M, N, K = shape
    p = qi.mx_problem(qi.FMT_MXFP4_E2M1, M, N, K, seed=9, bias=True)
    got = host_bits(run_mx(p))
    assert_close(got, oracle.gemm_mx(p.fmt, p.A, p.sA, p.B, p.sB, bias=p.bias), f"mxfp4 default dispatch {shape}")
    q = qi.nvfp4_problem(M, N, K, seed=10, bias=True)
    got = host_bits(run_nvfp4(q))
    assert_close(got, oracle.gemm_nvfp4(q.A, q.sA, q.B, q.sB, q.global_a, q.global_b, bias=q.bias),
                 f"nvfp4 default dispatch {shape}")
