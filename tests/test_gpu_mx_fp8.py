"""MXFP8, MXFP4 and FP8 per-token x per-channel GEMMs on the GPU against the
oracle, within |gpu - ref| <= 1e-2*|ref| + 1e-2*rms(ref) element-wise (ref
is the oracle's unrounded fp64 value) and cosine >= 0.99999.

K sweep after ROCm/mori PR #806's tests (K = 256, 512, 640, 1280, 2048:
one chunk, only the prologue's chunks, chunks refilled in the loop) and any
M unpadded (M = 1, 100, 1000).  Structured cases pin the scale-factor path:
constant elements with per-row / per-block scale codes have closed-form
results, so a misplaced scale byte cannot hide.
"""
import numpy as np
import pytest

import oracle
import qk_inputs as qi
from gpu_util import assert_close, host_bits, run_fp8, run_mx

pytestmark = pytest.mark.gpu

MX_SHAPES = [
    (1, 8, 32),
    (100, 136, 64),
    (128, 256, 256),
    (130, 264, 512),
    (1000, 520, 640),
    (256, 512, 1280),
    (300, 1040, 1792),
    (384, 768, 2048),
]

FMTS = [qi.FMT_MXFP8_E4M3, qi.FMT_MXFP4_E2M1]
FMT_IDS = ["mxfp8", "mxfp4"]


@pytest.mark.parametrize("shape", MX_SHAPES, ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("fmt", FMTS, ids=FMT_IDS)
def test_mx_matches_oracle(fmt, shape):
    M, N, K = shape
    p = qi.mx_problem(fmt, M, N, K, seed=M + K)
    got = host_bits(run_mx(p))
    ref = oracle.gemm_mx(fmt, p.A, p.sA, p.B, p.sB)
    assert_close(got, ref, f"fmt {fmt} {shape}")


@pytest.mark.parametrize("fmt", FMTS, ids=FMT_IDS)
def test_mx_with_bias(fmt):
    p = qi.mx_problem(fmt, 200, 264, 512, seed=11, bias=True)
    got = host_bits(run_mx(p))
    assert_close(got, oracle.gemm_mx(fmt, p.A, p.sA, p.B, p.sB, bias=p.bias), "bias")


def _ones(fmt, M, N, K):
    if fmt == qi.FMT_MXFP8_E4M3:
        return np.full((M, K), 0x38, np.uint8), np.full((N, K), 0x38, np.uint8)
    return np.full((M, K // 2), 0x22, np.uint8), np.full((N, K // 2), 0x22, np.uint8)


@pytest.mark.parametrize("fmt", FMTS, ids=FMT_IDS)
def test_mx_scale_layout_closed_form(fmt):
    # every element 1.0; sA[m,b] = 127 + da(m,b), sB[n,b] = 127 + db(n,b):
    # out[m,n] = sum_b 32 * 2^(da+db), exact in fp32 and in the oracle.
    M, N, K = 256, 512, 1024
    nb = K // 32
    A, B = _ones(fmt, M, N, K)
    m = np.arange(M)[:, None]
    n = np.arange(N)[:, None]
    b = np.arange(nb)[None, :]
    da = ((m * 7 + b * 3) % 5) - 2
    db = ((n * 5 + b) % 3) - 1
    sA = (127 + da).astype(np.uint8)
    sB = (127 + db).astype(np.uint8)
    p = qi.MxProblem(fmt, A, sA, B, sB, None, M, N, K)
    got = host_bits(run_mx(p))
    ref = oracle.gemm_mx(fmt, A, sA, B, sB)
    expect = (32.0 * np.exp2(da[:, None, :] + db[None, :, :])).sum(axis=2)
    assert np.array_equal(ref, expect)
    assert_close(got, ref, "closed-form scale layout")
    assert np.array_equal(got, qi.to_bf16_bits(ref.astype(np.float32))), "exact powers of two must round exactly"


@pytest.mark.parametrize("fmt", FMTS, ids=FMT_IDS)
def test_mx_single_block_scales(fmt):
    # one non-unit scale at a time pins (row, block) -> scale byte
    M, N, K = 128, 256, 512
    A, B = _ones(fmt, M, N, K)
    for (row, blk) in [(0, 0), (31, 3), (32, 4), (77, 9), (127, 15)]:
        sA = np.full((M, K // 32), 127, np.uint8)
        sB = np.full((N, K // 32), 127, np.uint8)
        sA[row, blk] = 130
        sB[200, blk] = 125
        p = qi.MxProblem(fmt, A, sA, B, sB, None, M, N, K)
        got = host_bits(run_mx(p))
        ref = oracle.gemm_mx(fmt, A, sA, B, sB)
        assert np.array_equal(got, qi.to_bf16_bits(ref.astype(np.float32))), (row, blk)


def test_mxfp4_nibble_order_with_identity():
    # A row i holds value 1.0 at element i only (low nibble for even i);
    # B = the same pattern, so out = identity; any nibble or K-offset error
    # in the operand path moves the ones.
    K = 64
    N = M = 64
    A = np.zeros((M, K // 2), np.uint8)
    for i in range(M):
        A[i, i // 2] = 0x02 if i % 2 == 0 else 0x20
    sA = np.full((M, K // 32), 127, np.uint8)
    p = qi.MxProblem(qi.FMT_MXFP4_E2M1, A, sA, A.copy(), sA.copy(), None, M, N, K)
    got = qi.from_bf16_bits(host_bits(run_mx(p)))
    assert np.array_equal(got, np.eye(M, dtype=np.float32))


def test_mxfp4_distinct_values_per_nibble():
    # A holds element values 0.5 (even k) and 3.0 (odd k); B holds 1.0 at one k
    M, N, K = 8, 64, 64
    A = np.full((M, K // 2), (0x5 << 4) | 0x1, np.uint8)   # low nibble 0.5, high nibble 3.0
    B = np.zeros((N, K // 2), np.uint8)
    for n in range(N):
        B[n, n // 2] = 0x02 if n % 2 == 0 else 0x20
    s = np.full((M, 2), 127, np.uint8)
    sB = np.full((N, 2), 127, np.uint8)
    p = qi.MxProblem(qi.FMT_MXFP4_E2M1, A, s, B, sB, None, M, N, K)
    got = qi.from_bf16_bits(host_bits(run_mx(p)))
    expect = np.tile(np.where(np.arange(N) % 2 == 0, 0.5, 3.0), (M, 1)).astype(np.float32)
    assert np.array_equal(got, expect)


FP8_SHAPES = [
    (1, 8, 16),
    (100, 136, 64),
    (130, 264, 256),
    (64, 2112, 7168),
    (1000, 520, 1792),
    (512, 768, 2048),
]


@pytest.mark.parametrize("bias", [False, True], ids=["nobias", "bias"])
@pytest.mark.parametrize("shape", FP8_SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_fp8_matches_oracle(shape, bias):
    M, N, K = shape
    p = qi.fp8_problem(M, N, K, seed=M + N, bias=bias)
    got = host_bits(run_fp8(p))
    ref = oracle.gemm_fp8_rowwise(p.A, p.B, p.sa, p.sb, bias=p.bias)
    assert_close(got, ref, f"fp8 {shape}")


def test_fp8_exact_small_integers():
    # E4M3 holds the integers -16..16 exactly; with unit scales the fp32
    # tensor-core sum of a short K is exact, so the result is bit-exact.
    rng = np.random.default_rng(1)
    M, N, K = 128, 256, 128
    vals = rng.integers(-4, 5, (M, K))
    wv = rng.integers(-4, 5, (N, K))
    A = qi.encode_e4m3(vals.astype(np.float32))
    B = qi.encode_e4m3(wv.astype(np.float32))
    p = qi.Fp8Problem(A, B, np.ones(M, np.float32), np.ones(N, np.float32), None, M, N, K)
    got = host_bits(run_fp8(p))
    exact = (vals @ wv.T).astype(np.float32)
    assert np.array_equal(got, qi.to_bf16_bits(exact))


@pytest.mark.parametrize("fmt", FMTS, ids=FMT_IDS)
@pytest.mark.parametrize("K,offset", [(1024, 0), (1024, 4), (896, 0), (96, 0)],
                         ids=["tma", "async-misaligned", "async", "loads"])
def test_mx_scale_staging_modes(fmt, K, offset):
    # The kernel fetches scale rows by TMA (K % 512 == 0 and 16-byte aligned
    # rows), by cp.async (K % 128 == 0 or rows only 4-byte aligned), or by
    # per-stage loads (other K); every mode must give the same result.
    import torch
    from gpu_util import to_dev, nan_out, host_bits
    import block_scaled_precision_tcgen05_gb300 as qk
    M, N = 300, 264
    p = qi.mx_problem(fmt, M, N, K, seed=K + offset)
    def shifted(x):
        flat = torch.zeros(x.size + 64, dtype=torch.uint8, device="cuda")
        view = flat[offset:offset + x.size].view(x.shape)
        view.copy_(to_dev(x))
        return view
    sA, sB = shifted(p.sA), shifted(p.sB)
    out = nan_out(M, N)
    qk.gemm_mx(fmt, to_dev(p.A), sA, to_dev(p.B), sB, None, out)
    torch.cuda.synchronize()
    assert_close(host_bits(out), oracle.gemm_mx(fmt, p.A, p.sA, p.B, p.sB), f"K={K} offset={offset}")
