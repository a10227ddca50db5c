"""NVFP4 GEMM (E2M1 elements, one UE4M3 scale per 16 K-elements, fp32
per-tensor scales) on the GPU against the oracle, within
|gpu - ref| <= 1e-2*|ref| + 1e-2*rms(ref) element-wise and cosine >= 0.99999.

Shapes cover any M unpadded, ragged N tiles, K from one 16-element block to
many ring passes, every scale-staging mode (TMA, cp.async, per-stage loads),
and a closed-form case whose per-block scale codes make a misplaced scale
byte visible."""
import numpy as np
import pytest
import torch

import block_scaled_precision_tcgen05_gb300 as qk
import oracle
import qk_inputs as qi
from gpu_util import assert_close, host_bits, nan_out, run_nvfp4, to_dev

pytestmark = pytest.mark.gpu

SHAPES = [
    (1, 8, 32),          # one row, K = two 16-blocks (per-stage scale loads)
    (100, 136, 64),      # cp.async scale rows
    (128, 256, 256),     # one tile, TMA scale rows
    (130, 264, 512),
    (1000, 520, 640),
    (256, 512, 1280),
    (300, 1040, 1792),
    (384, 768, 4096),
]


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_nvfp4_matches_oracle(shape):
    M, N, K = shape
    p = qi.nvfp4_problem(M, N, K, seed=M + K)
    got = host_bits(run_nvfp4(p))
    ref = oracle.gemm_nvfp4(p.A, p.sA, p.B, p.sB, p.global_a, p.global_b)
    assert_close(got, ref, f"nvfp4 {shape}")


def test_nvfp4_bias_and_default_global_scales():
    p = qi.nvfp4_problem(200, 264, 512, seed=11, bias=True)
    got = host_bits(run_nvfp4(p))
    assert_close(got, oracle.gemm_nvfp4(p.A, p.sA, p.B, p.sB, p.global_a, p.global_b, bias=p.bias), "bias")
    # NULL per-tensor scales mean 1.0
    got1 = host_bits(run_nvfp4(p, global_scales=False))
    assert_close(got1, oracle.gemm_nvfp4(p.A, p.sA, p.B, p.sB, 1.0, 1.0, bias=p.bias), "no global scales")


def test_nvfp4_scale_layout_closed_form():
    # every element 1.0 (E2M1 0x2); UE4M3 block scales with varied mantissas
    # and exponents: out[m,n] = ga*gb * sum_b 16 * sA[m,b] * sB[n,b]
    M, N, K = 256, 512, 1024
    nb = K // 16
    A = np.full((M, K // 2), 0x22, np.uint8)
    B = np.full((N, K // 2), 0x22, np.uint8)
    m = np.arange(M)[:, None]
    n = np.arange(N)[:, None]
    b = np.arange(nb)[None, :]
    sA = (0x30 + (m * 7 + b * 3) % 16).astype(np.uint8)   # 0.5 .. 1.875
    sB = (0x34 + (n * 5 + b) % 12).astype(np.uint8)       # 0.75 .. 2.75
    p = qi.Nvfp4Problem(A, sA, B, sB, 0.5, 4.0, None, M, N, K)
    got = host_bits(run_nvfp4(p))
    ref = oracle.gemm_nvfp4(A, sA, B, sB, 0.5, 4.0)
    dA = oracle.decode_ue4m3(np.arange(128))[sA]
    dB = oracle.decode_ue4m3(np.arange(128))[sB]
    expect = 2.0 * 16.0 * (dA[:, None, :] * dB[None, :, :]).sum(axis=2)
    assert np.array_equal(ref, expect)
    assert_close(got, ref, "closed-form NVFP4 scale layout")


def test_nvfp4_single_block_scale():
    # one nonzero scale byte per row pair: only block 5 of row 3 / column 7 counts
    M, N, K = 128, 256, 512
    A = np.full((M, K // 2), 0x22, np.uint8)
    B = np.full((N, K // 2), 0x22, np.uint8)
    sA = np.zeros((M, K // 16), np.uint8)
    sB = np.zeros((N, K // 16), np.uint8)
    sA[3, 5] = 0x40   # 2.0
    sB[7, 5] = 0x3C   # 1.5
    sA[10, :] = 0x38  # row 10: every block 1.0
    sB[7, :] = 0x3C
    p = qi.Nvfp4Problem(A, sA, B, sB, 1.0, 1.0, None, M, N, K)
    got = qi.from_bf16_bits(host_bits(run_nvfp4(p))).astype(np.float64)
    expect = np.zeros((M, N))
    expect[3, 7] = 16 * 2.0 * 1.5
    expect[10, 7] = 32 * 16 * 1.5
    assert np.array_equal(got, expect)


@pytest.mark.parametrize("K,offset", [(1024, 0), (1024, 4), (960, 0), (96, 0)],
                         ids=["tma", "async-misaligned", "async", "loads"])
def test_nvfp4_scale_staging_modes(K, offset):
    M, N = 300, 264
    p = qi.nvfp4_problem(M, N, K, seed=K + offset)

    def shifted(x):
        flat = torch.zeros(x.size + 64, dtype=torch.uint8, device="cuda")
        view = flat[offset:offset + x.size].view(x.shape)
        view.copy_(to_dev(x))
        return view

    out = nan_out(M, N)
    ga = to_dev(np.array([p.global_a], np.float32))
    gb = to_dev(np.array([p.global_b], np.float32))
    qk.gemm_nvfp4(to_dev(p.A), shifted(p.sA), to_dev(p.B), shifted(p.sB), ga, gb, None, out)
    torch.cuda.synchronize()
    ref = oracle.gemm_nvfp4(p.A, p.sA, p.B, p.sB, p.global_a, p.global_b)
    assert_close(host_bits(out), ref, f"K={K} offset={offset}")


def test_nvfp4_argument_errors():
    lib = qk.load_library()
    x = torch.zeros(64, dtype=torch.uint8, device="cuda")
    o = torch.zeros(64, dtype=torch.uint8, device="cuda")
    p = x.data_ptr()
    assert lib.qk_gemm_nvfp4(p, p, p, p, None, None, None, o.data_ptr(), 1, 8, 48, None) == qk.QK_ERR_ALIGN
    assert lib.qk_gemm_nvfp4(p, p, p, p, None, None, None, o.data_ptr(), 1, 12, 32, None) == qk.QK_ERR_ALIGN
    assert lib.qk_gemm_nvfp4(None, p, p, p, None, None, None, o.data_ptr(), 1, 8, 32, None) == qk.QK_ERR_ARG
    assert lib.qk_gemm_nvfp4(p, p, p, p, None, None, None, o.data_ptr(), 0, 8, 32, None) == qk.QK_OK
