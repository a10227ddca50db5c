"""FP8 per-token GEMM with fp16 and fp32 outputs (qk_gemm_fp8_rowwise_out;
ROCm/aiter PR #6262: gemm_a8w8_bpreshuffle takes the output dtype as an
argument).  The same x as the bf16 output, rounded to fp16 (nearest even,
+-inf beyond the fp16 range) or written as fp32 itself.

* Against the oracle's unrounded fp64 value within the FP8 tolerance, for
  both output types, with and without bias: few rows (these outputs run the
  2-SM tile kernel for every M), ragged M and N, several waves of tiles, and
  a split last wave.
* The fp16 output is the oracle's fp16 rounding of the fp32 output, bit for
  bit: both run the same tiles, so they hold the same x.  Checked on whole
  outputs (signed zeros included), and where the scales push x past the
  fp16 range (+-inf there, the finite x in fp32).
"""
import numpy as np
import pytest
import torch

import block_scaled_precision_tcgen05_gb300 as qk
import oracle
import qk_inputs as qi
from gpu_util import assert_close_values, bias_dev, to_dev

pytestmark = pytest.mark.gpu

SHAPES = [
    (7, 264, 512),        # few rows: one tile, mostly zero-filled rows
    (300, 1000, 2304),    # ragged M and N
    (1536, 1792, 2320),   # 42 tiles, a ragged last K-block
    (2560, 2560, 1920),   # 100 tiles: a full wave, then 24
]


def _run(p, dtype, sa=None):
    out = torch.full((p.M, p.N), float("nan"), dtype=dtype, device="cuda")
    qk.gemm_fp8_rowwise(to_dev(p.A), to_dev(p.B), to_dev(p.sa if sa is None else sa), to_dev(p.sb),
                        bias_dev(p.bias), out)
    torch.cuda.synchronize()
    return out


def _f16_bits(t):
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


@pytest.mark.parametrize("bias", [False, True], ids=["nobias", "bias"])
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_fp8_fp16_fp32_outputs(shape, bias):
    M, N, K = shape
    p = qi.fp8_problem(M, N, K, seed=M + N, bias=bias)
    o32 = _run(p, torch.float32)
    o16 = _run(p, torch.float16)
    tiles = qi.sample_tiles(M, N, 4, 9)
    g32, g16, refs = [], [], []
    for (m0, m1, n0, n1) in tiles:
        refs.append(oracle.gemm_fp8_rowwise(p.A, p.B, p.sa, p.sb, bias=p.bias, m0=m0, m1=m1, n0=n0, n1=n1).ravel())
        g32.append(o32[m0:m1, n0:n1].cpu().numpy().astype(np.float64).ravel())
        g16.append(o16[m0:m1, n0:n1].cpu().numpy().astype(np.float64).ravel())
    ref = np.concatenate(refs)[None, :]
    assert_close_values(np.concatenate(g32)[None, :], ref, f"fp32 out {shape}")
    assert_close_values(np.concatenate(g16)[None, :], ref, f"fp16 out {shape}")
    # the fp16 output is the fp32 x rounded to nearest even
    x = o32.cpu().numpy()
    rows = slice(0, min(M, 256))
    assert np.array_equal(_f16_bits(o16)[rows], oracle.f32_to_f16(x[rows])), "fp16 != rne(fp32)"
    assert qk.device_status() == 0


def test_fp8_fp16_overflow():
    # row scales 2^16 push |x| (about 0.9 * 2^16 typical) past 65520 in many
    # outputs: fp16 gives +-inf exactly where the oracle's rounding of the
    # finite fp32 x does
    M, N, K = 300, 264, 2048
    p = qi.fp8_problem(M, N, K, seed=5)
    big = (p.sa * np.float32(65536.0)).astype(np.float32)
    o32 = _run(p, torch.float32, sa=big)
    o16 = _run(p, torch.float16, sa=big)
    x = o32.cpu().numpy()
    assert np.array_equal(_f16_bits(o16), oracle.f32_to_f16(x))
    assert np.isinf(o16.cpu().numpy()).any() and np.isfinite(x).all(), "the case must reach fp16's overflow"
    ref = oracle.gemm_fp8_rowwise(p.A, p.B, big, p.sb)
    assert_close_values(x, ref, "fp32 with large row scales")


def test_fp8_out_dtype_argument():
    p = qi.fp8_problem(64, 128, 256, seed=1)
    A, B, sa, sb = (to_dev(v) for v in (p.A, p.B, p.sa, p.sb))
    out = qk.gemm_fp8_rowwise(A, B, sa, sb, out_dtype=torch.float32)
    assert out.dtype == torch.float32 and out.shape == (64, 128)
    with pytest.raises(ValueError):
        qk.gemm_fp8_rowwise(A, B, sa, sb, out_dtype=torch.float64)
    with pytest.raises(ValueError):             # out's dtype contradicts out_dtype
        qk.gemm_fp8_rowwise(A, B, sa, sb, out=torch.empty((64, 128), dtype=torch.float16, device="cuda"),
                            out_dtype=torch.float32)
