"""MXFP8, MXFP4 and NVFP4 GEMMs with fp16 and fp32 outputs (qk_gemm_mx_out,
qk_gemm_nvfp4_out; ROCm/aiter PR #6262: its FP4 GEMM gemm_a4w4 takes the
output dtype as an argument).  The same fp32 value as the bf16 output,
rounded to fp16 (nearest even, +-inf beyond the fp16 range) or written as
fp32 itself.

* Against the oracle's unrounded fp64 value within the MX tolerance, for both
  output types, with and without bias: few rows (these outputs run the 2-SM
  tile kernel for every M), ragged M and N, a ragged last K-block, and more
  tiles than SM pairs.  The fp32 output leaves through 16-byte stores from
  registers, the fp16 one through the staging blocks of the bf16 output.
* The fp16 output is the oracle's fp16 rounding of the fp32 output, bit for
  bit (both run the same tiles): checked on whole outputs, and with A's
  scales raised by 2^16 so that many values pass the fp16 range (+-inf
  there, the finite value in fp32).
* With every tile split into K-parts (QK_TAIL_SPLIT=3), the part that
  arrives last emits the sum through the same fp16 and fp32 paths (FP8
  per-token, MXFP4, NVFP4).
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
    (1536, 1792, 2080),   # a ragged last K-block (32 elements)
    (2560, 2560, 2048),   # 100 tiles: a full wave, then 24
]
FORMATS = ["mxfp8", "mxfp4", "nvfp4"]


def _problem(fmt, M, N, K, seed, bias):
    if fmt == "nvfp4":
        return qi.nvfp4_problem(M, N, K, seed=seed, bias=bias)
    return qi.mx_problem(qi.FMT_MXFP8_E4M3 if fmt == "mxfp8" else qi.FMT_MXFP4_E2M1, M, N, K, seed=seed, bias=bias)


def _run(fmt, p, dtype, sA=None):
    out = torch.full((p.M, p.N), float("nan"), dtype=dtype, device="cuda")
    sA = p.sA if sA is None else sA
    if fmt == "nvfp4":
        ga = to_dev(np.array([p.global_a], np.float32))
        gb = to_dev(np.array([p.global_b], np.float32))
        qk.gemm_nvfp4(to_dev(p.A), to_dev(sA), to_dev(p.B), to_dev(p.sB), ga, gb, bias_dev(p.bias), out)
    else:
        qk.gemm_mx(p.fmt, to_dev(p.A), to_dev(sA), to_dev(p.B), to_dev(p.sB), bias_dev(p.bias), out)
    torch.cuda.synchronize()
    return out


def _ref(fmt, p, sA=None, **region):
    sA = p.sA if sA is None else sA
    if fmt == "nvfp4":
        return oracle.gemm_nvfp4(p.A, sA, p.B, p.sB, p.global_a, p.global_b, bias=p.bias, **region)
    return oracle.gemm_mx(p.fmt, p.A, sA, p.B, p.sB, bias=p.bias, **region)


def _f16_bits(t):
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


@pytest.mark.parametrize("bias", [False, True], ids=["nobias", "bias"])
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("fmt", FORMATS)
def test_block_scaled_fp16_fp32_outputs(fmt, shape, bias):
    M, N, K = shape
    p = _problem(fmt, M, N, K, M + N + K, bias)
    o32 = _run(fmt, p, torch.float32)
    o16 = _run(fmt, p, torch.float16)
    g32, g16, refs = [], [], []
    for (m0, m1, n0, n1) in qi.sample_tiles(M, N, 3, 11):
        refs.append(_ref(fmt, p, m0=m0, m1=m1, n0=n0, n1=n1).ravel())
        g32.append(o32[m0:m1, n0:n1].cpu().numpy().astype(np.float64).ravel())
        g16.append(o16[m0:m1, n0:n1].cpu().numpy().astype(np.float64).ravel())
    ref = np.concatenate(refs)[None, :]
    assert_close_values(np.concatenate(g32)[None, :], ref, f"{fmt} fp32 out {shape}")
    assert_close_values(np.concatenate(g16)[None, :], ref, f"{fmt} fp16 out {shape}")
    rows = slice(0, min(M, 256))
    assert np.array_equal(_f16_bits(o16)[rows], oracle.f32_to_f16(o32.cpu().numpy()[rows])), "fp16 != rne(fp32)"
    assert qk.device_status() == 0


@pytest.mark.parametrize("fmt", ["mxfp8", "mxfp4"])
def test_block_scaled_fp16_overflow(fmt):
    # A's UE8M0 codes raised by 16 multiply every value by 2^16: many pass
    # 65520, where fp16 holds +-inf and fp32 the finite value
    M, N, K = 300, 264, 2048
    p = _problem(fmt, M, N, K, 5, False)
    sA = (p.sA.astype(np.int32) + 16).astype(np.uint8)
    o32 = _run(fmt, p, torch.float32, sA=sA)
    o16 = _run(fmt, p, torch.float16, sA=sA)
    x = o32.cpu().numpy()
    assert np.array_equal(_f16_bits(o16), oracle.f32_to_f16(x))
    assert np.isinf(o16.cpu().numpy()).any() and np.isfinite(x).all(), "the case must reach fp16's overflow"
    assert_close_values(x, _ref(fmt, p, sA=sA), f"{fmt} fp32 with raised scales")


def test_block_scaled_out_dtype_argument():
    p = _problem("mxfp4", 64, 128, 256, 1, False)
    args = [to_dev(v) for v in (p.A, p.sA, p.B, p.sB)]
    out = qk.gemm_mx(p.fmt, *args, out_dtype=torch.float32)
    assert out.dtype == torch.float32 and out.shape == (64, 128)
    with pytest.raises(ValueError):
        qk.gemm_mx(p.fmt, *args, out_dtype=torch.float64)
    q = _problem("nvfp4", 64, 128, 256, 1, False)
    out = qk.gemm_nvfp4(*[to_dev(v) for v in (q.A, q.sA, q.B, q.sB)], out_dtype=torch.float16)
    assert out.dtype == torch.float16 and out.shape == (64, 128)


@pytest.mark.parametrize("fmt", ["fp8", "mxfp4", "nvfp4"])
def test_out_types_with_tail_split(fmt, monkeypatch):
    # every tile split into three K-parts: the part that arrives last emits
    # the sum through the fp16 staging blocks or the fp32 direct stores
    monkeypatch.setenv("QK_TAIL_SPLIT", "3")
    M, N, K = 600, 776, 3872
    if fmt == "fp8":
        p = qi.fp8_problem(M, N, K, seed=41, bias=True)
        outs = {}
        for dt in (torch.float32, torch.float16):
            o = torch.full((M, N), float("nan"), dtype=dt, device="cuda")
            qk.gemm_fp8_rowwise(to_dev(p.A), to_dev(p.B), to_dev(p.sa), to_dev(p.sb), bias_dev(p.bias), o)
            outs[dt] = o
        torch.cuda.synchronize()
        ref_fn = lambda **r: oracle.gemm_fp8_rowwise(p.A, p.B, p.sa, p.sb, bias=p.bias, **r)
    else:
        p = _problem(fmt, M, N, K, 41, True)
        outs = {dt: _run(fmt, p, dt) for dt in (torch.float32, torch.float16)}
        ref_fn = lambda **r: _ref(fmt, p, **r)
    g32, g16, refs = [], [], []
    for (m0, m1, n0, n1) in qi.sample_tiles(M, N, 3, 12):
        refs.append(ref_fn(m0=m0, m1=m1, n0=n0, n1=n1).ravel())
        g32.append(outs[torch.float32][m0:m1, n0:n1].cpu().numpy().astype(np.float64).ravel())
        g16.append(outs[torch.float16][m0:m1, n0:n1].cpu().numpy().astype(np.float64).ravel())
    ref = np.concatenate(refs)[None, :]
    assert_close_values(np.concatenate(g32)[None, :], ref, f"{fmt} fp32 out, split")
    assert_close_values(np.concatenate(g16)[None, :], ref, f"{fmt} fp16 out, split")
    x = outs[torch.float32].cpu().numpy()
    assert np.array_equal(_f16_bits(outs[torch.float16])[:128], oracle.f32_to_f16(x[:128])), "fp16 != rne(fp32)"
    assert qk.device_status() == 0
